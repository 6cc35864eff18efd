// qsa_decode_partial: split-KV partial attention for decode tokens.
//
// "round 27 track b - qsa prep and merge", decision and correctness: the production
// decode kernel (qsa_attn2) computes per-chunk partials into `part` with a head stride
// of 258 floats (o[256], m, l) and a chunk stride of 24*258; its key loads are four
// bytes wide and its inner loops run over 8 values and over the heads.
//
// One CTA (256 threads) per (chunk k, group g, quarter of the group's 12 heads, token t):
// the head split gives the small decode batches four times as many CTAs to spread over the
// SMs, at the cost of each chunk's 64 rows being read by four CTAs (from L2 after the first).
// The chunk's cells (identity range or ids, ascending) are staged as int8 rows plus fp32
// scales in shared memory.  Logits: 8 lanes per cell, each lane owning 32 dims (two 16-dim
// runs, 128 apart) of the CTA's 3 query rows held in registers as fp32; int8 x scale is
// exact in fp32.  The softmax statistics use natural exp; each thread then owns one output
// dim for the 3 heads.  All arithmetic is fp32.
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kHS = 4;            // CTAs per group (head quarters)
constexpr int kHPC = kHPG / kHS;  // query heads per CTA
static_assert(kHPC == 3, "the weight layout below packs 3 heads in a float4");

__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(
    const __half* __restrict__ q, const int8_t* __restrict__ kq, const int8_t* __restrict__ vq,
    const __half* __restrict__ ksc, const __half* __restrict__ vsc, const int32_t* __restrict__ ids,
    float* __restrict__ part, int32_t* __restrict__ n_chunks, int chunk_cap, int pos0, Params p, int* status) {
  __shared__ __align__(16) int8_t s_k[kChunk][kD];
  __shared__ __align__(16) int8_t s_v[kChunk][kD];
  __shared__ float s_ksc[kChunk][kNB];
  __shared__ float s_vsc[kChunk][kNB];
  __shared__ int s_cell[kChunk];
  __shared__ float s_s[kHPC][kChunk];           // logits
  __shared__ __align__(16) float4 s_e[kChunk];  // per cell: exp(s - m) of the 3 heads, .w unused

  pdl_begin();
  const int k = blockIdx.x, g = blockIdx.y / kHS, hq = blockIdx.y % kHS, t = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h0 = g * kHPG + hq * kHPC;  // first query head of this CTA
  const long long n_kv = (long long)pos0 + t + 1;
  const bool identity = n_kv <= p.identity_max;
  const int n_set = identity ? (int)n_kv : p.topk;
  const int nc = (n_set + kChunk - 1) / kChunk;
  if (k == 0 && blockIdx.y == 0 && tid == 0) n_chunks[t] = nc;
  if (k >= nc) return;
  const int c0 = k * kChunk;
  const int cnt = min(kChunk, n_set - c0);

  if (tid < kChunk) {
    int cell = -1;
    if (tid < cnt) {
      cell = identity ? c0 + tid : ids[((size_t)t * kGroups + g) * p.topk + c0 + tid];
      if (cell < 0 || (long long)cell >= n_kv) {
        set_dev_status(status, QSA_DEV_BAD_ID);
        cell = -1;
      }
    }
    s_cell[tid] = cell;
  }
  // this lane's query dims: j*16 + 128*i + (0..15), i = 0, 1, for the CTA's 3 heads
  const int j = lane & 7;
  float qf[kHPC][32];
#pragma unroll
  for (int h = 0; h < kHPC; ++h) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)t * kHeads + h0 + h) * kD + j * 16 + 128 * i);
      const uint4 a = __ldg(src), b = __ldg(src + 1);
      const __half2* a2 = reinterpret_cast<const __half2*>(&a);
      const __half2* b2 = reinterpret_cast<const __half2*>(&b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 fa = __half22float2(a2[u]), fb = __half22float2(b2[u]);
        qf[h][16 * i + 2 * u] = fa.x;
        qf[h][16 * i + 2 * u + 1] = fa.y;
        qf[h][16 * i + 8 + 2 * u] = fb.x;
        qf[h][16 * i + 8 + 2 * u + 1] = fb.y;
      }
    }
  }
  __syncthreads();
  // int8 rows: 16 pieces of 16 bytes per row, K and V; all loads issued before the stores
  {
    uint4 kv[4], vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + u * kDecThreads, r = i >> 4, c16 = i & 15;
      const int cell = s_cell[r];
      kv[u] = make_uint4(0, 0, 0, 0);
      vv[u] = make_uint4(0, 0, 0, 0);
      if (cell >= 0) {
        kv[u] = __ldg(reinterpret_cast<const uint4*>(kq + ((size_t)cell * kGroups + g) * kD + c16 * 16));
        vv[u] = __ldg(reinterpret_cast<const uint4*>(vq + ((size_t)cell * kGroups + g) * kD + c16 * 16));
      }
    }
    const int r = tid >> 2, b = tid & 3;  // 64 cells x 4 blocks = 256 threads
    const int cell = s_cell[r];
    const float ks = cell >= 0 ? __half2float(ksc[((size_t)cell * kGroups + g) * kNB + b]) : 0.f;
    const float vs = cell >= 0 ? __half2float(vsc[((size_t)cell * kGroups + g) * kNB + b]) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = tid + u * kDecThreads, rr = i >> 4, c16 = i & 15;
      *reinterpret_cast<uint4*>(&s_k[rr][c16 * 16]) = kv[u];
      *reinterpret_cast<uint4*>(&s_v[rr][c16 * 16]) = vv[u];
    }
    s_ksc[r][b] = ks;
    s_vsc[r][b] = vs;
  }
  __syncthreads();

  // logits: 8 lanes per cell (4 cells per warp, 32 per pass), lane j over its 32 dims
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int r = pass * 32 + warp * 4 + (lane >> 3);
    float acc[kHPC] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 w = *reinterpret_cast<const uint4*>(&s_k[r][j * 16 + 128 * i]);
      const float sc = s_ksc[r][(j >> 2) + 2 * i];
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float kf = (float)(int8_t)(wv[u >> 2] >> (8 * (u & 3))) * sc;
#pragma unroll
        for (int h = 0; h < kHPC; ++h) acc[h] = fmaf(qf[h][16 * i + u], kf, acc[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < kHPC; ++h) {
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 1);
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 2);
      acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], 4);
    }
    if (j == 0) {
      const bool valid = s_cell[r] >= 0;
#pragma unroll
      for (int h = 0; h < kHPC; ++h) s_s[h][r] = valid ? acc[h] * p.sm_scale : -INFINITY;
    }
  }
  __syncthreads();

  // softmax statistics per head: warp h, lanes over cells (two each)
  if (warp < kHPC) {
    const int h = warp;
    const float a = s_s[h][lane], b = s_s[h][lane + 32];
    float m = fmaxf(a, b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float msafe = (m == -INFINITY) ? 0.f : m;
    const float ea = __expf(a - msafe), eb = __expf(b - msafe);
    float l = ea + eb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    reinterpret_cast<float*>(&s_e[lane])[h] = ea;
    reinterpret_cast<float*>(&s_e[lane + 32])[h] = eb;
    if (lane == 0) {
      float* dst = part + (((size_t)t * chunk_cap + k) * kHeads + h0 + h) * kPartStride;
      dst[kD] = m;
      dst[kD + 1] = l;
    }
  }
  __syncthreads();

  // o[h][d] = sum_r e[h][r] * v^[r][d]: thread = dim, 3 heads
  const int d = tid;
  float acc[kHPC] = {0.f, 0.f, 0.f};
  for (int r = 0; r < cnt; ++r) {
    const float v = (float)s_v[r][d] * s_vsc[r][d >> 6];
    const float4 e = s_e[r];
    acc[0] = fmaf(e.x, v, acc[0]);
    acc[1] = fmaf(e.y, v, acc[1]);
    acc[2] = fmaf(e.z, v, acc[2]);
  }
#pragma unroll
  for (int h = 0; h < kHPC; ++h)
    part[(((size_t)t * chunk_cap + k) * kHeads + h0 + h) * kPartStride + d] = acc[h];
}

}  // namespace

cudaError_t launch_decode_partial(const __half* q, const int8_t* kq, const int8_t* vq, const __half* ksc,
                                  const __half* vsc, const int32_t* ids, float* part, int32_t* n_chunks,
                                  int chunk_cap, int n_cells, int N, int pos0, Params p, int* status,
                                  cudaStream_t stream) {
  (void)n_cells;
  dim3 grid(chunk_cap, kGroups * kHS, N);
  return launch_pdl(decode_partial_kernel, grid, dim3(kDecThreads), 0, stream, q, kq, vq, ksc, vsc, ids, part, n_chunks,
                    chunk_cap, pos0, p, status);
}

}  // namespace qsa
