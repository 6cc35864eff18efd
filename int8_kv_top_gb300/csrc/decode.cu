// qsa_decode_partial: split-KV partial attention for decode tokens.
//
// "round 27 track b - qsa prep and merge", decision and correctness: the production
// decode kernel (qsa_attn2) computes per-chunk partials into `part` with a head stride
// of 258 floats (o[256], m, l) and a chunk stride of 24*258; its key loads are four
// bytes wide and its inner loops run over 8 values and over the heads.
//
// One CTA (256 threads) per (chunk k, group g, token t).  The chunk's 64 cells (identity
// range or ids, ascending) are staged as int8 rows plus fp32 scales in shared memory;
// logits use one warp per cell with lanes over 8-dim slices (int8 x scale is exact in
// fp32), the softmax statistics use natural exp, and each thread then owns one output
// dim for all 12 heads.  All arithmetic is fp32.
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kDecThreads = 256;

__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(
    const __half* __restrict__ q, const int8_t* __restrict__ kq, const int8_t* __restrict__ vq,
    const __half* __restrict__ ksc, const __half* __restrict__ vsc, const int32_t* __restrict__ ids,
    float* __restrict__ part, int32_t* __restrict__ n_chunks, int chunk_cap, int pos0, Params p, int* status) {
  __shared__ __align__(16) __half s_q[kHPG][kD];
  __shared__ __align__(16) int8_t s_k[kChunk][kD];
  __shared__ __align__(16) int8_t s_v[kChunk][kD];
  __shared__ float s_ksc[kChunk][kNB];
  __shared__ float s_vsc[kChunk][kNB];
  __shared__ int s_cell[kChunk];
  __shared__ float s_s[kHPG][kChunk];

  const int k = blockIdx.x, g = blockIdx.y, t = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long n_kv = (long long)pos0 + t + 1;
  const bool identity = n_kv <= p.identity_max;
  const int n_set = identity ? (int)n_kv : p.topk;
  const int nc = (n_set + kChunk - 1) / kChunk;
  if (k == 0 && g == 0 && tid == 0) n_chunks[t] = nc;
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
  for (int i = tid; i < kHPG * kD; i += kDecThreads) {
    const int h = i / kD, d = i % kD;
    s_q[h][d] = q[((size_t)t * kHeads + g * kHPG + h) * kD + d];
  }
  __syncthreads();
  // int8 rows: 16 chunks of 16 bytes per row, K and V
  for (int i = tid; i < kChunk * 16; i += kDecThreads) {
    const int r = i >> 4, c16 = i & 15;
    const int cell = s_cell[r];
    uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
    if (cell >= 0) {
      kv = *reinterpret_cast<const uint4*>(kq + ((size_t)cell * kGroups + g) * kD + c16 * 16);
      vv = *reinterpret_cast<const uint4*>(vq + ((size_t)cell * kGroups + g) * kD + c16 * 16);
    }
    *reinterpret_cast<uint4*>(&s_k[r][c16 * 16]) = kv;
    *reinterpret_cast<uint4*>(&s_v[r][c16 * 16]) = vv;
  }
  {
    const int r = tid >> 2, b = tid & 3;  // 64 cells x 4 blocks = 256 threads
    const int cell = s_cell[r];
    s_ksc[r][b] = cell >= 0 ? __half2float(ksc[((size_t)cell * kGroups + g) * kNB + b]) : 0.f;
    s_vsc[r][b] = cell >= 0 ? __half2float(vsc[((size_t)cell * kGroups + g) * kNB + b]) : 0.f;
  }
  __syncthreads();

  // logits: warp per cell, lane over dims lane*8 .. lane*8+7
  for (int r = warp; r < kChunk; r += kDecThreads / 32) {
    const float sc = s_ksc[r][lane >> 3];
    float kf[8];
    const uint2 w = *reinterpret_cast<const uint2*>(&s_k[r][lane * 8]);
#pragma unroll
    for (int j = 0; j < 4; ++j) kf[j] = (float)(int8_t)(w.x >> (8 * j)) * sc;
#pragma unroll
    for (int j = 0; j < 4; ++j) kf[4 + j] = (float)(int8_t)(w.y >> (8 * j)) * sc;
#pragma unroll
    for (int h = 0; h < kHPG; ++h) {
      float acc = 0.f;
      const uint4 qw = *reinterpret_cast<const uint4*>(&s_q[h][lane * 8]);
      const __half2* q2 = reinterpret_cast<const __half2*>(&qw);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 qf = __half22float2(q2[j]);
        acc = fmaf(qf.x, kf[2 * j], acc);
        acc = fmaf(qf.y, kf[2 * j + 1], acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) s_s[h][r] = (s_cell[r] >= 0) ? acc * p.sm_scale : -INFINITY;
    }
  }
  __syncthreads();

  // softmax statistics per head: lanes over cells (two each)
  for (int h = warp; h < kHPG; h += kDecThreads / 32) {
    const float a = s_s[h][lane], b = s_s[h][lane + 32];
    float m = fmaxf(a, b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float msafe = (m == -INFINITY) ? 0.f : m;
    const float ea = __expf(a - msafe), eb = __expf(b - msafe);
    float l = ea + eb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    s_s[h][lane] = ea;
    s_s[h][lane + 32] = eb;
    if (lane == 0) {
      float* dst = part + (((size_t)t * chunk_cap + k) * kHeads + g * kHPG + h) * kPartStride;
      dst[kD] = m;
      dst[kD + 1] = l;
    }
  }
  __syncthreads();

  // o[h][d] = sum_r e[h][r] * v^[r][d]
  const int d = tid;
  float acc[kHPG];
#pragma unroll
  for (int h = 0; h < kHPG; ++h) acc[h] = 0.f;
  for (int r = 0; r < cnt; ++r) {
    const float v = (float)s_v[r][d] * s_vsc[r][d >> 6];
#pragma unroll
    for (int h = 0; h < kHPG; ++h) acc[h] = fmaf(s_s[h][r], v, acc[h]);
  }
#pragma unroll
  for (int h = 0; h < kHPG; ++h)
    part[(((size_t)t * chunk_cap + k) * kHeads + g * kHPG + h) * kPartStride + d] = acc[h];
}

}  // namespace

cudaError_t launch_decode_partial(const __half* q, const int8_t* kq, const int8_t* vq, const __half* ksc,
                                  const __half* vsc, const int32_t* ids, float* part, int32_t* n_chunks,
                                  int chunk_cap, int n_cells, int N, int pos0, Params p, int* status,
                                  cudaStream_t stream) {
  (void)n_cells;
  dim3 grid(chunk_cap, kGroups, N);
  decode_partial_kernel<<<grid, kDecThreads, 0, stream>>>(q, kq, vq, ksc, vsc, ids, part, n_chunks, chunk_cap, pos0,
                                                         p, status);
  return cudaGetLastError();
}

}  // namespace qsa
