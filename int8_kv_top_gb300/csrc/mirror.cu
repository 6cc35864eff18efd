// The per-call fp16 mirror of the int8 KV cache used by both prefill kernels.
//
// The cache stays int8 with one fp16 scale per 64 elements ("round 6 track b - qsa flash",
// delivered change: half4 scales per cell).  Every prefill tile reads each cache cell many
// times (each 64-cell chunk by every later 128-row tile of its group; each selected cell by
// every token that selects it), so the call dequantises every cell it can see exactly once,
// k^ = fp16(code * scale) with a single rounding, into a caller workspace that the tiles then
// stream through L2.
#include <algorithm>

#include "common.cuh"

namespace qsa {
namespace {

// grid (ceil(n / 8), 2 groups), 256 threads: a warp per cell row, K and V.
__global__ void __launch_bounds__(256)
    dequant_mirror_kernel(const int8_t* __restrict__ kq, const int8_t* __restrict__ vq, const __half* __restrict__ ksc,
                          const __half* __restrict__ vsc, int n, __half* __restrict__ khat, __half* __restrict__ vhat) {
  pdl_begin();
  const int g = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 8 + warp;
  if (c >= n) return;
  const size_t row = ((size_t)c * kGroups + g) * kD + lane * 8;
  const int blk = lane >> 3;
  uint32_t o[4];
  const uint2 wk = *reinterpret_cast<const uint2*>(kq + row);
  dequant8(wk.x, wk.y, __half2half2(ksc[((size_t)c * kGroups + g) * kNB + blk]), o);
  *reinterpret_cast<uint4*>(khat + row) = make_uint4(o[0], o[1], o[2], o[3]);
  const uint2 wv = *reinterpret_cast<const uint2*>(vq + row);
  dequant8(wv.x, wv.y, __half2half2(vsc[((size_t)c * kGroups + g) * kNB + blk]), o);
  *reinterpret_cast<uint4*>(vhat + row) = make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------- batched prefill
// Sequence s of a batched call, {first pool cell, n_cells, pos0, first token row}: its tokens are
// the rows up to the next sequence's first row (n_tok for the last).  Returns the token count, or
// -1 when the entry breaks the cache contract, starts before the previous sequence's rows, or
// reaches beyond max_n_kv cells.
__device__ __forceinline__ int batch_seq_tokens(const int4* seqs, int s, int n_seq, int n_tok, long long n_pool,
                                                int max_n_kv, int4* e_out) {
  const int4 e = __ldg(&seqs[s]);
  const int next = s + 1 < n_seq ? __ldg(&seqs[s + 1].w) : n_tok;
  const int first_ok = s == 0 ? e.w == 0 : __ldg(&seqs[s - 1].w) <= e.w;
  const int T = next - e.w;
  *e_out = e;
  const bool ok = first_ok && e.x >= 0 && e.y >= 1 && e.z >= 0 && T >= 0 && next <= n_tok &&
                  (long long)e.z + T <= e.y && (long long)e.x + e.y <= n_pool && (long long)e.z + T <= max_n_kv;
  return ok ? T : -1;
}

// Identity tokens of a sequence at pos0 with T tokens: those with n_kv = pos0 + t + 1 <= identity_max.
__device__ __forceinline__ int batch_identity_tokens(int pos0, int T, int identity_max) {
  return min(max(identity_max - pos0, 0), T);
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanBins = 1024;  // super-chunk counts J = 1 .. 1024 (n_kv <= 131072)
constexpr int kSuper = 128;      // cells per super-chunk of the dense kernel
constexpr int kPairTok = 64;     // tokens per pair item of the dense kernel

// One CTA: the work list of the identity tokens' tiles, plan[0].x = pair count and plan[1 + i] =
// {first token row, end of the sequence's identity rows, pos0 - first row, first mirror row}, in
// decreasing order of super-chunks (a counting sort), so that the heaviest pairs start first.
__global__ void __launch_bounds__(kPlanThreads) batch_plan_kernel(const int4* __restrict__ seqs, int n_seq, int n_tok,
                                                                  long long n_pool, int max_n_kv, int identity_max,
                                                                  int rows_per_seq, int4* __restrict__ plan,
                                                                  int* status) {
  __shared__ int s_cnt[kPlanBins];
  __shared__ int s_wsum[kPlanThreads / 32];
  pdl_begin();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kPlanBins; i += kPlanThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int s = tid; s < n_seq; s += kPlanThreads) {
    int4 e;
    const int T = batch_seq_tokens(seqs, s, n_seq, n_tok, n_pool, max_n_kv, &e);
    if (T < 0) {
      set_dev_status(status, QSA_DEV_BAD_ID);
      continue;
    }
    const int nid = batch_identity_tokens(e.z, T, identity_max);
    for (int k = 0; k < nid; k += kPairTok) atomicAdd(&s_cnt[(e.z + min(k + kPairTok, nid) + kSuper - 1) / kSuper - 1], 1);
  }
  __syncthreads();
  // exclusive scan in decreasing J: thread i takes bin kPlanBins - 1 - i
  const int b = kPlanBins - 1 - tid;
  const int v = s_cnt[b];
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_wsum[warp] = x;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += s_wsum[w];
  const int excl = before + x - v;
  __syncthreads();
  s_cnt[b] = excl;
  if (tid == kPlanThreads - 1) plan[0] = make_int4(excl + v, 0, 0, 0);
  __syncthreads();
  for (int s = tid; s < n_seq; s += kPlanThreads) {
    int4 e;
    const int T = batch_seq_tokens(seqs, s, n_seq, n_tok, n_pool, max_n_kv, &e);
    if (T < 0) continue;
    const int nid = batch_identity_tokens(e.z, T, identity_max);
    for (int k = 0; k < nid; k += kPairTok) {
      const int pos = atomicAdd(&s_cnt[(e.z + min(k + kPairTok, nid) + kSuper - 1) / kSuper - 1], 1);
      plan[1 + pos] = make_int4(e.w + k, e.w + nid, e.z - e.w, s * rows_per_seq);
    }
  }
}

// grid (rows_per_seq / 8, 2 groups, n_seq), 256 threads: sequence s's identity cells (the cells its
// identity tokens see) into mirror rows s * rows_per_seq + c, zeros from there to the end of the
// last super-chunk the dense kernel reads, nothing beyond.
__global__ void __launch_bounds__(256)
    batch_mirror_kernel(const int8_t* __restrict__ kq, const int8_t* __restrict__ vq, const __half* __restrict__ ksc,
                        const __half* __restrict__ vsc, const int4* __restrict__ seqs, int n_seq, int n_tok,
                        long long n_pool, int max_n_kv, int identity_max, int rows_per_seq, __half* __restrict__ khat,
                        __half* __restrict__ vhat) {
  pdl_begin();
  const int g = blockIdx.y, s = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int4 e;
  const int T = batch_seq_tokens(seqs, s, n_seq, n_tok, n_pool, max_n_kv, &e);
  if (T < 0) return;
  const int nid = batch_identity_tokens(e.z, T, identity_max);
  const int nvis = nid > 0 ? e.z + nid : 0;
  const int c = blockIdx.x * 8 + warp;
  if (c >= (nvis + kSuper - 1) / kSuper * kSuper) return;
  const size_t dst = (((size_t)s * rows_per_seq + c) * kGroups + g) * kD + lane * 8;
  if (c >= nvis) {
    *reinterpret_cast<uint4*>(khat + dst) = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(vhat + dst) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const size_t cell = (size_t)e.x + c;
  const size_t row = (cell * kGroups + g) * kD + lane * 8;
  const int blk = lane >> 3;
  uint32_t o[4];
  const uint2 wk = *reinterpret_cast<const uint2*>(kq + row);
  dequant8(wk.x, wk.y, __half2half2(ksc[(cell * kGroups + g) * kNB + blk]), o);
  *reinterpret_cast<uint4*>(khat + dst) = make_uint4(o[0], o[1], o[2], o[3]);
  const uint2 wv = *reinterpret_cast<const uint2*>(vq + row);
  dequant8(wv.x, wv.y, __half2half2(vsc[(cell * kGroups + g) * kNB + blk]), o);
  *reinterpret_cast<uint4*>(vhat + dst) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

BatchedPrefillLayout batched_prefill_layout(int n_seq, int n_tok, int max_n_kv, int identity_max) {
  BatchedPrefillLayout L{};
  const int vis = std::min(identity_max, max_n_kv);  // cells an identity token can see
  L.rows_per_seq = vis > 0 ? (vis + kSuper - 1) / kSuper * kSuper : 0;
  L.max_pairs = (int)std::min<long long>((long long)n_tok / kPairTok + n_seq, (long long)n_tok);
  L.mirror_rows = (long long)n_seq * L.rows_per_seq;
  L.plan_bytes = ((size_t)(1 + L.max_pairs) * sizeof(int4) + 255) / 256 * 256;
  L.bytes = L.plan_bytes + 2 * (size_t)L.mirror_rows * kGroups * kD * sizeof(__half);
  return L;
}

cudaError_t launch_batched_prefill_prep(const int8_t* kq, const int8_t* vq, const __half* ksc, const __half* vsc,
                                        const int4* seqs, int n_seq, int n_tok, long long n_pool, int max_n_kv,
                                        int identity_max, const BatchedPrefillLayout& L, void* ws, int* status,
                                        cudaStream_t stream) {
  int4* plan = static_cast<int4*>(ws);
  __half* khat = reinterpret_cast<__half*>(static_cast<uint8_t*>(ws) + L.plan_bytes);
  __half* vhat = khat + (size_t)L.mirror_rows * kGroups * kD;
  cudaError_t e = launch_pdl(batch_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, seqs, n_seq, n_tok, n_pool,
                             max_n_kv, identity_max, L.rows_per_seq, plan, status);
  if (e != cudaSuccess || L.rows_per_seq == 0) return e;
  return launch_pdl(batch_mirror_kernel, dim3(L.rows_per_seq / 8, kGroups, n_seq), dim3(256), 0, stream, kq, vq, ksc,
                    vsc, seqs, n_seq, n_tok, n_pool, max_n_kv, identity_max, L.rows_per_seq, khat, vhat);
}

size_t prefill_workspace_bytes(int T, int pos0) {
  const size_t n = (size_t)pos0 + T;  // cells any token of the call can see
  return 2 * n * kGroups * kD * sizeof(__half);
}

cudaError_t launch_dequant_mirror(const int8_t* kq, const int8_t* vq, const __half* ksc, const __half* vsc, int n,
                                  __half* khat, __half* vhat, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(dequant_mirror_kernel, dim3((n + 7) / 8, kGroups), dim3(256), 0, stream, kq, vq, ksc, vsc, n, khat,
                    vhat);
}

}  // namespace qsa
