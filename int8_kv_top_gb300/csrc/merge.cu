// qsa_merge: log-sum-exp merge of split-KV decode partials.
//
// "round 27 track b - qsa prep and merge", decision: the merge loads each chunk's
// (m, l) pair as one aligned float2 (head stride 258 and chunk stride 24*258 keep the
// pair 8-byte aligned, correctness section) and takes the maximum in parallel.
//
// One CTA per (token, head), 128 threads, each producing two output dims from float2 loads
// of the chunk rows (a row of 258 floats starts 8-byte aligned, so float2 is the widest
// aligned access).  The first 64 chunks' (m, l) pairs and row slices are loaded before the
// chunk count is known (every chunk slot below the capacity is inside the buffer; slots past
// the count are never used), so the CTA waits on one round of loads rather than a chain.
// Every warp reduces M = max m and L = sum l * exp(m - M) itself with shuffles (lane = chunk),
// and takes the chunk weights exp(m_k - M) / L from lane k.  With a gate input the merged
// output is multiplied by sigmoid(gate) before it is stored.
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kMergeThreads = 128;
constexpr int kRegChunks = 64;  // chunks whose rows are loaded up front (two per lane)
constexpr int kMaxChunks = 1024;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ part,
                                                              const int32_t* __restrict__ n_chunks, int chunk_cap,
                                                              const __half* __restrict__ gate, float* __restrict__ xp,
                                                              int* status) {
  pdl_begin();
  const int t = blockIdx.x / kHeads, h = blockIdx.x % kHeads;
  const int tid = threadIdx.x, lane = tid & 31;
  const size_t cs = (size_t)kHeads * kPartStride;  // chunk stride
  const float* base = part + (size_t)t * chunk_cap * cs + (size_t)h * kPartStride;
  const int d = tid * 2;
  const int kk = min(chunk_cap, kRegChunks);

  float2 ml0 = make_float2(-INFINITY, 0.f), ml1 = make_float2(-INFINITY, 0.f);
  if (lane < kk) ml0 = __ldg(reinterpret_cast<const float2*>(base + lane * cs + kD));
  if (lane + 32 < kk) ml1 = __ldg(reinterpret_cast<const float2*>(base + (lane + 32) * cs + kD));
  float2 o[kRegChunks];
#pragma unroll
  for (int i = 0; i < kRegChunks; ++i)
    o[i] = i < kk ? __ldg(reinterpret_cast<const float2*>(base + i * cs + d)) : make_float2(0.f, 0.f);
  int nc = __ldg(n_chunks + t);
  if (nc < 1 || nc > chunk_cap) {
    if (tid == 0) set_dev_status(status, QSA_DEV_BAD_ID);
    *reinterpret_cast<float2*>(xp + ((size_t)t * kHeads + h) * kD + d) =
        make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    return;
  }
  if (lane >= nc) ml0 = make_float2(-INFINITY, 0.f);
  if (lane + 32 >= nc) ml1 = make_float2(-INFINITY, 0.f);

  // M and L over all nc chunks (lane = chunk; chunks past 64 are read here)
  float M = fmaxf(ml0.x, ml1.x);
  for (int k = kRegChunks + lane; k < nc; k += 32) M = fmaxf(M, base[k * cs + kD]);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, s));
  float e0 = lane < nc ? __expf(ml0.x - M) : 0.f, e1 = lane + 32 < nc ? __expf(ml1.x - M) : 0.f;
  float L = fmaf(ml0.y, e0, ml1.y * e1);
  for (int k = kRegChunks + lane; k < nc; k += 32) {
    const float2 ml = *reinterpret_cast<const float2*>(base + k * cs + kD);
    L = fmaf(ml.y, __expf(ml.x - M), L);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) L += __shfl_xor_sync(0xffffffffu, L, s);
  const float invL = 1.f / L;
  e0 *= invL;
  e1 *= invL;

  float2 a4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < kRegChunks; ++i) {
    const float w = __shfl_sync(0xffffffffu, i < 32 ? e0 : e1, i & 31);
    const float2 oi = i < nc ? o[i] : make_float2(0.f, 0.f);  // slots past nc hold stale data
    a4[i & 3].x = fmaf(w, oi.x, a4[i & 3].x);
    a4[i & 3].y = fmaf(w, oi.y, a4[i & 3].y);
  }
  for (int k = kRegChunks; k < nc; ++k) {
    const float2 ml = *reinterpret_cast<const float2*>(base + k * cs + kD);
    const float w = __expf(ml.x - M) * invL;
    const float2 ok = *reinterpret_cast<const float2*>(base + k * cs + d);
    a4[k & 3].x = fmaf(w, ok.x, a4[k & 3].x);
    a4[k & 3].y = fmaf(w, ok.y, a4[k & 3].y);
  }
  float2 acc =
      make_float2((a4[0].x + a4[1].x) + (a4[2].x + a4[3].x), (a4[0].y + a4[1].y) + (a4[2].y + a4[3].y));
  if (gate) {  // output gate: xp *= sigmoid(gate)
    const float2 gv = __half22float2(*reinterpret_cast<const __half2*>(gate + ((size_t)t * kHeads + h) * kD + d));
    acc.x *= gate_sigmoid(gv.x);
    acc.y *= gate_sigmoid(gv.y);
  }
  *reinterpret_cast<float2*>(xp + ((size_t)t * kHeads + h) * kD + d) = acc;
}

}  // namespace

cudaError_t launch_merge(const float* part, const int32_t* n_chunks, int N, int chunk_cap, const __half* gate,
                         float* xp, int* status, cudaStream_t stream) {
  if (chunk_cap > kMaxChunks) return cudaErrorInvalidValue;
  return launch_pdl(merge_kernel, dim3(N * kHeads), dim3(kMergeThreads), 0, stream, part, n_chunks, chunk_cap, gate,
                    xp, status);
}

}  // namespace qsa
