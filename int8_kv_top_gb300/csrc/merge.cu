// qsa_merge: log-sum-exp merge of split-KV decode partials.
//
// "round 27 track b - qsa prep and merge", decision: the merge loads each chunk's
// (m, l) pair as one aligned float2 (head stride 258 and chunk stride 24*258 keep the
// pair 8-byte aligned, correctness section) and takes the maximum in parallel.
//
// One CTA per (token, head).  Warp 0 reads the (m, l) pairs of all chunks with float2
// loads, reduces M = max m and L = sum l * exp(m - M) with shuffles and publishes the
// per-chunk weights exp(m - M) / L in shared memory; then 128 threads each produce two
// output dims from float2 loads of the chunk rows (a row of 258 floats starts 8-byte
// aligned, so float2 is the widest aligned access).
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kMergeThreads = 128;
constexpr int kMaxChunksSmem = 1024;

__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ part,
                                                              const int32_t* __restrict__ n_chunks, int chunk_cap,
                                                              float* __restrict__ xp, int* status) {
  __shared__ float w[kMaxChunksSmem];
  __shared__ int s_nc;
  const int t = blockIdx.x / kHeads, h = blockIdx.x % kHeads;
  const int tid = threadIdx.x;
  const size_t chunk_stride = (size_t)kHeads * kPartStride;
  const float* base = part + (size_t)t * chunk_cap * chunk_stride + (size_t)h * kPartStride;

  if (tid < 32) {
    int nc = n_chunks[t];
    if (nc < 1 || nc > chunk_cap) {
      if (tid == 0) set_dev_status(status, QSA_DEV_BAD_ID);
      nc = 0;
    }
    float M = -INFINITY;
    for (int k = tid; k < nc; k += 32) {
      const float2 ml = *reinterpret_cast<const float2*>(base + k * chunk_stride + kD);
      w[k] = ml.x;
      M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int k = tid; k < nc; k += 32) {
      const float l = base[k * chunk_stride + kD + 1];
      const float e = __expf(w[k] - M);
      w[k] = e;
      L = fmaf(l, e, L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float invL = (nc > 0) ? 1.f / L : __int_as_float(0x7fc00000);
    for (int k = tid; k < nc; k += 32) w[k] *= invL;
    if (tid == 0) s_nc = nc;
  }
  __syncthreads();
  const int nc = s_nc;
  const int d = tid * 2;
  float2 acc = make_float2(0.f, 0.f);
  for (int k = 0; k < nc; ++k) {
    const float2 o = *reinterpret_cast<const float2*>(base + k * chunk_stride + d);
    acc.x = fmaf(w[k], o.x, acc.x);
    acc.y = fmaf(w[k], o.y, acc.y);
  }
  if (nc == 0) acc = make_float2(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
  *reinterpret_cast<float2*>(xp + ((size_t)t * kHeads + h) * kD + d) = acc;
}

}  // namespace

cudaError_t launch_merge(const float* part, const int32_t* n_chunks, int N, int chunk_cap, float* xp, int* status,
                         cudaStream_t stream) {
  if (chunk_cap > kMaxChunksSmem) return cudaErrorInvalidValue;
  merge_kernel<<<N * kHeads, kMergeThreads, 0, stream>>>(part, n_chunks, chunk_cap, xp, status);
  return cudaGetLastError();
}

}  // namespace qsa
