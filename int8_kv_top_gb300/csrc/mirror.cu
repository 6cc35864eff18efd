// The per-call fp16 mirror of the int8 KV cache used by both prefill kernels.
//
// The cache stays int8 with one fp16 scale per 64 elements ("round 6 track b - qsa flash",
// delivered change: half4 scales per cell).  Every prefill tile reads each cache cell many
// times (each 64-cell chunk by every later 128-row tile of its group; each selected cell by
// every token that selects it), so the call dequantises every cell it can see exactly once,
// k^ = fp16(code * scale) with a single rounding, into a caller workspace that the tiles then
// stream through L2.
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

}  // namespace

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
