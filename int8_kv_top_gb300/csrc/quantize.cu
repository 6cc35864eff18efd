// qsa_prep_quantize: fp16 rows -> int8 codes + one fp16 scale per 64 elements.
//
// The pages' fused prep kernel writes the int8 cache buffers (kq vq ksc vsc) but never
// states the quantiser ("round 27 track b - qsa prep and merge", correctness and
// rejected prep fusion).  This is the symmetric absmax rule: per 64-element block
// a = max |x|, scale = fp16_rn(a / 127) with the division in IEEE fp32,
// code = clamp(round-half-away(x / scale) in IEEE fp32, -127, 127); scale 0 -> codes 0.
//
// One warp per block of 64 elements, two elements per lane.
#include "common.cuh"

namespace qsa {
namespace {

__global__ void __launch_bounds__(256) quantize_kernel(const __half* __restrict__ x, int64_t n_blocks,
                                                       int8_t* __restrict__ xq, __half* __restrict__ xsc) {
  pdl_begin();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t blk = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < n_blocks; blk += warps) {
    const __half2 v2 = *reinterpret_cast<const __half2*>(x + blk * kBlk + lane * 2);
    const float x0 = __low2float(v2), x1 = __high2float(v2);
    float a = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const __half sh = __float2half_rn(__fdiv_rn(a, 127.0f));
    const float s = __half2float(sh);
    int c0 = 0, c1 = 0;
    if (s != 0.f) {
      c0 = (int)fminf(fmaxf(roundf(__fdiv_rn(x0, s)), -127.f), 127.f);
      c1 = (int)fminf(fmaxf(roundf(__fdiv_rn(x1, s)), -127.f), 127.f);
    }
    const uint16_t packed = (uint16_t)((uint8_t)(int8_t)c0 | ((uint16_t)(uint8_t)(int8_t)c1 << 8));
    *reinterpret_cast<uint16_t*>(xq + blk * kBlk + lane * 2) = packed;
    if (lane == 0) xsc[blk] = (s == 0.f) ? __ushort_as_half(0) : sh;
  }
}

}  // namespace

cudaError_t launch_quantize(const __half* x, int64_t n_rows, int8_t* xq, __half* xsc, cudaStream_t stream) {
  const int64_t n_blocks = n_rows * kNB;
  if (n_blocks == 0) return cudaSuccess;
  const int64_t want = (n_blocks + 7) / 8;
  const int grid = (int)(want < 152 * 32 ? want : 152 * 32);
  return launch_pdl(quantize_kernel, dim3(grid), dim3(256), 0, stream, x, n_blocks, xq, xsc);
}

}  // namespace qsa
