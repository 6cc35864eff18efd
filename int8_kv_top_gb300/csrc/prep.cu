// qsa_prep: the fused prep of T new tokens (the pages' qsa_prep, "round 27 track b - qsa prep
// and merge": decision and rejected prep fusion name its raw rows, gains, norm_rope step and mrope
// variants; correctness lists its outputs qcur, kq, vq, ksc, vsc).  The library's readings of
// the unstated formulas:
//   q, k rows: y = x / sqrt(mean(x^2) + eps) * gamma, then the rotary embedding with halves
//              paired (i, i + rd/2), theta_i = p * base^(-2i/rd) (mrope: p of the pair's section)
//              (y_i, y_{i+rd/2}) -> (y_i cos - y_{i+rd/2} sin, y_{i+rd/2} cos + y_i sin)
//   outputs:   qcur = fp16(q rows); kcur = fp16(k rows) (optional); the cache cell pos0 + t gets
//              quantise(kcur) and quantise(v rows), the absmax rule of qsa_prep_quantize.
//
// One CTA (256 threads) per token.  The token's rd/2 rotation angles are formed once: the
// angle p * inv_freq_i in fp64 (inv_freq from a host-built fp64 table), reduced modulo 2 pi in
// fp64, then sincosf in fp32 (positions up to 65,536 keep the angle to about 1e-7 rad).  Then a
// warp per row: lane = 8 consecutive dims (one 16-byte load), the sum of squares by shuffles,
// the rotation partner (dim +- rd/2) on lane ^ (rd/16), and the quantiser's 64-element blocks
// on lanes 8b .. 8b+7.
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kPrepRows = kHeads + 2 * kGroups;  // 24 q rows, 2 k rows, 2 v rows per token

struct PrepCfg {
  double inv_freq[kD / 2];  // base^(-2i / rd), i < rd / 2
  int rotary_dim, sec0, sec1;
  float eps;
};

// The quantiser of qsa_prep_quantize, on a lane's 8 values of a 64-element block held by the
// 8 lanes 8b .. 8b+7: IEEE fp32 a / 127 rounded to fp16, codes round-half-away(x / s) clamped.
__device__ __forceinline__ void quantize8(const float (&x)[8], int8_t* dst_codes, __half* dst_scale, int lane) {
  float a = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) a = fmaxf(a, fabsf(x[u]));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const __half sh = __float2half_rn(__fdiv_rn(a, 127.0f));
  const float s = __half2float(sh);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    int c = 0;
    if (s != 0.f) c = (int)fminf(fmaxf(roundf(__fdiv_rn(x[u], s)), -127.f), 127.f);
    w[u >> 2] |= (uint32_t)(uint8_t)(int8_t)c << (8 * (u & 3));
  }
  *reinterpret_cast<uint2*>(dst_codes) = make_uint2(w[0], w[1]);
  if ((lane & 7) == 0) *dst_scale = (s == 0.f) ? __ushort_as_half(0) : sh;
}

__global__ void __launch_bounds__(256) prep_kernel(const __half* __restrict__ q_raw, const __half* __restrict__ k_raw,
                                                   const __half* __restrict__ v_raw, const float* __restrict__ q_gamma,
                                                   const float* __restrict__ k_gamma, const int32_t* __restrict__ pos3,
                                                   int pos0, const __grid_constant__ PrepCfg cfg,
                                                   __half* __restrict__ qcur, __half* __restrict__ kcur,
                                                   int8_t* __restrict__ kq, __half* __restrict__ ksc,
                                                   int8_t* __restrict__ vq, __half* __restrict__ vsc) {
  __shared__ float2 s_cs[kD / 2];  // (cos, sin) of pair i
  pdl_begin();
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rd = cfg.rotary_dim, h2 = rd / 2;
  if (tid < h2) {
    int p = pos0 + t;
    if (pos3) p = __ldg(pos3 + 3 * t + (tid < cfg.sec0 ? 0 : (tid < cfg.sec0 + cfg.sec1 ? 1 : 2)));
    const double ang = (double)p * cfg.inv_freq[tid];
    const double k = rint(ang * 0.15915494309189535);                         // 1 / (2 pi)
    const double red = fma(-k, 2.4492935982947064e-16, fma(-k, 6.283185307179586, ang));  // ang - 2 pi k
    float sn, cs;
    sincosf((float)red, &sn, &cs);
    s_cs[tid] = make_float2(cs, sn);
  }
  __syncthreads();
  const int cell = pos0 + t;
  for (int r = warp; r < kPrepRows; r += 8) {
    const bool is_v = r >= kHeads + kGroups, is_k = !is_v && r >= kHeads;
    const int g = is_v ? r - kHeads - kGroups : r - kHeads;  // group of a k or v row
    const __half* src = is_v ? v_raw + ((size_t)t * kGroups + g) * kD
                             : (is_k ? k_raw + ((size_t)t * kGroups + g) * kD : q_raw + ((size_t)t * kHeads + r) * kD);
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    float x[8];
    {
      const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 f = __half22float2(h[u]);
        x[2 * u] = f.x;
        x[2 * u + 1] = f.y;
      }
    }
    if (!is_v) {
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) ss = fmaf(x[u], x[u], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rs = 1.f / sqrtf(ss * (1.f / kD) + cfg.eps);
      const float* gam = is_k ? k_gamma : q_gamma;
      const float4 g0 = __ldg(reinterpret_cast<const float4*>(gam) + 2 * lane);
      const float4 g1 = __ldg(reinterpret_cast<const float4*>(gam) + 2 * lane + 1);
      const float gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = x[u] * rs * gw[u];
      // rotation: dims 8 lane + u < rd pair with dim +- h2 on lane ^ (rd / 16)
      const int d0 = 8 * lane;
      float other[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) other[u] = __shfl_xor_sync(0xffffffffu, x[u], rd >> 4);
      if (d0 < rd) {
        const bool first = d0 < h2;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float2 c = s_cs[(d0 + u) & (h2 - 1)];
          x[u] = first ? x[u] * c.x - other[u] * c.y : x[u] * c.x + other[u] * c.y;
        }
      }
    }
    if (!is_k && !is_v) {  // qcur
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int u = 0; u < 4; ++u) ow[u] = pack_half2(x[2 * u], x[2 * u + 1]);
      *reinterpret_cast<uint4*>(qcur + ((size_t)t * kHeads + r) * kD + 8 * lane) = o;
      continue;
    }
    if (is_k) {  // the cache holds the fp16 rounding of the k row, quantised
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ow[u] = pack_half2(x[2 * u], x[2 * u + 1]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ow[u]));
        x[2 * u] = f.x;
        x[2 * u + 1] = f.y;
      }
      if (kcur) *reinterpret_cast<uint4*>(kcur + ((size_t)t * kGroups + g) * kD + 8 * lane) = o;
    }
    int8_t* codes = (is_k ? kq : vq) + ((size_t)cell * kGroups + g) * kD + 8 * lane;
    __half* scale = (is_k ? ksc : vsc) + ((size_t)cell * kGroups + g) * kNB + (lane >> 3);
    quantize8(x, codes, scale, lane);
  }
}

}  // namespace

cudaError_t launch_prep(const __half* q_raw, const __half* k_raw, const __half* v_raw, const float* q_gamma,
                        const float* k_gamma, const int32_t* pos3, int T, int pos0, double base, int rotary_dim,
                        float eps, const int* sections, __half* qcur, __half* kcur, int8_t* kq, __half* ksc,
                        int8_t* vq, __half* vsc, cudaStream_t stream) {
  PrepCfg cfg{};
  for (int i = 0; i < rotary_dim / 2; ++i) cfg.inv_freq[i] = pow(base, -2.0 * i / rotary_dim);
  cfg.rotary_dim = rotary_dim;
  cfg.sec0 = sections[0];
  cfg.sec1 = sections[1];
  cfg.eps = eps;
  return launch_pdl(prep_kernel, dim3(T), dim3(256), 0, stream, q_raw, k_raw, v_raw, q_gamma, k_gamma, pos3, pos0, cfg,
                    qcur, kcur, kq, ksc, vq, vsc);
}

}  // namespace qsa
