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
// One CTA (256 threads) per token; each warp issues the loads of all its rows (and the gains)
// before it uses any, so a CTA waits on one memory round trip.  The token's rd/2 rotation
// angles are formed once, in fp32 with the product's error recovered and a three-part 2 pi
// (rope_angle), then sincosf.  Then a warp per row: lane = 8 consecutive dims (one 16-byte load),
// the sum of squares by shuffles, the rotation partner (dim +- rd/2) on lane ^ (rd/16), and the
// quantiser's 64-element blocks on lanes 8b .. 8b+7.
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kPrepRows = kHeads + 2 * kGroups;  // 24 q rows, 2 k rows, 2 v rows per token

struct PrepCfg {
  float inv_hi[kD / 2], inv_lo[kD / 2];  // base^(-2i / rd) as a float pair hi + lo, i < rd / 2
  int rotary_dim, sec0, sec1;
  float eps;
};

// theta = p * (hi + lo) reduced to about [-pi, pi], all in fp32 (GB300's fp64 rate is low): the
// product's rounding error is recovered exactly with an fma, and 2 pi is split Cody-Waite style
// into C1 (8 significant bits, so k * C1 is exact for k < 2^16) + C2 + C3.  For positions up to
// 2^17 the result is within about 3e-7 of the exact angle modulo 2 pi.
__device__ __forceinline__ float rope_angle(int p, float hi, float lo) {
  const float P = (float)p;
  const float prod = P * hi;
  const float err = fmaf(P, hi, -prod) + P * lo;  // p * (hi + lo) - prod
  const float k = rintf(prod * 0.15915494309189535f);
  float r = fmaf(-k, 6.28125f, prod);  // exact: k * C1 has at most 22 significant bits
  r = fmaf(-k, 1.9353071795864769e-3f, r);
  r = fmaf(-k, 1.0253131677018246e-11f, r);
  return r + err;
}

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
  // this warp's rows r = warp + 8 j (j < 4, r < 28) and the gains: every load issued before any use
  constexpr int kRowsPerWarp = (kPrepRows + 7) / 8;
  uint4 raw[kRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 8 * j;
    raw[j] = make_uint4(0u, 0u, 0u, 0u);
    if (r < kPrepRows) {
      const __half* src = r >= kHeads + kGroups ? v_raw + ((size_t)t * kGroups + (r - kHeads - kGroups)) * kD
                          : r >= kHeads ? k_raw + ((size_t)t * kGroups + (r - kHeads)) * kD
                                        : q_raw + ((size_t)t * kHeads + r) * kD;
      raw[j] = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    }
  }
  const float4 qg0 = __ldg(reinterpret_cast<const float4*>(q_gamma) + 2 * lane);
  const float4 qg1 = __ldg(reinterpret_cast<const float4*>(q_gamma) + 2 * lane + 1);
  const float4 kg0 = __ldg(reinterpret_cast<const float4*>(k_gamma) + 2 * lane);
  const float4 kg1 = __ldg(reinterpret_cast<const float4*>(k_gamma) + 2 * lane + 1);
  if (tid < h2) {
    int p = pos0 + t;
    if (pos3) p = __ldg(pos3 + 3 * t + (tid < cfg.sec0 ? 0 : (tid < cfg.sec0 + cfg.sec1 ? 1 : 2)));
    float sn, cs;
    sincosf(rope_angle(p, cfg.inv_hi[tid], cfg.inv_lo[tid]), &sn, &cs);
    s_cs[tid] = make_float2(cs, sn);
  }
  __syncthreads();
  const int cell = pos0 + t;
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 8 * j;
    if (r >= kPrepRows) break;  // warp-uniform
    const bool is_v = r >= kHeads + kGroups, is_k = !is_v && r >= kHeads;
    const int g = is_v ? r - kHeads - kGroups : r - kHeads;  // group of a k or v row
    float x[8];
    {
      const __half2* h = reinterpret_cast<const __half2*>(&raw[j]);
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
      const float gw[8] = {is_k ? kg0.x : qg0.x, is_k ? kg0.y : qg0.y, is_k ? kg0.z : qg0.z, is_k ? kg0.w : qg0.w,
                           is_k ? kg1.x : qg1.x, is_k ? kg1.y : qg1.y, is_k ? kg1.z : qg1.z, is_k ? kg1.w : qg1.w};
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
  for (int i = 0; i < rotary_dim / 2; ++i) {
    const double inv = pow(base, -2.0 * i / rotary_dim);
    cfg.inv_hi[i] = (float)inv;
    cfg.inv_lo[i] = (float)(inv - (double)cfg.inv_hi[i]);
  }
  cfg.rotary_dim = rotary_dim;
  cfg.sec0 = sections[0];
  cfg.sec1 = sections[1];
  cfg.eps = eps;
  return launch_pdl(prep_kernel, dim3(T), dim3(256), 0, stream, q_raw, k_raw, v_raw, q_gamma, k_gamma, pos3, pos0, cfg,
                    qcur, kcur, kq, ksc, vq, vsc);
}

}  // namespace qsa
