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
// One CTA (256 threads, at most 48 registers: five CTAs per SM) per token; each warp issues the
// loads of all its rows before it uses any, so a CTA waits on one memory round trip, and the gains
// are read per row from L1.  More CTAs per SM hide more of that round trip: a persistent form that
// loads the next token's rows during the current one held fewer CTAs per SM and ran slower.  The token's rd/2 rotation
// angles are formed once, in fp32 with the product's error recovered and a three-part 2 pi
// (rope_angle), then sincosf, into shared memory; each lane then keeps its own four (cos, sin)
// pairs in registers for all the token's rows.  A warp takes a row at a time with the lanes laid
// out around the rotation: lane l < R = rd / 8 holds the four rotation pairs (4l + u, 4l + u + rd/2),
// lanes l >= R hold 8 consecutive unrotated dims rd + 8 (l - R) ..; so every lane holds 8 values in
// two 4-dim runs at dims (a, b), the rotation needs no exchange between lanes, and the row's
// sum of squares and the quantiser's four 64-element block maxima are warp reductions.
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

// Dims of this lane's two 4-dim runs (see above): (a, b) with values x[0..3] at a .. a + 3 and
// x[4..7] at b .. b + 3.
__device__ __forceinline__ void lane_dims(int lane, int rd, int& a, int& b) {
  const int R = rd >> 3;
  if (lane < R) {
    a = 4 * lane;
    b = a + (rd >> 1);
  } else {
    a = rd + 8 * (lane - R);
    b = a + 4;
  }
}

__device__ __forceinline__ void unpack4(uint2 w, float* x) {
  const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  x[0] = f0.x;
  x[1] = f0.y;
  x[2] = f1.x;
  x[3] = f1.y;
}

// The quantiser of qsa_prep_quantize on one 256-element row held as above: per 64-element block
// IEEE fp32 a / 127 rounded to fp16, codes round-half-away(x / s) clamped to +-127 (all zero and
// a +0 scale for an all-zero block).  The block maxima are reduced over the whole warp.
__device__ __forceinline__ void quantize_row(const float (&x)[8], int a, int b, int8_t* codes, __half* scales,
                                             int lane) {
  float m[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int blk = (u < 4 ? a : b) >> 6;  // a run never crosses a block (4-aligned, 64-element blocks)
    const float v = fabsf(x[u]);
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = (blk == k) ? fmaxf(m[k], v) : m[k];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], __shfl_xor_sync(0xffffffffu, m[k], o));
  __half sh[4];
  float sv[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    sh[k] = __float2half_rn(__fdiv_rn(m[k], 127.0f));
    sv[k] = __half2float(sh[k]);
  }
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int blk = (u < 4 ? a : b) >> 6;
    const float s = blk == 0 ? sv[0] : blk == 1 ? sv[1] : blk == 2 ? sv[2] : sv[3];
    int c = 0;
    if (s != 0.f) c = (int)fminf(fmaxf(roundf(__fdiv_rn(x[u], s)), -127.f), 127.f);
    w[u >> 2] |= (uint32_t)(uint8_t)(int8_t)c << (8 * (u & 3));
  }
  *reinterpret_cast<uint32_t*>(codes + a) = w[0];
  *reinterpret_cast<uint32_t*>(codes + b) = w[1];
  if (lane == 0) {
    __half o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = sv[k] == 0.f ? __ushort_as_half(0) : sh[k];
    *reinterpret_cast<uint2*>(scales) = *reinterpret_cast<const uint2*>(o);
  }
}

__global__ void __launch_bounds__(256, 5) prep_kernel(const __half* __restrict__ q_raw, const __half* __restrict__ k_raw,
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
  const bool rot_lane = lane < (rd >> 3);
  int da, db;
  lane_dims(lane, rd, da, db);
  // this warp's rows r = warp + 8 j (j < 4, r < 28) and the gains: every load issued before any use
  constexpr int kRowsPerWarp = (kPrepRows + 7) / 8;
  uint2 ra[kRowsPerWarp], rb[kRowsPerWarp];
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 8 * j;
    ra[j] = make_uint2(0u, 0u);
    rb[j] = make_uint2(0u, 0u);
    if (r < kPrepRows) {
      const __half* src = r >= kHeads + kGroups ? v_raw + ((size_t)t * kGroups + (r - kHeads - kGroups)) * kD
                          : r >= kHeads ? k_raw + ((size_t)t * kGroups + (r - kHeads)) * kD
                                        : q_raw + ((size_t)t * kHeads + r) * kD;
      ra[j] = __ldg(reinterpret_cast<const uint2*>(src + da));
      rb[j] = __ldg(reinterpret_cast<const uint2*>(src + db));
    }
  }
  if (tid < h2) {
    int p = pos0 + t;
    if (pos3) p = __ldg(pos3 + 3 * t + (tid < cfg.sec0 ? 0 : (tid < cfg.sec0 + cfg.sec1 ? 1 : 2)));
    float sn, cs;
    sincosf(rope_angle(p, cfg.inv_hi[tid], cfg.inv_lo[tid]), &sn, &cs);
    s_cs[tid] = make_float2(cs, sn);
  }
  __syncthreads();
  // this lane's four rotation pairs 4 lane + u (rotated lanes only)
  float2 cs4[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) cs4[u] = rot_lane ? s_cs[da + u] : make_float2(1.f, 0.f);
  const int cell = pos0 + t;
#pragma unroll
  for (int j = 0; j < kRowsPerWarp; ++j) {
    const int r = warp + 8 * j;
    if (r >= kPrepRows) break;  // warp-uniform
    const bool is_v = r >= kHeads + kGroups, is_k = !is_v && r >= kHeads;
    const int g = is_v ? r - kHeads - kGroups : r - kHeads;  // group of a k or v row
    float x[8];
    unpack4(ra[j], x);
    unpack4(rb[j], x + 4);
    if (!is_v) {
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) ss = fmaf(x[u], x[u], ss);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rs = 1.f / sqrtf(ss * (1.f / kD) + cfg.eps);
      const float* gam = is_k ? k_gamma : q_gamma;  // this lane's gains (L1-resident after the first CTAs)
      const float4 ga = __ldg(reinterpret_cast<const float4*>(gam + da));
      const float4 gb = __ldg(reinterpret_cast<const float4*>(gam + db));
      const float gw[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = x[u] * rs * gw[u];
      if (rot_lane) {  // pairs (x[u], x[4 + u]) = dims (a + u, a + u + rd / 2)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float lo = x[u], hi = x[4 + u];
          x[u] = lo * cs4[u].x - hi * cs4[u].y;
          x[4 + u] = hi * cs4[u].x + lo * cs4[u].y;
        }
      }
    }
    if (!is_k && !is_v) {  // qcur
      __half* dst = qcur + ((size_t)t * kHeads + r) * kD;
      *reinterpret_cast<uint2*>(dst + da) = make_uint2(pack_half2(x[0], x[1]), pack_half2(x[2], x[3]));
      *reinterpret_cast<uint2*>(dst + db) = make_uint2(pack_half2(x[4], x[5]), pack_half2(x[6], x[7]));
      continue;
    }
    if (is_k) {  // the cache holds the fp16 rounding of the k row, quantised
      uint32_t ow[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ow[u] = pack_half2(x[2 * u], x[2 * u + 1]);
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ow[u]));
        x[2 * u] = f.x;
        x[2 * u + 1] = f.y;
      }
      if (kcur) {
        __half* dst = kcur + ((size_t)t * kGroups + g) * kD;
        *reinterpret_cast<uint2*>(dst + da) = make_uint2(ow[0], ow[1]);
        *reinterpret_cast<uint2*>(dst + db) = make_uint2(ow[2], ow[3]);
      }
    }
    int8_t* codes = (is_k ? kq : vq) + ((size_t)cell * kGroups + g) * kD;
    __half* scale = (is_k ? ksc : vsc) + ((size_t)cell * kGroups + g) * kNB;
    quantize_row(x, da, db, codes, scale, lane);
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
