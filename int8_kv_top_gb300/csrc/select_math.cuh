// Exact integer arithmetic of the selection score, shared by the selection kernels
// (select.cu) and the fused decode layer (decode_fused.cu).
//
// Every fp16 value is an integer multiple of 2^-24, so the sum over a group's 12 query heads
// (Qsum) is an exact 64-bit integer in those units, and 2^48 * score / sm_scale =
// sum_b (ksc_b 2^24) * sum_{d in b} (Qsum_d 2^24) kq_d is an exact 128-bit integer.  The fast
// scores use Qsum split as hi = fp16(Qsum) and lo = fp16(Qsum - hi), whose products with int8
// codes are exact in fp32; the residual Qsum - hi - lo enters the error bound.
#pragma once
#include "common.cuh"

namespace qsa {

// fp16 value times 2^24 as an exact integer (finite values).
__device__ __forceinline__ long long half_int24(uint16_t h) {
  const int e = (h >> 10) & 31, m = h & 1023;
  const long long v = (e == 0) ? (long long)m : ((long long)(1024 + m) << (e - 1));
  return (h & 0x8000) ? -v : v;
}

// Round an exact integer multiple of 2^-24 (a = |value| * 2^24) to fp16, nearest-even.
// Returns the fp16 magnitude bits and sets *r to the rounded magnitude in the same units.
// Magnitudes below 2048 units are fp16 values already (subnormal below 1024, e = 1 above)
// and their bit pattern is the integer itself; above, 11 significant bits are kept.
__device__ __forceinline__ uint32_t units_to_half_mag(unsigned long long a, unsigned long long* r) {
  if (a < 2048ull) {
    *r = a;
    return (uint32_t)a;
  }
  int s = 53 - __clzll((long long)a);  // bit length - 11 (>= 1)
  unsigned long long mant = a >> s;
  const unsigned long long rem = a & ((1ull << s) - 1), half = 1ull << (s - 1);
  if (rem > half || (rem == half && (mant & 1ull))) ++mant;
  if (mant == 2048ull) {
    mant = 1024ull;
    ++s;
  }
  const int e = s + 1;  // value = mant * 2^(e - 25), biased exponent e
  if (e > 30) {         // beyond the fp16 range: infinity, like a rounding conversion
    *r = a;
    return 0x7C00u;
  }
  *r = mant << s;
  return ((uint32_t)e << 10) | (uint32_t)(mant - 1024ull);
}

__device__ __forceinline__ __half signed_half(uint32_t mag_bits, bool neg) {
  return __ushort_as_half((unsigned short)(mag_bits | (neg ? 0x8000u : 0u)));
}

// Qsum_d = sum of the group's 12 query heads at dim d for token t (exact, units of 2^-24), split
// into hi = fp16(Qsum) and lo = fp16(Qsum - hi); e = |Qsum - hi - lo| and h = |hi| + |lo|;
// `exact` receives Qsum itself.  All arithmetic is exact in 64-bit integers: Qsum of 12 fp16
// values is below 2^44 units, and block sums of |residual| and |hi| + |lo| stay below 2^51.
__device__ __forceinline__ void qsum_split_exact(const __half* __restrict__ q, int t, int g, int d, __half& hi, __half& lo,
                                           long long& e, long long& h_abs, long long& exact) {
  const uint16_t* qt = reinterpret_cast<const uint16_t*>(q) + ((size_t)t * kHeads + g * kHPG) * kD;
  long long sum = 0;
#pragma unroll
  for (int h = 0; h < kHPG; ++h) sum += half_int24(__ldg(qt + h * kD + d));
  unsigned long long rh, rl;
  const bool neg = sum < 0;
  const uint32_t hb = units_to_half_mag((unsigned long long)(neg ? -sum : sum), &rh);
  hi = signed_half(hb, neg);
  const long long rest = sum - (neg ? -(long long)rh : (long long)rh);  // exact
  const bool neg2 = rest < 0;
  const uint32_t lb = units_to_half_mag((unsigned long long)(neg2 ? -rest : rest), &rl);
  lo = signed_half(lb, neg2);
  e = rest - (neg2 ? -(long long)rl : (long long)rl);  // exact residual
  if (e < 0) e = -e;
  h_abs = (long long)rh + (long long)rl;
  exact = sum;
}

__device__ __forceinline__ void qsum_split(const __half* __restrict__ q, int t, int g, int d, __half& hi, __half& lo,
                                           long long& e, long long& h_abs) {
  long long exact;
  qsum_split_exact(q, t, g, d, hi, lo, e, h_abs, exact);
}

}  // namespace qsa
