// qsa_select: per-(token, group) top-k cell selection with an exact ranking.
//
// The pages split selection into qsa_score (per-token, per-cell scores; "round 27 track b
// - qsa prep and merge", decision: it unrolls its four-value dot products) and qsa_topk,
// skipped below the 2051/2052 budget boundary ("round 6 track b - qsa flash", experiment
// contract and delivered change).  The score of cell c for token t and group g is the sum
// over the group's 12 heads of sm_scale * q . k^, equal scores going to the lower index.
//
// GB300 design (four launches on the caller's stream; calls with at most kSmallRows selected
// rows use two, score_small_kernel in place of 1 and 2):
//  1. prep_q:  Qsum = sum_h q over the group's 12 heads, exact in 64-bit integers, split as
//              hi = fp16(Qsum), lo = fp16(Qsum - hi); per 64-dim block the residual norm
//              E_b = sum |Qsum - hi - lo| and H_b = sum (|hi| + |lo|).
//     prep_k:  int8 K codes as fp16 (exact integers) for every cell a selected token can
//              see, and kmax_b = max |ksc| per group and block.
//  2. score:   tcgen05 GEMM with one TMEM accumulator per 64-dim scale block:
//                S_b[t][c] = sum_{d in b} (hi + lo)[t][d] * kq[c][d]   (products exact in fp32)
//              epilogue  s~[t][c] = fp16(sm_scale * sum_b ksc[c][b] * S_b[t][c]).
//              128-row x 128-cell tiles; B is staged one 64-dim block at a time in a TMA-fed
//              ring, and each block's accumulator is released as soon as the epilogue has
//              loaded it.
//  3. topk:    one 512-thread CTA per (token, group) holds the row's scores in registers.
//              |s~ - s| <= a + b|s~| rigorously (a: fp16 rounding of Qsum and fp32
//              accumulation, from E_b, H_b, kmax; b: fp16 storage), and U(f) = f + a + b|f|,
//              L(f) = f - a - b|f| are increasing, so with tau = the k-th largest s~, cells
//              with L(s~) > U(tau) are surely in, cells with U(s~) < L(tau) surely out.
//              tau is found from a sampled bracket, one compare pass and an exact radix
//              select inside the bracket (full radix passes when the bracket misses).  The
//              band between is re-scored with EXACT integer keys (every fp16 value is an
//              integer multiple of 2^-24, so 2^48 * score / sm_scale = sum_b (ksc_b 2^24) *
//              sum_{d in b} (Qsum_d 2^24) kq_d, in 128-bit integers) and resolved by (key
//              desc, index asc); a band beyond shared-memory capacity takes an exact radix
//              select over recomputed keys.  Ids are emitted in ascending order.
#include "common.cuh"
#include "select_math.cuh"

namespace qsa {
namespace {

// ----------------------------------------------------------------- workspace layout
constexpr int kGM = 128, kGN = 128, kGK = 64, kGStages = 4;
constexpr int kMaxCells = 65536;
constexpr int kTkThreads = 512;
static_assert(kTkThreads >= 256, "top-k stages a 256-entry histogram and 256 Qsum dims one per thread");
constexpr int kCandCap = 2048;
constexpr int kBandCap = 512;
// hist 2 KB | qsum (padded) | band keys + ids | candidate ids + keys | selection bitmap | staged band rows
constexpr int kSmallRows = 8;   // calls with at most this many selected rows score on the CUDA cores
constexpr int kStageRows = 64;  // band cells whose code rows are staged in shared memory at once
// Staged code rows are kD + 16 bytes apart, so the four cells a warp keys at once start in
// different banks.
constexpr int kStageStride = kD + 16;
// Qsum_d sits at slot d + d / 32: the 8 lanes that form one cell's exact key read dims 32 j + t
// (j = 0..7) at the same time, which without the pad would all fall in one bank.
constexpr int kQsumSlots = kD + kD / 32;
constexpr int kOffBandKey = 2048 + kQsumSlots * 8;  // 4160, 16-byte aligned
constexpr int kTopkSmem = kOffBandKey + kBandCap * 20 + kCandCap * 6 + kMaxCells / 8 + kStageRows * (kStageStride + 8);

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  int t_sel, T_sel, T_pad, n_max, n_pad;
  size_t off_kmax, off_hist1, zero_bytes, off_eh, off_qhi, off_kc, off_scores, total;
};

WsLayout ws_layout(int T, int pos0, Params p) {
  WsLayout L{};
  L.t_sel = first_selected_token(pos0, p.identity_max);
  L.T_sel = T > L.t_sel ? T - L.t_sel : 0;
  L.T_pad = (int)align_up((size_t)L.T_sel, kGM);
  L.n_max = pos0 + T;  // largest n_kv of the call
  L.n_pad = (int)align_up((size_t)L.n_max, 256);
  size_t o = 0;
  L.off_kmax = o;
  L.off_hist1 = o + 8 * sizeof(float);
  // few-row calls: per (group, row) 256-bin histograms of the scores' high key bytes, which
  // score_small_kernel fills for topk_kernel; zeroed together with kmax
  const size_t hist_bytes = L.T_sel <= kSmallRows ? (size_t)kGroups * L.T_sel * 256 * sizeof(unsigned) : 0;
  L.zero_bytes = 8 * sizeof(float) + hist_bytes;
  o = align_up(o + L.zero_bytes, 1024);
  L.off_eh = o;
  o = align_up(o + (size_t)kGroups * L.T_sel * 8 * sizeof(float), 1024);
  L.off_qhi = o;
  o = align_up(o + (size_t)kGroups * L.T_pad * kD * 2 * 2, 1024);  // hi and lo
  L.off_kc = o;
  o = align_up(o + (size_t)kGroups * L.n_pad * kD * 2, 1024);
  L.off_scores = o;
  o = align_up(o + (size_t)kGroups * L.T_sel * L.n_pad * 2, 1024);
  L.total = o;
  return L;
}

// ----------------------------------------------------------------- 1. prep
// prep_q: grid (T_pad, 2), 256 threads: thread = dim.  Row layout of qhl: for each 64-dim block
// b, [hi_b (64) | lo_b (64)] at columns 128 b .. 128 b + 127, with Qsum = hi + lo + residual.
//
// E_b = sum |residual| and H_b = sum (|hi| + |lo|) over each 64-dim block (two warps), one
// row, 256 threads (thread = dim); threads 0-3 write eh[0..3] = E_b and eh[4..7] = H_b.
__device__ __forceinline__ void write_eh(long long e, long long h_abs, float* __restrict__ eh_row,
                                         long long* s_e, long long* s_h) {
  const int d = threadIdx.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    e += __shfl_xor_sync(0xffffffffu, e, o);
    h_abs += __shfl_xor_sync(0xffffffffu, h_abs, o);
  }
  if ((d & 31) == 0) {
    s_e[d >> 5] = e;
    s_h[d >> 5] = h_abs;
  }
  __syncthreads();
  if (d < kNB) {
    constexpr float kUnit = 5.9604644775390625e-8f;  // 2^-24, exact scaling
    eh_row[d] = __ll2float_ru(s_e[2 * d] + s_e[2 * d + 1]) * kUnit;
    eh_row[kNB + d] = __ll2float_ru(s_h[2 * d] + s_h[2 * d + 1]) * kUnit;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(256) prep_q_kernel(const __half* __restrict__ q, int t_sel, int T_sel, int T_pad,
                                                     __half* __restrict__ qhl, float* __restrict__ eh) {
  pdl_begin();
  const int r = blockIdx.x, g = blockIdx.y, d = threadIdx.x;
  __half hi = __ushort_as_half(0), lo = __ushort_as_half(0);
  long long e = 0, h_abs = 0;
  if (r < T_sel) qsum_split(q, t_sel + r, g, d, hi, lo, e, h_abs);
  __half* dst = qhl + ((size_t)g * T_pad + r) * (2 * kD) + (d >> 6) * 128 + (d & 63);
  dst[0] = hi;
  dst[64] = lo;
  if (r >= T_sel) return;
  __shared__ long long s_e[8], s_h[8];
  write_eh(e, h_abs, eh + ((size_t)g * T_sel + r) * 8, s_e, s_h);
}

// grid (min(n_pad / 8, kPrepKCtas), 2), 256 threads: a warp per cell row (lane = 8 codes),
// CTAs striding over the rows.  Each CTA reduces its |ksc| maxima before one atomic per
// scale block.
constexpr int kPrepKCtas = 1024;
__global__ void __launch_bounds__(256) prep_k_kernel(const int8_t* __restrict__ kq, const __half* __restrict__ ksc,
                                                     int n_max, int n_pad, __half* __restrict__ kc,
                                                     float* __restrict__ kmax) {
  pdl_begin();
  const int g = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = lane >> 3;
  float amax = 0.f;
  for (int c = blockIdx.x * 8 + warp; c < n_pad; c += gridDim.x * 8) {
    uint4 outw = make_uint4(0, 0, 0, 0);
    if (c < n_max) {
      const uint2 w = *reinterpret_cast<const uint2*>(kq + ((size_t)c * kGroups + g) * kD + lane * 8);
      uint32_t o[4];
      dequant8(w.x, w.y, __half2half2(__ushort_as_half(0x3C00)), o);  // scale 1: exact codes
      outw = make_uint4(o[0], o[1], o[2], o[3]);
      if ((lane & 7) == 0) amax = fmaxf(amax, fabsf(__half2float(ksc[((size_t)c * kGroups + g) * kNB + blk])));
    }
    *reinterpret_cast<uint4*>(kc + ((size_t)g * n_pad + c) * kD + lane * 8) = outw;
  }
  __shared__ float s_max[8][kNB];
  if ((lane & 7) == 0) s_max[warp][blk] = amax;
  __syncthreads();
  if (threadIdx.x < kNB) {
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_max[w][threadIdx.x]);
    atomicMax(reinterpret_cast<int*>(kmax) + g * kNB + threadIdx.x, __float_as_int(m));
  }
}

// ----------------------------------------------------------------- 2. score GEMM
// CTA: 128 rows x nt_per_cta tiles of 128 cells.  TMEM holds one M128 x N128 fp32 accumulator per
// 64-dim scale block (4 x 128 columns).  The B operand is staged one 64-dim block at a time
// ([128 cells][64] SW128, 16 KB) in a kGStages ring; per block the MMA issuer runs hi_b then
// lo_b against the same codes (8 K16 steps) and commits that block's accumulator.  The epilogue
// frees each block's accumulator as soon as it has loaded it, so the next tile's MMAs on block b
// wait only for that load, not for the whole epilogue: no second accumulator set is needed.
constexpr int kNtPerCtaMax = 16;               // at most 2048 cells per CTA
constexpr int kSmemA = kGM * kD * 2 * 2;       // 128 KB: 8 k-blocks (hi_b, lo_b) of [128 rows][64] SW128
constexpr int kSmemBStage = kGN * kGK * 2;     // 16 KB: one 64-dim block of [128 cells][64] SW128
constexpr int kSmemStg = kGM * kGN * 2;          // 32 KB: the tile's fp16 scores, 2 boxes of [128 rows][64] SW128
constexpr int kScoreSmem = kSmemA + kGStages * kSmemBStage + kSmemStg + 1024;

struct __align__(8) ScoreBars {
  uint64_t a_full, b_full[kGStages], b_empty[kGStages], acc_full[kNB], acc_empty[kNB], drain;
};

constexpr int kScoreThreads = 384;  // warp 0 TMA, warp 1 MMA, warps 4-11 epilogue

__device__ __forceinline__ void epilogue_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__global__ void __launch_bounds__(kScoreThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 const __grid_constant__ CUtensorMap map_s, const __half* __restrict__ ksc, int T_sel, int T_pad, int n_pad,
                 int n_base, int m_tiles, int n_chunks, int nt_per_cta, float sm_scale, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ ScoreBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int per_g = m_tiles * n_chunks;
  const int g = blockIdx.x / per_g;
  const int m = (blockIdx.x % per_g) / n_chunks, nch = blockIdx.x % n_chunks;
  const int r0 = m * kGM;
  const int r_last = min(r0 + kGM, T_sel) - 1;
  const int n_kv_hi = n_base + r_last + 1;  // cells the tile's last row can see
  const int nt_begin = nch * nt_per_cta;
  const int nt_end = min(nt_begin + nt_per_cta, (n_kv_hi + kGN - 1) / kGN);
  const int n_tiles = nt_end - nt_begin;
  if (n_tiles <= 0) {  // uniform over the CTA, before any allocation
    pdl_begin();         // still waits, so the grid never completes ahead of the kernel before it
    return;
  }

  if (tid == 0) {
    s_abort = 0;
    mbar_init(&bars.a_full, 1);
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(&bars.b_full[i], 1);
      mbar_init(&bars.b_empty[i], 1);
    }
    for (int b = 0; b < kNB; ++b) {
      mbar_init(&bars.acc_full[b], 1);
      mbar_init(&bars.acc_empty[b], 8);  // the 8 epilogue warps, once they have loaded block b
    }
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_begin();
  uint8_t* sA = smem;
  uint8_t* sB = smem + kSmemA;
  const int n_blocks = n_tiles * kNB;  // B stages this CTA consumes: (tile, 64-dim block)

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&map_a);
      tma_prefetch_desc(&map_b);
      mbar_arrive_expect_tx(&bars.a_full, kSmemA);
      for (int kb = 0; kb < 2 * kD / kGK; ++kb)
        tma_load_2d(sA + kb * (kGM * 128), &map_a, &bars.a_full, kb * kGK, g * T_pad + r0);
      int issued = 0;
      for (int j = 0; j < n_blocks; ++j) {
        const int st = j % kGStages;
        if (j >= kGStages && !mbar_wait(&bars.b_empty[st], ((j / kGStages) & 1) ^ 1, status, &s_abort)) break;
        mbar_arrive_expect_tx(&bars.b_full[st], kSmemBStage);
        tma_load_2d(sB + st * kSmemBStage, &map_b, &bars.b_full[st], (j % kNB) * kGK,
                    g * n_pad + (nt_begin + j / kNB) * kGN);
        issued = j + 1;
      }
      mbar_wait(&bars.a_full, 0, status);
      for (int j = max(0, issued - kGStages); j < issued; ++j)
        mbar_wait(&bars.b_full[j % kGStages], (j / kGStages) & 1, status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kGM, kGN, 0, 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      bool ok = mbar_wait(&bars.a_full, 0, status, &s_abort);
      tc_fence_after();
      const uint64_t ad0 = sdesc_sw128(a0, 16, 1024);
      for (int j = 0; ok && j < n_blocks; ++j) {
        const int i = j / kNB, b = j % kNB, st = j % kGStages;
        if (i >= 1 && !mbar_wait(&bars.acc_empty[b], (i - 1) & 1, status, &s_abort)) { ok = false; break; }
        if (!mbar_wait(&bars.b_full[st], (j / kGStages) & 1, status, &s_abort)) { ok = false; break; }
        tc_fence_after();
        const uint64_t bd0 = sdesc_sw128(b0 + st * kSmemBStage, 16, 1024);
#pragma unroll
        for (int part = 0; part < 2; ++part)  // hi_b then lo_b against the same codes
#pragma unroll
          for (int kk = 0; kk < kGK / 16; ++kk)
            umma_ss(tmem + b * kGN, ad0 + (uint64_t)(((2 * b + part) * (kGM * 128) + kk * 32) >> 4),
                    bd0 + (uint64_t)((kk * 32) >> 4), idesc, (part > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars.b_empty[st]);
        umma_commit(&bars.acc_full[b]);
      }
      umma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0, status);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // epilogue: warps 4-7 take cells 0-63 of each 128-cell tile, warps 8-11 cells 64-127; thread
    // = row.  The tile's K scales of group g are staged (fp16, block-major) before the tile, so that
    // a block's 64 cells come in as eight 16-byte broadcast loads.  The scores go to a 128B-swizzled
    // shared-memory tile that one thread stores with two TMA box stores: the warps do not wait on
    // global stores, and cells past a row's causal end (inside its padded width, never read) and
    // rows past T_sel (clipped by the tensor map) need no masking.
    __shared__ __align__(16) __half s_scale[kNB][kGN];
    const int quarter = warp & 3, c0 = (warp >= 8) ? 64 : 0;
    const int et = tid - 128;  // 0..255
    const int rl = quarter * 32 + lane;  // tile row
    const int n_lim = n_base + T_sel;  // cells that exist for this call
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* stg_row = smem + kSmemA + kGStages * kSmemBStage + (c0 >> 6) * (kGM * 128) + rl * 128;
    bool dead = false;  // after a failed wait keep meeting the epilogue barriers, skip the work
    auto load_scales = [&](int i, __half (&dst)[2]) {  // this thread stages two scales per tile
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int e = et + 256 * x, cell = e >> 2, b = e & 3;
        const int c = (nt_begin + i) * kGN + cell;
        dst[x] = (i < n_tiles && c < n_lim) ? ksc[((size_t)c * kGroups + g) * kNB + b] : __ushort_as_half(0);
      }
    };
    __half sc_next[2];
    load_scales(0, sc_next);
    for (int i = 0; i < n_tiles; ++i) {
      const int n0 = (nt_begin + i) * kGN;
#pragma unroll
      for (int x = 0; x < 2; ++x) {  // s_scale is free: every thread passed the previous tile's barrier A
        const int e = et + 256 * x;
        s_scale[e & 3][e >> 2] = sc_next[x];
      }
      load_scales(i + 1, sc_next);  // one tile ahead: the loads overlap this tile's work
      epilogue_bar();
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
#pragma unroll
      for (int b = 0; b < kNB; ++b) {
        if (!dead) dead = !mbar_wait_warp(&bars.acc_full[b], i & 1, status, &s_abort);
        if (dead) continue;
        tc_fence_after();
        uint32_t v[2][32];
        tmem_ld32(lane_base + b * kGN + c0, v[0]);
        tmem_ld32(lane_base + b * kGN + c0 + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.acc_empty[b]);  // the next tile's block-b MMAs may start
        const uint4* sv = reinterpret_cast<const uint4*>(&s_scale[b][c0]);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const uint4 s8 = sv[q8];
          const uint32_t sw[4] = {s8.x, s8.y, s8.z, s8.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&sw[u]));
            const int j = 8 * q8 + 2 * u;
            acc[j] = fmaf(f.x, __uint_as_float(v[j >> 5][j & 31]), acc[j]);
            acc[j + 1] = fmaf(f.y, __uint_as_float(v[(j + 1) >> 5][(j + 1) & 31]), acc[j + 1]);
          }
        }
      }
      // barrier A: every thread is done with s_scale, and the previous tile's store has read the
      // staging tile
      if (et == 0 && i > 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      epilogue_bar();
      if (!dead) {
        // this thread's 64 scores: 128 B of row rl in box c0 / 64, 16-byte chunks swizzled by rl mod 8
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const int j = 8 * ch;
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(stg_row + ((ch ^ (rl & 7)) << 4))),
                       "r"(pack_half2(acc[j] * sm_scale, acc[j + 1] * sm_scale)),
                       "r"(pack_half2(acc[j + 2] * sm_scale, acc[j + 3] * sm_scale)),
                       "r"(pack_half2(acc[j + 4] * sm_scale, acc[j + 5] * sm_scale)),
                       "r"(pack_half2(acc[j + 6] * sm_scale, acc[j + 7] * sm_scale))
                       : "memory");
        }
      }
      fence_proxy_async_smem();  // the staging writes are visible to the TMA engine
      epilogue_bar();            // barrier B: the whole tile is staged
      if (et == 0) {
        const uint8_t* stg = smem + kSmemA + kGStages * kSmemBStage;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb)
          asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                           reinterpret_cast<uint64_t>(&map_s)),
                       "r"(n0 + 64 * hb), "r"(r0), "r"(g), "r"(smem_u32(stg + hb * (kGM * 128)))
                       : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
    }
    // every score store has completed before the CTA leaves
    if (et == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// Unsigned key with the order of the fp16 values (finite values and -inf).
__device__ __forceinline__ uint32_t fp16_order_key(uint16_t b) {
  return (b & 0x8000u) ? (uint32_t)(~b & 0xFFFFu) : (uint32_t)(b | 0x8000u);
}

// ----------------------------------------------------------------- 2b. score for few rows
// Decode-sized calls (at most kSmallRows selected rows) have no GEMM to feed the tensor
// cores, so the same scores are computed on the CUDA cores straight from the int8 codes:
// per 64-dim block S_b = sum over the block of (hi + lo) * kq in fp32 (128 exact products,
// summed in a different order than the MMA but within the same bound), then
// s~ = fp16(sm_scale * fma(ksc_3, S_3, fma(ksc_2, S_2, fma(ksc_1, S_1, ksc_0 * S_0)))),
// the epilogue of the GEMM.  The kernel also takes kmax_b = max |ksc| (prep_k's job on the
// GEMM path), and for each row the 256-bin histogram of the high byte of its scores' order keys
// over the row's causal cells (counted in shared memory, one global atomic per non-empty bin),
// so that topk_kernel starts from the k-th largest score's bin.  grid (ceil(n_max / 64), 2),
// 256 threads: warp = 8 cells, lane = 8 dims.
__global__ void __launch_bounds__(256) score_small_kernel(const int8_t* __restrict__ kq, const __half* __restrict__ ksc,
                                                          const __half* __restrict__ q, int t_sel, int T_sel, int n_max,
                                                          int n_pad, int n_base, float sm_scale,
                                                          __half* __restrict__ scores, float* __restrict__ kmax,
                                                          unsigned* __restrict__ hist1, float* __restrict__ eh) {
  __shared__ __align__(16) float s_hl[kSmallRows][2 * kD];  // per row: [hi_b | lo_b] per block b
  __shared__ float s_max[8][kNB];
  __shared__ unsigned s_h1[kSmallRows][256];
  __shared__ long long s_e[8], s_h[8];
  pdl_begin();
  const int g = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < T_sel * 256; i += 256) s_h1[i >> 8][i & 255] = 0u;
  // the rows' Qsum hi/lo split (prep_q's arithmetic), thread = dim, all rows' loads in flight
  // together; CTA 0 also writes E_b, H_b
  long long e[kSmallRows], h_abs[kSmallRows];
  {
    const int d = threadIdx.x;
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r) {
      e[r] = 0;
      h_abs[r] = 0;
      if (r < T_sel) {
        __half hi, lo;
        qsum_split(q, t_sel + r, g, d, hi, lo, e[r], h_abs[r]);
        s_hl[r][(d >> 6) * 128 + (d & 63)] = __half2float(hi);
        s_hl[r][(d >> 6) * 128 + 64 + (d & 63)] = __half2float(lo);
      }
    }
  }
  if (blockIdx.x == 0) {
#pragma unroll
    for (int r = 0; r < kSmallRows; ++r)
      if (r < T_sel) write_eh(e[r], h_abs[r], eh + ((size_t)g * T_sel + r) * 8, s_e, s_h);
  }
  __syncthreads();
  const int blk = lane >> 3;
  const int col = blk * 128 + (lane & 7) * 8;  // this lane's 8 hi values; lo at +64
  float amax = 0.f;
  // the warp's 8 cells: codes and scales all loaded before any use, so their latencies overlap
  uint2 wk[8];
  __half hs[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = min(blockIdx.x * 64 + warp * 8 + i, n_max - 1);  // clamped: rows past n_max are not used
    wk[i] = __ldg(reinterpret_cast<const uint2*>(kq + ((size_t)c * kGroups + g) * kD + lane * 8));
    hs[i] = ksc[((size_t)c * kGroups + g) * kNB + blk];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = blockIdx.x * 64 + warp * 8 + i;
    if (c >= n_max) break;  // uniform over the warp
    const uint2 w = wk[i];
    float kf[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      kf[j] = (float)(int8_t)(w.x >> (8 * j));
      kf[4 + j] = (float)(int8_t)(w.y >> (8 * j));
    }
    const float my_sc = __half2float(hs[i]);
    amax = fmaxf(amax, fabsf(my_sc));
    const float sc0 = __shfl_sync(0xffffffffu, my_sc, 0), sc1 = __shfl_sync(0xffffffffu, my_sc, 8);
    const float sc2 = __shfl_sync(0xffffffffu, my_sc, 16), sc3 = __shfl_sync(0xffffffffu, my_sc, 24);
    for (int r = 0; r < T_sel; ++r) {
      const float4* hp = reinterpret_cast<const float4*>(&s_hl[r][col]);
      const float4 h0 = hp[0], h1 = hp[1], l0 = hp[16], l1 = hp[17];  // lo = hi + 64 floats
      float p = h0.x * kf[0];
      p = fmaf(h0.y, kf[1], p);
      p = fmaf(h0.z, kf[2], p);
      p = fmaf(h0.w, kf[3], p);
      p = fmaf(h1.x, kf[4], p);
      p = fmaf(h1.y, kf[5], p);
      p = fmaf(h1.z, kf[6], p);
      p = fmaf(h1.w, kf[7], p);
      p = fmaf(l0.x, kf[0], p);
      p = fmaf(l0.y, kf[1], p);
      p = fmaf(l0.z, kf[2], p);
      p = fmaf(l0.w, kf[3], p);
      p = fmaf(l1.x, kf[4], p);
      p = fmaf(l1.y, kf[5], p);
      p = fmaf(l1.z, kf[6], p);
      p = fmaf(l1.w, kf[7], p);
      p += __shfl_xor_sync(0xffffffffu, p, 1);
      p += __shfl_xor_sync(0xffffffffu, p, 2);
      p += __shfl_xor_sync(0xffffffffu, p, 4);  // S_b on every lane of block b
      const float S0 = __shfl_sync(0xffffffffu, p, 0), S1 = __shfl_sync(0xffffffffu, p, 8);
      const float S2 = __shfl_sync(0xffffffffu, p, 16), S3 = __shfl_sync(0xffffffffu, p, 24);
      float acc = fmaf(sc0, S0, 0.f);
      acc = fmaf(sc1, S1, acc);
      acc = fmaf(sc2, S2, acc);
      acc = fmaf(sc3, S3, acc);
      if (lane == 0) {
        const __half sv = __float2half_rn(acc * sm_scale);
        scores[((size_t)g * T_sel + r) * n_pad + c] = sv;
        if (c < n_base + r + 1) atomicAdd(&s_h1[r][fp16_order_key(__half_as_ushort(sv)) >> 8], 1u);
      }
    }
  }
  if ((lane & 7) == 0) s_max[warp][blk] = amax;
  __syncthreads();
  if (threadIdx.x < kNB) {
    float m = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = fmaxf(m, s_max[w][threadIdx.x]);
    atomicMax(reinterpret_cast<int*>(kmax) + g * kNB + threadIdx.x, __float_as_int(m));
  }
  for (int i = threadIdx.x; i < T_sel * 256; i += 256) {
    const unsigned v = s_h1[i >> 8][i & 255];
    if (v) atomicAdd(hist1 + ((size_t)g * T_sel + (i >> 8)) * 256 + (i & 255), v);
  }
}

// ----------------------------------------------------------------- 3. top-k
struct Key128 {
  long long hi;
  unsigned long long lo;
};
__device__ __forceinline__ Key128 split128(__int128 k) { return {(long long)(k >> 64), (unsigned long long)k}; }
__device__ __forceinline__ bool key_gt(Key128 a, Key128 b) { return a.hi != b.hi ? a.hi > b.hi : a.lo > b.lo; }
__device__ __forceinline__ bool key_eq(Key128 a, Key128 b) { return a.hi == b.hi && a.lo == b.lo; }

// Exact key of cell c: sum_b ksc_b 2^24 * sum_{d in b} qsum_d kq_d  (qsum in units of 2^-24).
__device__ __forceinline__ __int128 exact_key(const long long* __restrict__ s_qsum, const int8_t* __restrict__ krow,
                                              const __half* __restrict__ srow) {
  __int128 key = 0;
#pragma unroll 1
  for (int b = 0; b < kNB; ++b) {
    long long acc = 0;
    const int4* k16 = reinterpret_cast<const int4*>(krow + b * kBlk);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int4 w = __ldg(k16 + i);
      const int ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int by = 0; by < 4; ++by)
          acc += s_qsum[b * (kBlk + 2) + (i >> 1) + i * 16 + j * 4 + by] * (long long)(int8_t)(ws[j] >> (8 * by));
    }
    key += (__int128)half_int24(__half_as_ushort(srow[b])) * (__int128)acc;
  }
  return key;
}

__device__ __forceinline__ uint16_t key_to_bits(uint32_t k) {
  return (k & 0x8000u) ? (uint16_t)(k & 0x7FFFu) : (uint16_t)(~k & 0xFFFFu);
}
__device__ __forceinline__ float order_key_to_float(uint32_t k) {
  const uint16_t b = (k & 0x8000u) ? (uint16_t)(k & 0x7FFFu) : (uint16_t)(~k & 0xFFFFu);
  return __half2float(__ushort_as_half(b));
}

// Block-wide sum of one int per thread.
__device__ __forceinline__ int block_sum(int v, int* s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  int t = (lane < (int)(blockDim.x >> 5)) ? s_red[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

// Find the bin holding the `need`-th largest element given a 256-bin histogram in smem
// (bins scanned from high to low).  Returns the bin and sets *above = count in higher bins.
// One warp: the bin (counting down from 255) that holds the need-th largest element of `hist`,
// and how many elements lie in higher bins; bin -1 if there is none.  Lane l owns bins
// 255-8l .. 248-8l, read as two 16-byte words.
__device__ __forceinline__ void warp_find_bin(const unsigned* hist, int need, int lane, int& found, int& found_above) {
  const uint4* h4 = reinterpret_cast<const uint4*>(hist + 248 - 8 * lane);
  const uint4 lo4 = h4[0], hi4 = h4[1];  // bins 248-8l .. 251-8l, 252-8l .. 255-8l
  const int cnt[8] = {(int)hi4.w, (int)hi4.z, (int)hi4.y, (int)hi4.x, (int)lo4.w, (int)lo4.z, (int)lo4.y, (int)lo4.x};
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) sum += cnt[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int run = incl - sum;  // elements in higher bins than this lane's first
  found = -1;
  found_above = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (found < 0 && run < need && run + cnt[i] >= need) {
      found = 255 - 8 * lane - i;
      found_above = run;
    }
    run += cnt[i];
  }
  const unsigned who = __ballot_sync(0xffffffffu, found >= 0);
  if (who) {
    const int src = __ffs(who) - 1;
    found = __shfl_sync(0xffffffffu, found, src);
    found_above = __shfl_sync(0xffffffffu, found_above, src);
  }
}

// Block-wide: warp 0 searches, every thread gets the bin and the count above it.
__device__ __forceinline__ int find_bin_desc(const unsigned* hist, int need, int* above, int* s_tmp) {
  if (threadIdx.x < 32) {
    int f, fa;
    warp_find_bin(hist, need, threadIdx.x, f, fa);
    if (threadIdx.x == 0) {
      s_tmp[0] = f;
      s_tmp[1] = fa;
    }
  }
  __syncthreads();
  const int b = s_tmp[0];
  *above = s_tmp[1];
  __syncthreads();
  return b;
}

// Two independent searches at once: warp 0 on (h0, need0), warp 1 on (h1, need1).  A search whose
// use flag is false (uniform) reports bin -1 and 0 above.
__device__ __forceinline__ void find_bin_desc2(const unsigned* h0, int need0, bool use0, const unsigned* h1, int need1,
                                               bool use1, int* b0, int* above0, int* b1, int* above1, int* s_tmp) {
  const int w = threadIdx.x >> 5;
  if (w < 2) {
    int f = -1, fa = 0;
    if (w == 0 ? use0 : use1) warp_find_bin(w == 0 ? h0 : h1, w == 0 ? need0 : need1, threadIdx.x & 31, f, fa);
    if ((threadIdx.x & 31) == 0) {
      s_tmp[2 * w] = f;
      s_tmp[2 * w + 1] = fa;
    }
  }
  __syncthreads();
  *b0 = s_tmp[0];
  *above0 = s_tmp[1];
  *b1 = s_tmp[2];
  *above1 = s_tmp[3];
  __syncthreads();
}

// Histogram increment (shared-memory atomics resolve same-bin lanes in hardware).
__device__ __forceinline__ void warp_hist_add(bool pred, unsigned bin, unsigned* hist) {
  if (pred) atomicAdd(&hist[bin], 1u);
}

// Bounds of the score error: a (absolute) and b (relative to the stored fp16 value).
struct Bound {
  float a, b;
  __device__ float U(float f) const { return f + a + b * fabsf(f); }
  __device__ float L(float f) const { return f - a - b * fabsf(f); }
};

// Block-wide exclusive prefix sum; returns this thread's offset and the total.
__device__ __forceinline__ int block_excl_scan(int v, int* s_red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) s_red[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? s_red[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_red[32 + lane] = w;  // inclusive over warps
  }
  __syncthreads();
  *total = s_red[32 + 31];
  return x - v + (warp > 0 ? s_red[32 + warp - 1] : 0);
}

// 8-bit mask of the halves of w (cell 8m + j -> bit j) that are >= th (cmp = 0) or > th (1).
// Each packed compare gives 0xFFFF per true half; bits 0 and 16 of compare i go to bits 2i and
// 16 + 2i, and one fold moves the high halves down to the odd bits 2i + 1.
__device__ __forceinline__ uint32_t mask8(const uint4& w, __half2 th, int strict) {
  const uint32_t* u = reinterpret_cast<const uint32_t*>(&w);
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = *reinterpret_cast<const __half2*>(&u[i]);
    const uint32_t x = strict ? __hgt2_mask(h, th) : __hge2_mask(h, th);
    m |= (x & 0x00010001u) << (2 * i);
  }
  return (m | (m >> 15)) & 0xFFu;
}

// Smallest finite order key k (0x0400 .. 0xFBFF) with pred(k), 0xFC00 if none; pred monotone
// (false .. true).  Called by all 32 lanes of a warp: each round tests 32 evenly spaced keys up to hi
// and keeps the gap where pred turns true, so four rounds cover the 63,488 finite keys.
template <class P>
__device__ uint32_t first_key_warp(P pred) {
  const uint32_t lane = threadIdx.x & 31u;
  uint32_t lo = 0x0400u, hi = 0xFBFFu;  // answer in [lo, hi] while pred(hi)
  if (!pred(hi)) return 0xFC00u;        // none (uniform: every lane evaluates the same key)
  while (lo < hi) {
    const uint32_t step = (hi - lo + 30u) / 31u;  // lane 31 reaches hi
    const uint32_t k = lo + lane * step;
    const unsigned b = __ballot_sync(0xffffffffu, k >= hi || pred(k));
    const uint32_t first = (uint32_t)__ffs(b) - 1u;  // exists: lanes past hi vote true
    if (first == 0u) return lo;                      // pred(lo)
    const uint32_t nhi = lo + first * step;
    lo = lo + (first - 1u) * step + 1u;              // pred false at lo + (first - 1) step
    hi = nhi < hi ? nhi : hi;
  }
  return lo;
}

// One 512-thread CTA per (token, group).  Thread tid owns cells [tid*V, tid*V + V) of the
// row in registers (fp16 pairs); every pass over the row is a packed fp16 compare against a
// threshold, because the error-band tests are monotone in the stored score.
template <int V>
__global__ void __launch_bounds__(kTkThreads, (V <= 64 ? 2 : 1))
    topk_kernel(const __half* __restrict__ scores, const __half* __restrict__ q, const int8_t* __restrict__ kq,
                const __half* __restrict__ ksc, const float* __restrict__ eh, const float* __restrict__ kmax,
                const unsigned* __restrict__ hist1, int32_t* __restrict__ ids, int t_sel, int T_sel, int n_pad,
                int pos0, int K, float sm_scale, int* status) {
  pdl_begin();
  extern __shared__ __align__(16) uint8_t topk_smem[];
  unsigned* s_hist = reinterpret_cast<unsigned*>(topk_smem);                   // [2][256]
  long long* s_qsum = reinterpret_cast<long long*>(topk_smem + 2048);          // [kQsumSlots], padded
  Key128* s_band_key = reinterpret_cast<Key128*>(topk_smem + kOffBandKey);     // [kBandCap]
  int* s_band_idx = reinterpret_cast<int*>(s_band_key + kBandCap);             // [kBandCap]
  int* s_cand_idx = s_band_idx + kBandCap;                                     // [kCandCap]
  uint16_t* s_cand_key = reinterpret_cast<uint16_t*>(s_cand_idx + kCandCap);   // [kCandCap]
  unsigned* s_bits = reinterpret_cast<unsigned*>(s_cand_key + kCandCap);       // [kMaxCells / 32]
  int8_t* s_stage = reinterpret_cast<int8_t*>(s_bits + kMaxCells / 32);          // [kStageRows][kStageStride] codes
  uint2* s_stage_sc = reinterpret_cast<uint2*>(s_stage + kStageRows * kStageStride);  // [kStageRows] 4 fp16 scales
  __shared__ int s_red[64];
  __shared__ int s_tmp[8];
  __shared__ int s_cnt[2];          // 0: candidates, 1: band
  __shared__ uint32_t s_thr[2];     // order keys: surely-in threshold, band threshold
  __shared__ Bound s_bound;

  // rows are taken last-written first: the score kernel writes group 1's last rows last, and those
  // are the ones most likely still in L2 when the first wave of this kernel starts
  const int r = gridDim.x - 1 - blockIdx.x, g = gridDim.y - 1 - blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nwarps = kTkThreads / 32;
  const int t = t_sel + r;
  const int n_kv = pos0 + t + 1;
  const __half* row = scores + ((size_t)g * T_sel + r) * n_pad;
  // few-row calls: the row's high-byte histogram, loaded now so its latency overlaps the row's
  const unsigned h1_pre = (hist1 != nullptr && tid < 256) ? __ldg(hist1 + ((size_t)g * T_sel + r) * 256 + tid) : 0u;

  if (tid < kD) {  // exact Qsum in units of 2^-24
    long long sq = 0;
    const __half* qt = q + ((size_t)t * kHeads + g * kHPG) * kD + tid;
#pragma unroll
    for (int h = 0; h < kHPG; ++h) sq += half_int24(__half_as_ushort(qt[h * kD]));
    s_qsum[tid + (tid >> 5)] = sq;
  }
  for (int i = tid; i < 512; i += kTkThreads) s_hist[i] = 0u;
  for (int i = tid; i < (n_kv + 31) / 32; i += kTkThreads) s_bits[i] = 0u;
  if (tid == 0) {
    // |s~ - s| <= a + b |s~|: a covers the residual of Qsum after its fp16 hi + lo split
    // (E_b) and the fp32 accumulation of 128 exact products per block (128 * 2^-23 of the
    // absolute sum, with |kq| <= 128) plus the epilogue's roundings (2^-21); b covers the
    // fp16 rounding of the stored score.  Both doubled for margin.
    const float* e = eh + ((size_t)g * T_sel + r) * 8;
    float acc = 0.f;
    for (int b = 0; b < kNB; ++b) acc += kmax[g * kNB + b] * (e[b] + e[kNB + b] * (1.5258789e-05f + 4.7683716e-07f));
    s_bound.a = 2.f * (sm_scale * 128.f * acc + 1.2e-7f);
    s_bound.b = 2.f * 4.8852e-04f;
    s_cnt[0] = 0;
    s_cnt[1] = 0;
  }

  // this thread's cells in registers; cells past n_kv read as -inf
  uint4 w[V / 8];
  const int c0 = tid * V;
#pragma unroll
  for (int m = 0; m < V / 8; ++m) {
    const int c = c0 + 8 * m;
    uint4 x = make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);
    if (c < n_kv) {
      x = __ldg(reinterpret_cast<const uint4*>(row + c));
      if (c + 8 > n_kv) {
        uint16_t* hh = reinterpret_cast<uint16_t*>(&x);
        for (int j = 0; j < 8; ++j)
          if (c + j >= n_kv) hh[j] = 0xFC00u;
      }
    }
    w[m] = x;
  }
  auto half_bits = [](const uint4& x, int j) -> uint16_t {  // select chain: no local-memory indexing
    const int wd = j >> 1;
    const uint32_t v = wd == 0 ? x.x : wd == 1 ? x.y : wd == 2 ? x.z : x.w;
    return (uint16_t)(v >> (16 * (j & 1)));
  };
  __syncthreads();

  // ---- tau: bracket from a 1-in-8 sample (cells 0, 8, 16, ...), then one compare pass
  const int n_samp = (n_kv + 7) / 8;
  uint32_t key_hi = 0xFBFFu, key_lo = 0x0400u;  // finite range
  // with the row's high-byte histogram given (few-row calls), the k-th largest key is found
  // from it directly and no bracket is needed
  bool bracket = hist1 == nullptr && n_samp >= 64;
  if (bracket) {
    const float ks = (float)K * n_samp / n_kv;
    const int margin = (int)(3.f * sqrtf(ks) + 16.f);
    const int r_hi = (int)ks - margin;  // sample ranks (1-based) bracketing the k-th largest
    const int r_lo = (int)ceilf(ks) + margin;
#pragma unroll
    for (int m = 0; m < V / 8; ++m)
      warp_hist_add(c0 + 8 * m < n_kv, fp16_order_key(half_bits(w[m], 0)) >> 8, s_hist);
    __syncthreads();
    int ab_hi = 0, ab_lo = 0, b_hi = -1, b_lo = -1;
    find_bin_desc2(s_hist, r_hi, r_hi >= 1, s_hist, r_lo, r_lo <= n_samp, &b_hi, &ab_hi, &b_lo, &ab_lo, s_tmp);
    for (int i = tid; i < 512; i += kTkThreads) s_hist[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int m = 0; m < V / 8; ++m) {
      const bool v = c0 + 8 * m < n_kv;
      const uint32_t k = fp16_order_key(half_bits(w[m], 0));
      warp_hist_add(v && (int)(k >> 8) == b_hi, k & 0xFFu, s_hist);
      warp_hist_add(v && (int)(k >> 8) == b_lo, k & 0xFFu, s_hist + 256);
    }
    __syncthreads();
    int f_hi, f_lo, dummy0, dummy1;
    find_bin_desc2(s_hist, r_hi - ab_hi, b_hi >= 0, s_hist + 256, r_lo - ab_lo, b_lo >= 0, &f_hi, &dummy0, &f_lo, &dummy1,
                   s_tmp);
    if (b_hi >= 0) key_hi = ((uint32_t)b_hi << 8) | (uint32_t)f_hi;
    if (b_lo >= 0) key_lo = ((uint32_t)b_lo << 8) | (uint32_t)f_lo;
    key_hi = min(key_hi, 0xFBFFu);
    key_lo = max(key_lo, 0x0400u);
  }
  int above = 0;
  if (bracket) {
    const __half2 thi = __half2half2(__ushort_as_half(key_to_bits(key_hi)));
    const __half2 tlo = __half2half2(__ushort_as_half(key_to_bits(key_lo)));
    // key_lo <= key <= key_hi (padding is -inf): 8-cell masks packed four to a register
    uint32_t in[(V / 8 + 3) / 4] = {};
    int n = 0;
#pragma unroll
    for (int m = 0; m < V / 8; ++m) {
      const uint32_t gt = mask8(w[m], thi, 1);
      above += __popc(gt);
      const uint32_t msk = mask8(w[m], tlo, 0) & ~gt;
      in[m >> 2] |= msk << (8 * (m & 3));
      n += __popc(msk);
    }
    // one scan and one shared-memory atomic per warp: lanes take consecutive ranges of slots
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (tot) {  // warp-uniform
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_cnt[0], tot);
      int slot = __shfl_sync(0xffffffffu, base, 0) + incl - n;
#pragma unroll
      for (int m = 0; m < V / 8; ++m) {
        uint32_t bits = (in[m >> 2] >> (8 * (m & 3))) & 0xFFu;
        while (bits) {
          const int j = __ffs(bits) - 1;
          bits &= bits - 1;
          if (slot < kCandCap) {
            s_cand_idx[slot] = c0 + 8 * m + j;
            s_cand_key[slot] = (uint16_t)fp16_order_key(half_bits(w[m], j));
          }
          ++slot;
        }
      }
    }
  }
  const int A0 = bracket ? block_sum(above, s_red) : 0;
  const int Cn = s_cnt[0];
  const int need_c = K - A0;
  bracket = bracket && Cn <= kCandCap && need_c >= 1 && need_c <= Cn;
  for (int i = tid; i < 512; i += kTkThreads) s_hist[i] = 0u;
  __syncthreads();
  // exact order key of the k-th largest score: among the candidates, or over the whole row
  uint32_t tau_key;
  {
    int ab1, ab2, b1, b2;
    if (bracket) {
      for (int base = warp * 32; base < Cn; base += kTkThreads) {
        const int i = base + lane;
        warp_hist_add(i < Cn, i < Cn ? (uint32_t)s_cand_key[i] >> 8 : 0u, s_hist);
      }
      __syncthreads();
      b1 = find_bin_desc(s_hist, need_c, &ab1, s_tmp);
      for (int base = warp * 32; base < Cn; base += kTkThreads) {
        const int i = base + lane;
        const uint32_t k = i < Cn ? (uint32_t)s_cand_key[i] : 0u;
        warp_hist_add(i < Cn && (int)(k >> 8) == b1, k & 0xFFu, s_hist + 256);
      }
      __syncthreads();
      b2 = find_bin_desc(s_hist + 256, need_c - ab1, &ab2, s_tmp);
    } else if (hist1 != nullptr) {
      if (tid < 256) s_hist[tid] = h1_pre;
      __syncthreads();
      b1 = find_bin_desc(s_hist, K, &ab1, s_tmp);
      // low byte of the keys in bin b1, from the row held in registers
#pragma unroll
      for (int m = 0; m < V / 8; ++m) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t k = fp16_order_key(half_bits(w[m], j));
          if (c0 + 8 * m + j < n_kv && (int)(k >> 8) == b1) atomicAdd(&s_hist[256 + (k & 0xFFu)], 1u);
        }
      }
      __syncthreads();
      b2 = find_bin_desc(s_hist + 256, K - ab1, &ab2, s_tmp);
    } else {
      for (int c = tid; c < n_kv; c += kTkThreads) atomicAdd(&s_hist[fp16_order_key(__half_as_ushort(row[c])) >> 8], 1u);
      __syncthreads();
      b1 = find_bin_desc(s_hist, K, &ab1, s_tmp);
      for (int c = tid; c < n_kv; c += kTkThreads) {
        const uint32_t k = fp16_order_key(__half_as_ushort(row[c]));
        if ((int)(k >> 8) == b1) atomicAdd(&s_hist[256 + (k & 0xFFu)], 1u);
      }
      __syncthreads();
      b2 = find_bin_desc(s_hist + 256, K - ab1, &ab2, s_tmp);
    }
    if (b1 < 0 || b2 < 0) {  // cannot happen with K <= n_kv; leave the row unwritten
      if (tid == 0) set_dev_status(status, QSA_DEV_BAND_OVERFLOW);
      return;
    }
    tau_key = ((uint32_t)b1 << 8) | (uint32_t)b2;
  }

  // ---- thresholds: surely in <=> key >= k_def, undecided <=> k_band <= key < k_def
  if (warp < 2) {  // the two thresholds are searched by two warps at once
    const Bound bd = s_bound;
    const float tau = order_key_to_float(tau_key);
    const float Ut = bd.U(tau), Lt = bd.L(tau);
    const uint32_t kt = warp == 0 ? first_key_warp([&](uint32_t k) { return bd.L(order_key_to_float(k)) > Ut; })
                                  : first_key_warp([&](uint32_t k) { return bd.U(order_key_to_float(k)) >= Lt; });
    if (lane == 0) s_thr[warp] = kt;
  }
  __syncthreads();
  const uint32_t k_def = s_thr[0], k_band = s_thr[1];
  // the bracket is usable only if everything above it is surely in and below it surely out
  bracket = bracket && k_def <= key_hi + 1u && k_band >= key_lo;
  int n_def = 0;
  if (bracket) {
    for (int i = tid; i < Cn; i += kTkThreads) {
      const int c = s_cand_idx[i];
      const uint32_t k = s_cand_key[i];
      if (k >= k_def) {
        ++n_def;
      } else if (k >= k_band) {
        const int slot = atomicAdd(&s_cnt[1], 1);
        if (slot < kBandCap) s_band_idx[slot] = c;
      }
    }
  } else {
    const __half2 tdef = __half2half2(__ushort_as_half(key_to_bits(min(k_def, 0xFBFFu))));
    const __half2 tband = __half2half2(__ushort_as_half(key_to_bits(k_band)));
#pragma unroll
    for (int m = 0; m < V / 8; ++m) {
      const uint32_t def = (k_def <= 0xFBFFu) ? mask8(w[m], tdef, 0) : 0u;
      n_def += __popc(def);
      uint32_t bnd = mask8(w[m], tband, 0) & ~def;
      while (bnd) {
        const int j = __ffs(bnd) - 1;
        bnd &= bnd - 1;
        const int slot = atomicAdd(&s_cnt[1], 1);
        if (slot < kBandCap) s_band_idx[slot] = c0 + 8 * m + j;
      }
    }
  }
  const int A = (bracket ? A0 : 0) + block_sum(n_def, s_red);
  const int B = s_cnt[1];
  const int need = K - A;  // 1 <= need <= B by construction

  if (B <= kBandCap) {
    // exact keys: the band cells' code rows and scales are staged in shared memory by the
    // whole CTA in one round of copies (kStageRows at a time), then a warp per cell (lane = 8
    // codes of block lane / 8) forms the 64-bit block sums and the 128-bit key
    for (int i0 = 0; i0 < B; i0 += kStageRows) {
      const int nb = min(kStageRows, B - i0);
      for (int x = tid; x < nb * 16; x += kTkThreads) {
        const int c = s_band_idx[i0 + (x >> 4)];
        cp_async16(s_stage + (x >> 4) * kStageStride + (x & 15) * 16,
                   kq + ((size_t)c * kGroups + g) * kD + (x & 15) * 16);
      }
      for (int x = tid; x < nb; x += kTkThreads) {
        const int c = s_band_idx[i0 + x];
        s_stage_sc[x] = *reinterpret_cast<const uint2*>(ksc + ((size_t)c * kGroups + g) * kNB);
      }
      cp_async_wait_all();
      __syncthreads();
      // four cells per warp, 8 lanes per cell: lane j of a cell takes dims 32 j .. 32 j + 31 (two
      // lanes per 64-dim block); the four block terms sc_b * S_b (128-bit) are formed on four
      // lanes at once and summed across them
      const int cs = lane >> 3, j = lane & 7;
      for (int ib = warp * 4; ib < nb; ib += nwarps * 4) {
        const int i = ib + cs;
        const bool have = i < nb;
        long long part0 = 0, part1 = 0;
        if (have) {
          const uint4* src = reinterpret_cast<const uint4*>(s_stage + i * kStageStride + j * 32);
          const uint4 xa = src[0], xb = src[1];
          const uint32_t wv[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
          const long long* qs = s_qsum + j * 33;  // dims 32 j .. 32 j + 31 (padded slots)
#pragma unroll
          for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int by = 0; by < 4; by += 2) {
              part0 += qs[4 * u + by] * (long long)(int8_t)(wv[u] >> (8 * by));
              part1 += qs[4 * u + by + 1] * (long long)(int8_t)(wv[u] >> (8 * by + 8));
            }
        }
        long long part = part0 + part1;
        part += __shfl_xor_sync(0xffffffffu, part, 1);  // S_b on both lanes of block b = j / 2
        __int128 k128 = 0;
        if (have && (j & 1) == 0) {
          const uint2 sw = s_stage_sc[i];
          const uint32_t word = (j >> 2) ? sw.y : sw.x;
          k128 = (__int128)half_int24((uint16_t)(word >> (16 * ((j >> 1) & 1)))) * part;
        }
        // sum the four block terms of the cell (lanes j = 0, 2, 4, 6)
#pragma unroll
        for (int o = 2; o <= 4; o <<= 1) {
          const unsigned long long lo = (unsigned long long)k128;
          const long long hi = (long long)(k128 >> 64);
          const unsigned long long lo2 = __shfl_xor_sync(0xffffffffu, lo, o);
          const long long hi2 = __shfl_xor_sync(0xffffffffu, hi, o);
          k128 += (__int128)(((unsigned __int128)(unsigned long long)hi2 << 64) | lo2);
        }
        if (have && j == 0) s_band_key[i0 + i] = split128(k128);
      }
      __syncthreads();  // the staging area is reused by the next round
    }
    // rank of each band cell by (key desc, index asc): a warp per cell, lanes over the band
    for (int i = warp; i < B; i += nwarps) {
      const Key128 ki = s_band_key[i];
      const int ci = s_band_idx[i];
      int rank = 0;
      for (int jj = lane; jj < B; jj += 32) {
        const Key128 kj = s_band_key[jj];
        rank += key_gt(kj, ki) || (key_eq(kj, ki) && s_band_idx[jj] < ci);
      }
      rank = __reduce_add_sync(0xffffffffu, rank);
      if (lane == 0 && rank < need) atomicOr(&s_bits[ci >> 5], 1u << (ci & 31));
    }
  } else {
    // large band (many near-ties): exact radix select over the band, keys recomputed per
    // pass, 16 passes of 8 bits over the biased 128-bit key (cells read from the score row)
    auto in_band = [&](int c) -> bool {
      const uint32_t k = fp16_order_key(__half_as_ushort(row[c]));
      return k >= k_band && k < k_def;
    };
    auto bkey = [&](int c) -> unsigned __int128 {
      unsigned __int128 kb = (unsigned __int128)exact_key(s_qsum, kq + ((size_t)c * kGroups + g) * kD,
                                                          ksc + ((size_t)c * kGroups + g) * kNB);
      return kb ^ ((unsigned __int128)1 << 127);
    };
    unsigned __int128 pre = 0;
    int rem = need;
    for (int pass = 0; pass < 16; ++pass) {
      for (int i = tid; i < 256; i += kTkThreads) s_hist[i] = 0u;
      __syncthreads();
      const int shift = 120 - 8 * pass;
      for (int c = tid; c < n_kv; c += kTkThreads) {
        if (!in_band(c)) continue;
        const unsigned __int128 kb = bkey(c);
        if (pass == 0 || (kb >> (shift + 8)) == (pre >> (shift + 8))) atomicAdd(&s_hist[(unsigned)(kb >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      int ab;
      const int bin = find_bin_desc(s_hist, rem, &ab, s_tmp);
      rem -= ab;
      pre |= (unsigned __int128)(unsigned)bin << shift;
    }
    // every band key above pre, and the `rem` lowest-index cells equal to it: warp w scans
    // the contiguous range [w * span, (w + 1) * span), so ties are met in index order
    __shared__ int s_wsum[nwarps];
    const int span = (n_kv + nwarps - 1) / nwarps;
    const int cb = warp * span, ce = min(n_kv, cb + span);
    int my_ties = 0;
    for (int base = cb; base < ce; base += 32) {
      const int c = base + lane;
      const bool tie = c < ce && in_band(c) && bkey(c) == pre;
      my_ties += __popc(__ballot_sync(0xffffffffu, tie));
    }
    if (lane == 0) s_wsum[warp] = my_ties;
    __syncthreads();
    int before = 0;
    for (int x = 0; x < warp; ++x) before += s_wsum[x];
    for (int base = cb; base < ce; base += 32) {
      const int c = base + lane;
      bool gt = false, tie = false;
      if (c < ce && in_band(c)) {
        const unsigned __int128 kb = bkey(c);
        gt = kb > pre;
        tie = kb == pre;
      }
      const unsigned mm = __ballot_sync(0xffffffffu, tie);
      const int rank = before + __popc(mm & ((1u << lane) - 1u));
      before += __popc(mm);
      if (gt || (tie && rank < rem)) atomicOr(&s_bits[c >> 5], 1u << (c & 31));
    }
  }
  __syncthreads();

  // ---- emit ascending ids: surely-in cells (key >= k_def) plus the chosen band cells
  const __half2 tdef = __half2half2(__ushort_as_half(key_to_bits(min(k_def, 0xFBFFu))));
  uint32_t keep[V / 8];
  int n_keep = 0;
#pragma unroll
  for (int m = 0; m < V / 8; ++m) {
    const int c = c0 + 8 * m;
    uint32_t k = (k_def <= 0xFBFFu) ? mask8(w[m], tdef, 0) : 0u;
    if (c < n_kv) k |= (s_bits[c >> 5] >> (c & 31)) & 0xFFu;
    keep[m] = k;
    n_keep += __popc(k);
  }
  int total;
  int pos = block_excl_scan(n_keep, s_red, &total);
  if (total != K && tid == 0) set_dev_status(status, QSA_DEV_BAND_OVERFLOW);
  int32_t* dst = ids + ((size_t)t * kGroups + g) * K;
#pragma unroll
  for (int m = 0; m < V / 8; ++m) {
    uint32_t k = keep[m];
    while (k) {
      const int j = __ffs(k) - 1;
      k &= k - 1;
      if (pos < K) dst[pos] = c0 + 8 * m + j;
      ++pos;
    }
  }
}

// 3D map over the score matrix [2][T_sel][n_pad] fp16: box = 64 cells x 128 rows x 1 group, 128B
// swizzle (the staged tile's layout); rows past T_sel are clipped on store.
bool make_scores_map(CUtensorMap* map, void* base, int n_pad, int T_sel) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)n_pad, (cuuint64_t)T_sel, (cuuint64_t)kGroups};
  const cuuint64_t strides[2] = {(cuuint64_t)n_pad * 2, (cuuint64_t)n_pad * 2 * (cuuint64_t)T_sel};
  const cuuint32_t box[3] = {64u, (cuuint32_t)kGM, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool make_2d_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                 uint32_t box_outer) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The score GEMM: CTAs of 128 rows x nt_per_cta 128-cell tiles (one CTA per SM).  nt_per_cta is
// the one in [4, kNtPerCtaMax] with the shortest span in tile times, ceil(CTAs / SMs) x nt_per_cta,
// so that the last wave of CTAs is nearly full.
cudaError_t launch_score_gemm(const WsLayout& L, int pos0, __half* qhi, __half* kc, const __half* ksc, __half* sc,
                              float sm_scale, int* status, cudaStream_t stream) {
  // per device, set once (0 = not yet): the shared-memory attribute is set and the SM count read;
  // threads that race here both set the same attribute and store the same count
  static std::atomic<int> n_sms[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  cudaError_t e;
  int sms = n_sms[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    if ((e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScoreSmem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (sms < 1) return cudaErrorInvalidConfiguration;
    n_sms[dev].store(sms, std::memory_order_release);
  }
  CUtensorMap ma, mb, ms;
  if (!make_2d_map(&ma, qhi, 2 * kD, (uint64_t)kGroups * L.T_pad, kGK, kGM) ||
      !make_2d_map(&mb, kc, kD, (uint64_t)kGroups * L.n_pad, kGK, kGN) || !make_scores_map(&ms, sc, L.n_pad, L.T_sel))
    return cudaErrorInvalidValue;
  const int m_tiles = L.T_pad / kGM;
  const int n_tiles = L.n_pad / kGN;
  int nt_per = kNtPerCtaMax;
  long long best = -1;
  for (int x = kNtPerCtaMax; x >= 4; --x) {
    const long long ctas = (long long)kGroups * m_tiles * ((n_tiles + x - 1) / x);
    const long long span = (ctas + sms - 1) / sms * x;
    if (best < 0 || span < best) {
      best = span;
      nt_per = x;
    }
  }
  const int n_chunks = (n_tiles + nt_per - 1) / nt_per;
  const int n_base = pos0 + L.t_sel;  // n_kv of selected row r is n_base + r + 1
  return launch_pdl(score_kernel, dim3(kGroups * m_tiles * n_chunks), dim3(kScoreThreads), kScoreSmem, stream, ma, mb,
                    ms, ksc, L.T_sel, L.T_pad, L.n_pad, n_base, m_tiles, n_chunks, nt_per, sm_scale, status);
}

}  // namespace

int select_max_cells() { return kMaxCells; }

size_t select_workspace_bytes(int T, int pos0, int n_cells, Params p) {
  (void)n_cells;
  const WsLayout L = ws_layout(T, pos0, p);
  if (L.T_sel == 0) return 0;
  if (L.n_max > kMaxCells || p.topk > kMaxCells) return 0;  // row (fp16) must fit in shared memory
  return L.total;
}

cudaError_t launch_select(const __half* q, const int8_t* kq, const __half* ksc, int n_cells, int T, int pos0,
                          int32_t* ids, void* ws, Params p, int* status, cudaStream_t stream) {
  (void)n_cells;
  const WsLayout L = ws_layout(T, pos0, p);
  if (L.T_sel == 0) return cudaSuccess;
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* kmax = reinterpret_cast<float*>(base + L.off_kmax);
  float* eh = reinterpret_cast<float*>(base + L.off_eh);
  __half* qhi = reinterpret_cast<__half*>(base + L.off_qhi);
  __half* kc = reinterpret_cast<__half*>(base + L.off_kc);
  __half* sc = reinterpret_cast<__half*>(base + L.off_scores);

  unsigned* hist1 = reinterpret_cast<unsigned*>(base + L.off_hist1);
  cudaError_t e = cudaMemsetAsync(kmax, 0, L.zero_bytes, stream);  // kmax and (few-row calls) the histograms
  if (e != cudaSuccess) return e;
  if (L.T_sel <= kSmallRows) {  // the few-rows path forms the Qsum split itself
    e = launch_pdl(score_small_kernel, dim3((L.n_max + 63) / 64, kGroups), dim3(256), 0, stream, kq, ksc, q, L.t_sel,
                   L.T_sel, L.n_max, L.n_pad, pos0 + L.t_sel, p.sm_scale, sc, kmax, hist1, eh);
    if (e != cudaSuccess) return e;
  } else {
    e = launch_pdl(prep_q_kernel, dim3(L.T_pad, kGroups), dim3(256), 0, stream, q, L.t_sel, L.T_sel, L.T_pad, qhi,
                   eh);  // hi/lo
    if (e != cudaSuccess) return e;
    e = launch_pdl(prep_k_kernel, dim3(min(L.n_pad / 8, kPrepKCtas), kGroups), dim3(256), 0, stream, kq, ksc, L.n_max,
                   L.n_pad, kc, kmax);
    if (e != cudaSuccess) return e;
    if ((e = launch_score_gemm(L, pos0, qhi, kc, ksc, sc, p.sm_scale, status, stream)) != cudaSuccess) return e;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const dim3 grid(L.T_sel, kGroups);
  auto run = [&](auto kern) -> cudaError_t {
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkSmem);
    if (err != cudaSuccess) return err;
    const unsigned* h1 = L.T_sel <= kSmallRows ? hist1 : nullptr;
    return launch_pdl(kern, grid, dim3(kTkThreads), kTopkSmem, stream, sc, q, kq, ksc, eh, kmax, h1, ids, L.t_sel,
                      L.T_sel, L.n_pad, pos0, p.topk, p.sm_scale, status);
  };
  if (L.n_max <= 16 * kTkThreads) return run(topk_kernel<16>);
  if (L.n_max <= 32 * kTkThreads) return run(topk_kernel<32>);
  if (L.n_max <= 64 * kTkThreads) return run(topk_kernel<64>);
  return run(topk_kernel<128>);
}

}  // namespace qsa
