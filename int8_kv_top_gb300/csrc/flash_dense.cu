// qsa_flash_prefill, identity tokens (n_kv <= identity_max): dense causal attention of
// fp16 queries over the KV cache on the tcgen05 tensor cores.
//
// The pages' qsa_flash runs one threadgroup per (KV head, token) over 64-cell chunks:
// partial S for 12 heads, combine and scale by 1/16, max/exp per head, fp16 P, PV
// accumulate with per-head rescale ("opus_r9_qsa", what changed; "round 6 track b - qsa
// flash", delivered change: per-cell half4 K and V scales, identity ids while
// n_kv <= 2051).  That design serves a GPU without a matrix unit big enough for a 128-row
// tile.  Here the 12 heads of a group share their K/V rows, so a CTA owns a 128-row tile
// of (token, head) pairs of one group, 32 tokens x 4 heads, and every 64-cell chunk is a
// dense M=128 contraction over the call's fp16 mirror of the cache (mirror.cu: each cell
// dequantised once per call instead of once per tile that reads it):
//
//   warps 0, 2  TMA: fp16 K^ and V^ chunk tiles, four 128B-swizzled boxes of [64 cells][64
//               dims] each, which is exactly the UMMA operand layout; K^ in a 3-stage ring
//               released by QK(j), V^ in a 2-stage ring released by PV(j); warp 0 also loads
//               the Q tile, four boxes of [32 tokens][4 heads][64 dims]
//   warp 1      TMEM owner + QK issue:   S  = Q K^T  (A = Q K-major, B = K^ K-major)  M=128 N=64  K=256
//   warp 3      PV issue:                O += P V^   (A = P from TMEM, B = V^ MN-major) M=128 N=256 K=64
//   warps 4-11  two warpgroups, one (token, head) row per thread in each, half of the
//               columns each: online softmax on S in base-2 units (max exchanged through
//               shared memory, exp2, row sums), fp16 P -> TMEM over S, lazy O rescale (only
//               when the running max grows by more than 2^8), final 1/l and fp16 out.
// QK and PV are issued by two threads so that neither waits for the other's barrier round
// trips; four S/P buffers let QK run up to four chunks ahead of PV.
//
// TMEM columns: O [0,256)  S/P buffers [256 + 64 b, 320 + 64 b), b = 0..3.
// Every mbarrier wait is bounded; a timeout sets the status word and the CTA drains.
#include <cstring>

#include "common.cuh"

namespace qsa {
namespace {

constexpr int kTok = 32;               // tokens per row tile
constexpr int kHQ = 4;                 // heads per row tile
constexpr int kRows = kTok * kHQ;      // 128 = UMMA M
constexpr int kKV = 64;                // cells per chunk (UMMA N of QK^T)
constexpr int kThreads = 384;
constexpr int kKStages = 3, kVStages = 2;  // K^ freed by QK(j), V^ by PV(j): separate rings
constexpr int kNS = 4;                     // S/P buffers
constexpr int kHalfTile = kKV * kD * 2;    // one fp16 tile (K^ or V^), 32 KB
constexpr int kSmemV = kKStages * kHalfTile;                   // V ring after the K ring
constexpr int kSmemQ = (kKStages + kVStages) * kHalfTile;      // Q tile: 4 blocks of [128 rows][128 B]
constexpr int kQBytes = kRows * kD * 2;                        // 64 KB
constexpr int kSmemTotal = kSmemQ + kQBytes;                   // 224 KB
constexpr int kSmemAlloc = kSmemTotal + 1024;                  // + alignment slack
constexpr uint32_t kColO = 0, kColS = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct __align__(8) Bars {
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  // pv_done[i mod kNS]: PV(i) complete (frees S/P buffer i mod kNS, and O holds every PV <= i).
  // Waits are never two phases behind: QK(j) waits for PV(j - kNS), the softmax for PV(j - 1)
  // only after QK(j) (hence PV(j - kNS)) is done.
  uint64_t s_full[kNS], p_full[kNS], pv_done[kNS];
  uint64_t q_full, drain_qk, drain_pv;
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  uint32_t a[16], b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a[i] = r[i];
    b[i] = r[16 + i];
  }
  tmem_st16(taddr, a);
  tmem_st16(taddr + 16, b);
}

__global__ void __launch_bounds__(kThreads, 1)
    flash_dense_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_q, __half* __restrict__ out, int pos0, int t_begin,
                       int t_end, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_ttiles = (t_end - t_begin + kTok - 1) / kTok;
  const int item = blockIdx.x;
  const int ttile = n_ttiles - 1 - item / 6;  // heaviest (latest) token tiles first
  const int g = (item % 6) / 3, hq = item % 3;
  const int t0 = t_begin + ttile * kTok;
  const int t_last = min(t0 + kTok, t_end) - 1;
  const int n_kv_max = pos0 + t_last + 1;
  const int J = (n_kv_max + kKV - 1) / kKV;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 8);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.drain_qk, 1);
    mbar_init(&bars.drain_pv, 1);
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

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers (K^ + Q: warp 0, V^: warp 2)
    if (lane == 0) {
      const bool is_v = warp == 2;
      const CUtensorMap* map = is_v ? &map_v : &map_k;
      const int nst = is_v ? kVStages : kKStages;
      uint64_t* full = is_v ? bars.v_full : bars.k_full;
      uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
      uint8_t* ring = smem + (is_v ? kSmemV : 0);
      tma_prefetch_desc(map);
      if (!is_v) {  // Q tile: rows = 32 tokens x 4 heads (token-major), 64 dims per box
        tma_prefetch_desc(&map_q);
        mbar_arrive_expect_tx(&bars.q_full, kQBytes);
#pragma unroll
        for (int blk = 0; blk < kNB; ++blk)
          tma_load_3d(smem + kSmemQ + blk * (kRows * 128), &map_q, &bars.q_full, blk * 64, g * kHPG + hq * kHQ, t0);
      }
      int issued = 0;
      for (int j = 0; j < J; ++j) {
        const int s = j % nst;
        if (j >= nst && !mbar_wait(&empty[s], ((j / nst) & 1) ^ 1, status, &s_abort)) break;
        uint8_t* dst = ring + s * kHalfTile;
        mbar_arrive_expect_tx(&full[s], kHalfTile);
#pragma unroll
        for (int blk = 0; blk < kNB; ++blk) tma_load_3d(dst + blk * (kKV * 128), map, &full[s], blk * 64, g, j * kKV);
        issued = j + 1;
      }
      // drain: the loads of the last stages must have landed before the CTA exits
      for (int j = max(0, issued - nst); j < issued; ++j) mbar_wait(&full[j % nst], (j / nst) & 1, status);
      if (!is_v) mbar_wait(&bars.q_full, 0, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ QK issue
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_f16_f32(kRows, kKV, 0, 0);
      const uint32_t k0 = smem_u32(smem);
      const uint64_t qdesc = sdesc_sw128(smem_u32(smem + kSmemQ), 16, 1024);
      bool ok = mbar_wait(&bars.q_full, 0, status, &s_abort);
      for (int j = 0; ok && j < J; ++j) {
        const int b = j % kNS, s = j % kKStages;
        if (j >= kNS && !mbar_wait(&bars.pv_done[b], ((j / kNS) - 1) & 1, status, &s_abort)) break;  // P(j - 4) read
        if (!mbar_wait(&bars.k_full[s], (j / kKStages) & 1, status, &s_abort)) break;
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(k0 + s * kHalfTile, 16, 1024);
        const uint32_t scol = tmem + kColS + b * 64;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          umma_ss(scol, qdesc + (uint64_t)(((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                  kdesc + (uint64_t)(((kk >> 2) * (kKV * 128) + (kk & 3) * 32) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
        umma_commit(&bars.s_full[b]);
        umma_commit(&bars.k_empty[s]);
      }
      // drain: everything issued must complete before TMEM is released
      umma_commit(&bars.drain_qk);
      mbar_wait(&bars.drain_qk, 0, status);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------ PV issue
    if (lane == 0) {
      const uint32_t idesc_pv = idesc_f16_f32(kRows, kD, 0, 1);
      const uint32_t v0 = smem_u32(smem + kSmemV);
      for (int i = 0; i < J; ++i) {
        const int b = i % kNS, s = i % kVStages;
        if (!mbar_wait(&bars.p_full[b], (i / kNS) & 1, status, &s_abort)) break;
        if (!mbar_wait(&bars.v_full[s], (i / kVStages) & 1, status, &s_abort)) break;
        tc_fence_after();
        // descriptor built once; the start-address field (bytes >> 4, low bits) advances per K step
        const uint64_t vdesc = sdesc_sw128(v0 + s * kHalfTile, kKV * 128, 1024);
        const uint32_t pcol = tmem + kColS + b * 64;
#pragma unroll
        for (int kk = 0; kk < kKV / 16; ++kk)
          umma_ts(tmem + kColO, pcol + kk * 8, vdesc + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                  (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars.pv_done[b]);
        umma_commit(&bars.v_empty[s]);
      }
      umma_commit(&bars.drain_pv);
      mbar_wait(&bars.drain_pv, 0, status);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax rows
    // Two warpgroups share every row: warps 4-7 take S columns 0-31 of each chunk and O
    // dims 0-127, warps 8-11 columns 32-63 and dims 128-255; they exchange half-row maxima
    // and sums through shared memory.
    __shared__ float s_xm[2][kRows];  // half-row maxima, then half-row sums
    const int wg = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane == tile row
    const int tl = r >> 2, hl = r & 3;
    const int t = t0 + tl;
    const bool row_valid = t <= t_last;
    const int h = g * kHPG + hq * kHQ + hl;
    const int n_kv_row = row_valid ? pos0 + t + 1 : 0;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);

    float m_run = -INFINITY, l_run = 0.f;  // l_run: this half of the row
    bool ok = true;
    for (int j = 0; j < J; ++j) {
      const int b = j % kNS;
      const bool w_ok = mbar_wait_warp(&bars.s_full[b], (j / kNS) & 1, status, &s_abort);
      if (named_bar_any(1, 256, !w_ok || !ok)) { ok = false; break; }  // both warpgroups leave together
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(lane_base + kColS + b * 64 + wg * 32, sr);
      tmem_wait_ld();
      float s[32];
      float m_half = -INFINITY;
      const int lim = n_kv_row - j * kKV - wg * 32;  // cells i < lim are causal for this row
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = (i < lim) ? __uint_as_float(sr[i]) * scale_log2 : -INFINITY;
        m_half = fmaxf(m_half, s[i]);
      }
      s_xm[wg][r] = m_half;
      named_bar_any(1, 256, false);
      const float m_tile = fmaxf(m_half, s_xm[wg ^ 1][r]);
      const float m_new = fmaxf(m_run, m_tile);
      if (j == 0) {
        m_run = m_new;
      } else {
        const bool need = m_new > m_run + kRescaleThreshold;  // identical in both warpgroups
        if (__any_sync(0xffffffffu, need)) {
          // O must hold every PV issued so far before it is rescaled in place
          if (mbar_wait_warp(&bars.pv_done[(j - 1) % kNS], ((j - 1) / kNS) & 1, status, &s_abort)) {
            tc_fence_after();
            const float f = need ? fast_exp2(m_run - m_new) : 1.f;
#pragma unroll 1
            for (int c0 = wg * 128; c0 < wg * 128 + 128; c0 += 32) {
              uint32_t o[32];
              tmem_ld32(lane_base + kColO + c0, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
              tmem_st32(lane_base + kColO + c0, o);
            }
            tmem_wait_st();
            if (need) {
              l_run *= f;
              m_run = m_new;
            }
          } else {
            ok = false;  // reported at the next tile's collective barrier
          }
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pw[16];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = fast_exp2(s[2 * i] - m_use), p1 = fast_exp2(s[2 * i + 1] - m_use);
        lsum += p0 + p1;
        pw[i] = pack_half2(p0, p1);
      }
      l_run += lsum;
      tmem_st16(lane_base + kColS + b * 64 + wg * 16, pw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.p_full[b]);
    }
    if (!named_bar_any(1, 256, !ok)) {  // uniform: a failure in the last chunk is seen by all
      s_xm[wg][r] = l_run;
      named_bar_any(1, 256, false);
      const float l_tot = l_run + s_xm[wg ^ 1][r];
      const bool e_ok = mbar_wait_warp(&bars.pv_done[(J - 1) % kNS], ((J - 1) / kNS) & 1, status, &s_abort);
      if (e_ok) {
        tc_fence_after();
        const float inv_l = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
        __half* dst = out + ((size_t)(row_valid ? t : 0) * kHeads + h) * kD;
#pragma unroll 1
        for (int c0 = wg * 128; c0 < wg * 128 + 128; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + c0, o);
          tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_half2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// 3D map over a fp16 mirror [n][2][256]: box = 64 dims x 1 group x 64 cells, 128B swizzle.
bool make_mirror_map(CUtensorMap* map, const __half* base, int n) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kGroups, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * kGroups * 2};
  const cuuint32_t box[3] = {64u, 1u, (cuuint32_t)kKV};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D map over q [T][24][256]: box = 64 dims x 4 heads x 32 tokens, 128B swizzle; the box
// lands as the [128 rows][64 dims] block of a row tile (row = token * 4 + head).  Tokens past
// T read as zeros.
bool make_q_map(CUtensorMap* map, const __half* q, int T) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kHeads, (cuuint64_t)T};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * kHeads * 2};
  const cuuint32_t box[3] = {64u, (cuuint32_t)kHQ, (cuuint32_t)kTok};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_flash_dense(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                               cudaStream_t stream) {
  if (t_end <= t_begin) return cudaSuccess;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(flash_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  const int n = a.pos0 + a.T;  // cells in the mirror
  CUtensorMap mk, mv, mq;
  if (!make_mirror_map(&mk, khat, n) || !make_mirror_map(&mv, vhat, n) || !make_q_map(&mq, a.q, a.T))
    return cudaErrorInvalidValue;
  const int n_ttiles = (t_end - t_begin + kTok - 1) / kTok;
  const float scale_log2 = a.p.sm_scale * kLog2e;
  flash_dense_kernel<<<n_ttiles * 6, kThreads, kSmemAlloc, stream>>>(mk, mv, mq, a.out, a.pos0, t_begin, t_end,
                                                                    scale_log2, a.status);
  return cudaGetLastError();
}

}  // namespace qsa
