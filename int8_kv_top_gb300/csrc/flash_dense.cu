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
// dequantised once per call instead of once per tile that reads it).
//
// Two CTAs of a cluster form a pair over 64 consecutive tokens (rank 0 the first 32, rank 1
// the next 32; same group and head quad) and the cache is taken in 128-cell super-chunks, each
// ONE M=256 x N=128 contraction issued by rank 0 with .cta_group::2: each CTA holds its own 128
// Q rows, half of the K^ super-chunk (64 cells) and half of the V^ super-chunk (128 dims), and
// the hardware shares the B halves between the two SMs.  A chain of N=64 K16 steps runs at
// about 52 cycles each against 32 of arithmetic, N=128 at about 67 against 64, so the wide QK
// keeps the tensor pipe near its rate; per SM and 128 cells the shared-memory traffic is 96 KB
// of QK operands, 32 KB of PV operand and 64 KB of TMA writes.
//
//   warps 0, 2  TMA (both CTAs): this CTA's K^ half (four 128B-swizzled boxes of [64 cells]
//               [64 dims]) into a 3-stage ring and V^ half (two boxes of [128 cells][64 dims])
//               into a 2-stage ring, released by the pair MMA's multicast commit; warp 0 also
//               loads the Q tile, four boxes of [32 tokens][4 heads][64 dims]
//   warp 1      TMEM (pair allocation in both CTAs); rank 0: MMA issue, in the order
//               QK(0), QK(1), PV(0), QK(2), PV(1), ...
//                 S = Q K^T  (A = Q K-major, B = K^ K-major)  M=256 N=128 K=256
//                 O += P V^  (A = P from TMEM, B = V^ MN-major)  M=256 N=256 K=128
//               rank 1: forwards its Q and K^ arrivals to rank 0's barriers
//   warp 3      rank 1: forwards its V^ arrivals
//   warps 4-11  (both CTAs) two warpgroups, one (token, head) row per thread in each, half
//               of the columns each: online softmax on S in base-2 units (max exchanged
//               through shared memory, exp2, row sums), fp16 P -> TMEM over S, lazy O rescale
//               (only when the running max grows by more than 2^8), 1/l at the item's end;
//               P ready is signalled on rank 0's barrier.
//   warps 12-15 (both CTAs, plain launches) epilogue: O / l to fp16 and out, one row per thread,
//               while the softmax warpgroups and the tensor pipe start the next item; O is
//               released to the next item's first PV once it has been read from TMEM.  A gated
//               launch has no such warpgroup: the softmax warpgroups write O / l * sigmoid(gate)
//               out themselves, half the dims each, after the item's last PV.
// Two S/P buffers let QK(j + 1) run while super-chunk j is in the softmax.
//
// TMEM columns (each CTA): O [0,256)  S/P buffers [256 + 128 b, 384 + 128 b), b = 0, 1.
// Every mbarrier wait is bounded; a timeout sets the status word and both CTAs drain to the
// closing cluster barrier.
#include <algorithm>
#include <climits>
#include <cstring>

#include "common.cuh"

namespace qsa {
namespace {

constexpr int kTok = 32;               // tokens per CTA tile
constexpr int kHQ = 4;                 // heads per tile
constexpr int kRows = kTok * kHQ;      // 128 rows per CTA, 256 per pair (UMMA M)
constexpr int kKV = 128;               // cells per super-chunk (UMMA N of QK^T)
constexpr int kKStages = 3, kVStages = 2;  // K^ freed by QK(j), V^ by PV(j): separate rings
constexpr int kNS = 2;                     // S/P buffers
constexpr int kHalfK = (kKV / 2) * kD * 2;   // this CTA's K^ half: 64 cells x 256 dims fp16, 32 KB
constexpr int kHalfV = kKV * (kD / 2) * 2;   // this CTA's V^ half: 128 cells x 128 dims fp16, 32 KB
constexpr int kSmemV = kKStages * kHalfK;                 // V ring after the K ring
constexpr int kSmemQ = kSmemV + kVStages * kHalfV;        // Q tile: 4 blocks of [128 rows][128 B]
constexpr int kQBytes = kRows * kD * 2;                   // 64 KB
constexpr int kSmemTotal = kSmemQ + kQBytes;              // 224 KB
constexpr int kSmemAlloc = kSmemTotal + 1024;             // + alignment slack
constexpr uint32_t kColO = 0, kColS = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint16_t kBothCtas = 0x3;

// Same layout in both CTAs.  Rank 0's k_full / v_full / q_full complete on its own TMA bytes
// plus two arrivals (its producer's, and rank 1's forwarder once rank 1's half has landed);
// rank 1's complete on its own bytes and one arrival.  k_empty / v_empty / s_full / pv_done
// receive the pair MMA's multicast commits in both CTAs; p_full (rank 0) counts the 16
// softmax warps of the pair.
struct __align__(8) Bars {
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  // pv_done[i mod kNS]: PV(i) complete (frees S/P buffer i mod kNS, and O holds every PV <= i).
  // Waits are never two phases behind: QK(j) waits for PV(j - kNS), the softmax for PV(j - 1)
  // only after QK(j) (hence PV(j - kNS)) is done.
  uint64_t s_full[kNS], p_full[kNS], pv_done[kNS];
  uint64_t q_full, q_empty, o_free, drain;  // q_empty: last QK of an item done; o_free (rank 0): O read out
  // o_full: the item's last PV is complete (O final); l_full / l_empty: the per-row 1/l slot handed
  // from the softmax warpgroups to the epilogue warpgroup and back
  uint64_t o_full, l_full, l_empty;
};

// Items (pair of 32-token tiles, group, head quad), heaviest (latest tokens) first; a
// cluster takes every nC-th item in snake order so that the clusters' loads even out.  A
// batched call (many sequences) reads its pairs from a work list built on the device, already
// sorted heaviest first: {first token row, end of the sequence's identity rows, pos0 - first
// row of the sequence, first row of the sequence's mirror}.
struct Item {
  int g, hq, t0p, J;  // t0p: first token of the pair; J: super-chunks
  int t_end, p0, cbase;  // rows >= t_end are not this item's; n_kv(t) = p0 + t + 1; first mirror row
};
__device__ __forceinline__ Item item_at(int q, const int4* plan, int n_pairs, int t_begin, int t_end, int pos0) {
  Item it;
  it.g = (q % 6) / 3;
  it.hq = q % 3;
  if (plan != nullptr) {
    const int4 e = __ldg(&plan[1 + q / 6]);
    it.t0p = e.x;
    it.t_end = e.y;
    it.p0 = e.z;
    it.cbase = e.w;
  } else {
    it.t0p = t_begin + (n_pairs - 1 - q / 6) * 2 * kTok;
    it.t_end = t_end;
    it.p0 = pos0;
    it.cbase = 0;
  }
  const int t_last_pair = min(it.t0p + 2 * kTok, it.t_end) - 1;
  it.J = (it.p0 + t_last_pair + 1 + kKV - 1) / kKV;
  return it;
}
__device__ __forceinline__ int item_of(int c, int nC, int n, int n_items) {
  const int q = n * nC + ((n & 1) ? nC - 1 - c : c);
  return q < n_items ? q : -1;
}

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

// One (token, head) row per thread: O columns [c_begin, c_end) of the thread's TMEM lane, times
// 1/l (and the gate's sigmoid), rounded to fp16 once and stored.  The 4 lanes of a group hold the
// 4 heads of one token, whose output rows are adjacent.  Per 64 dims each lane packs its row into
// 4 blocks of 16 dims (32 B); a two-step butterfly gives lane g block g of all 4 rows, and each
// 32-byte store of a warp then writes 8 whole 128-byte row segments instead of 32 scattered
// pieces.  `loaded()` runs once the last piece is in registers: O may be overwritten after it.
template <typename F>
__device__ __forceinline__ void store_o_rows(uint32_t lane_base, int c_begin, int c_end, float inv_l, __half* gdst,
                                             const __half* grow, bool tok_valid, int lane, F&& loaded) {
  const int g0 = lane & 1, g1 = (lane >> 1) & 1;
#pragma unroll 1
  for (int c0 = c_begin; c0 < c_end; c0 += 64) {
    uint32_t oa[32], ob[32];
    tmem_ld32(lane_base + kColO + c0, oa);
    tmem_ld32(lane_base + kColO + c0 + 32, ob);
    tmem_wait_ld();
    if (c0 + 64 == c_end) loaded();
    uint32_t B[32];  // block b (dims c0 + 16 b ..) = words 8 b .. 8 b + 7
    if (grow) {  // output gate: o / l * sigmoid(gate), rounded to fp16 once
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t* src = hh ? ob : oa;
        uint4 gw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) gw[u] = __ldg(reinterpret_cast<const uint4*>(grow + c0 + 32 * hh) + u);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = i % 4 == 0 ? gw[i / 4].x : i % 4 == 1 ? gw[i / 4].y : i % 4 == 2 ? gw[i / 4].z : gw[i / 4].w;
          const float2 gv = __half22float2(*reinterpret_cast<const __half2*>(&w));
          B[16 * hh + i] = pack_half2(__uint_as_float(src[2 * i]) * inv_l * gate_sigmoid(gv.x),
                                      __uint_as_float(src[2 * i + 1]) * inv_l * gate_sigmoid(gv.y));
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        B[i] = pack_half2(__uint_as_float(oa[2 * i]) * inv_l, __uint_as_float(oa[2 * i + 1]) * inv_l);
        B[16 + i] = pack_half2(__uint_as_float(ob[2 * i]) * inv_l, __uint_as_float(ob[2 * i + 1]) * inv_l);
      }
    }
#pragma unroll
    for (int b1 = 0; b1 < 2; ++b1)  // blocks (b1, 1 - g0) to and from lane ^ 1
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t x0 = B[(2 * b1) * 8 + i], x1 = B[(2 * b1 + 1) * 8 + i];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, g0 ? x0 : x1, 1);
        B[(2 * b1) * 8 + i] = g0 ? got : x0;
        B[(2 * b1 + 1) * 8 + i] = g0 ? x1 : got;
      }
#pragma unroll
    for (int e0 = 0; e0 < 2; ++e0)  // blocks (1 - g1, e0) to and from lane ^ 2
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t x0 = B[e0 * 8 + i], x1 = B[(2 + e0) * 8 + i];
        const uint32_t got = __shfl_xor_sync(0xffffffffu, g1 ? x0 : x1, 2);
        B[e0 * 8 + i] = g1 ? got : x0;
        B[(2 + e0) * 8 + i] = g1 ? x1 : got;
      }
    if (tok_valid) {  // block e = dims c0 + 16 gq .. of head e's row
#pragma unroll
      for (int e = 0; e < 4; ++e)
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(gdst + e * kD + c0),
                     "r"(B[8 * e]), "r"(B[8 * e + 1]), "r"(B[8 * e + 2]), "r"(B[8 * e + 3]), "r"(B[8 * e + 4]),
                     "r"(B[8 * e + 5]), "r"(B[8 * e + 6]), "r"(B[8 * e + 7])
                     : "memory");
    }
  }
}

// kEpiWG: a fourth warpgroup writes O out while the softmax warpgroups and the tensor pipe go on
// with the next item (512 threads).  Without it (384 threads) the softmax warpgroups write O
// themselves, half the dims each: the gated launch, whose sigmoid work would otherwise compete
// with the next item's softmax for issue slots while O is still held in TMEM.
template <bool kEpiWG>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kEpiWG ? 512 : 384, 1)
    flash_dense_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_q, const __half* __restrict__ gate,
                       __half* __restrict__ out, const int4* __restrict__ plan, int pos0, int t_begin, int t_end,
                       float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ float s_invl[kRows];  // 1/l per row of the item being written out
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int n_ttiles = (t_end - t_begin + kTok - 1) / kTok;
  const int n_pairs = (n_ttiles + 1) / 2;
  const int c = blockIdx.x >> 1, nC = gridDim.x >> 1;

  if (tid == 0) {
    s_abort = 0;
    const uint32_t n_in = rank == 0 ? 2u : 1u;  // arrivals that complete a full barrier
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], n_in);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], n_in);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 16);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.q_full, n_in);
    mbar_init(&bars.q_empty, 1);
    mbar_init(&bars.o_free, kEpiWG ? 8 : 16);  // the warps that read O out, in both CTAs
    mbar_init(&bars.o_full, 1);
    mbar_init(&bars.l_full, 4);  // the first softmax warpgroup's 4 warps
    mbar_init(&bars.l_empty, 4); // the epilogue's 4 warps
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive or commit
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_begin();
  const int n_items = (plan != nullptr ? __ldg(&plan[0].x) : n_pairs) * 6;  // a work list comes from the previous launch

  // Global super-chunk index gj (over this cluster's items) drives every ring's stage and phase.
  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------ TMA producers (K^ + Q: warp 0, V^: warp 2)
    if (lane == 0) {
      const bool is_v = warp == 2;
      const CUtensorMap* map = is_v ? &map_v : &map_k;
      const int nst = is_v ? kVStages : kKStages;
      const uint32_t bytes = is_v ? kHalfV : kHalfK;
      uint64_t* full = is_v ? bars.v_full : bars.k_full;
      uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
      uint8_t* ring = smem + (is_v ? kSmemV : 0);
      tma_prefetch_desc(map);
      if (!is_v) tma_prefetch_desc(&map_q);
      int gj = 0, n = 0;
      bool ok = true;
      for (; ok; ++n) {
        const int q = item_of(c, nC, n, n_items);
        if (q < 0) break;
        const Item it = item_at(q, plan, n_pairs, t_begin, t_end, pos0);
        if (!is_v) {  // Q tile (rows = 32 tokens x 4 heads, token-major), once the last QK of the previous item is done
          if (n > 0 && !mbar_wait(&bars.q_empty, (n - 1) & 1, status, &s_abort)) break;
          mbar_arrive_expect_tx(&bars.q_full, kQBytes);
#pragma unroll
          for (int blk = 0; blk < kNB; ++blk)
            tma_load_3d(smem + kSmemQ + blk * (kRows * 128), &map_q, &bars.q_full, blk * 64, it.g * kHPG + it.hq * kHQ,
                        it.t0p + (int)rank * kTok);
        }
        for (int j = 0; j < it.J; ++j, ++gj) {
          const int s = gj % nst;
          if (gj >= nst && !mbar_wait(&empty[s], ((gj / nst) & 1) ^ 1, status, &s_abort)) {
            ok = false;
            break;
          }
          uint8_t* dst = ring + s * bytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          if (is_v) {  // dims 128 rank .. 128 rank + 127 of the super-chunk's cells
#pragma unroll
            for (int blk = 0; blk < 2; ++blk)
              tma_load_3d(dst + blk * (kKV * 128), map, &full[s], (int)rank * 128 + blk * 64, it.g,
                          it.cbase + j * kKV);
          } else {     // cells 128 j + 64 rank .. + 63, all dims
#pragma unroll
            for (int blk = 0; blk < kNB; ++blk)
              tma_load_3d(dst + blk * ((kKV / 2) * 128), map, &full[s], blk * 64, it.g,
                          it.cbase + j * kKV + (int)rank * (kKV / 2));
          }
        }
      }
      // drain: this CTA's last loads must have landed before it exits
      for (int k = max(0, gj - nst); k < gj; ++k) mbar_wait(&full[k % nst], (k / nst) & 1, status);
      if (!is_v && n > 0) mbar_wait(&bars.q_full, (n - 1) & 1, status);
    }
  } else if (warp == 1 && rank == 1) {
    // ------------------------------------------------------------ rank 1: forward Q and K^ arrivals
    if (lane == 0) {
      const uint32_t q_rem = mapa_shared(smem_u32(&bars.q_full), 0);
      const uint32_t k_rem = mapa_shared(smem_u32(&bars.k_full[0]), 0);
      int gj = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int q = item_of(c, nC, n, n_items);
        if (q < 0) break;
        const Item it = item_at(q, plan, n_pairs, t_begin, t_end, pos0);
        if (!mbar_wait(&bars.q_full, n & 1, status, &s_abort)) break;
        mbar_arrive_cluster(q_rem);
        for (int j = 0; j < it.J; ++j, ++gj) {
          const int s = gj % kKStages;
          if (!mbar_wait(&bars.k_full[s], (gj / kKStages) & 1, status, &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(k_rem + 8u * (uint32_t)s);
        }
      }
    }
    __syncwarp();
  } else if (warp == 3 && rank == 1) {
    // ------------------------------------------------------------ rank 1: forward V^ arrivals
    if (lane == 0) {
      const uint32_t v_rem = mapa_shared(smem_u32(&bars.v_full[0]), 0);
      int gj = 0;
      bool ok = true;
      for (int n = 0; ok; ++n) {
        const int q = item_of(c, nC, n, n_items);
        if (q < 0) break;
        const Item it = item_at(q, plan, n_pairs, t_begin, t_end, pos0);
        for (int j = 0; j < it.J; ++j, ++gj) {
          const int s = gj % kVStages;
          if (!mbar_wait(&bars.v_full[s], (gj / kVStages) & 1, status, &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(v_rem + 8u * (uint32_t)s);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ rank 0: MMA issue
    // One thread issues QK(j + 1) before PV(j), so the in-order tensor pipe never holds the
    // S of the next super-chunk behind a PV: QK(j + 1) needs its buffer back from PV(j - 1)
    // (the two share no accumulator, so that completion is awaited), PV(j) needs P(j).  The
    // thread polls (no suspend, no sleep): the tensor pipe's instruction queue is short, and a
    // late wake-up after a completion leaves it idle.
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_f16_f32(2 * kRows, kKV, 0, 0);
      const uint32_t idesc_pv = idesc_f16_f32(2 * kRows, kD, 0, 1);
      const uint32_t k0 = smem_u32(smem), v0 = smem_u32(smem + kSmemV);
      const uint64_t qdesc = sdesc_sw128(smem_u32(smem + kSmemQ), 16, 1024);
      // gj: global super-chunk index (rings, buffers and phases); a PV with restart = true
      // overwrites O, so the previous item's O must have been read out (o_free)
      auto issue_qk = [&](int gj) -> bool {
        const int b = gj % kNS, s = gj % kKStages;
        if (gj >= kNS && !mbar_wait_poll(&bars.pv_done[b], ((gj / kNS) - 1) & 1, status, &s_abort)) return false;
        if (!mbar_wait_poll(&bars.k_full[s], (gj / kKStages) & 1, status, &s_abort)) return false;
        tc_fence_after();
        const uint64_t kdesc = sdesc_sw128(k0 + s * kHalfK, 16, 1024);
        const uint32_t scol = tmem + kColS + b * kKV;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          umma2_ss(scol, qdesc + (uint64_t)(((kk >> 2) * (kRows * 128) + (kk & 3) * 32) >> 4),
                   kdesc + (uint64_t)(((kk >> 2) * ((kKV / 2) * 128) + (kk & 3) * 32) >> 4), idesc_qk,
                   kk > 0 ? 1u : 0u);
        umma2_commit(&bars.s_full[b], kBothCtas);
        umma2_commit(&bars.k_empty[s], kBothCtas);
        return true;
      };
      auto issue_pv = [&](int gj, bool restart) -> bool {
        const int b = gj % kNS, s = gj % kVStages;
        if (!mbar_wait_poll(&bars.p_full[b], (gj / kNS) & 1, status, &s_abort)) return false;
        if (!mbar_wait_poll(&bars.v_full[s], (gj / kVStages) & 1, status, &s_abort)) return false;
        tc_fence_after();
        // descriptor built once; the start-address field (bytes >> 4, low bits) advances per K step
        const uint64_t vdesc = sdesc_sw128(v0 + s * kHalfV, kKV * 128, 1024);
        const uint32_t pcol = tmem + kColS + b * kKV;
#pragma unroll
        for (int kk = 0; kk < kKV / 16; ++kk)
          umma2_ts(tmem + kColO, pcol + kk * 8, vdesc + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                   (!restart || kk > 0) ? 1u : 0u);
        umma2_commit(&bars.pv_done[b], kBothCtas);
        umma2_commit(&bars.v_empty[s], kBothCtas);
        return true;
      };
      bool ok = true;
      int base = 0;
      for (int n = 0; ok; ++n) {
        const int q = item_of(c, nC, n, n_items);
        if (q < 0) break;
        const int J = item_at(q, plan, n_pairs, t_begin, t_end, pos0).J;
        ok = mbar_wait_poll(&bars.q_full, n & 1, status, &s_abort) && issue_qk(base);
        if (ok && J == 1) umma2_commit(&bars.q_empty, kBothCtas);  // Q no longer read
        for (int j = 0; ok && j < J; ++j) {
          if (j + 1 < J) {
            ok = issue_qk(base + j + 1);
            if (ok && j + 2 == J) umma2_commit(&bars.q_empty, kBothCtas);
          }
          if (ok && j == 0 && n > 0) ok = mbar_wait_poll(&bars.o_free, (n - 1) & 1, status, &s_abort);
          ok = ok && issue_pv(base + j, j == 0);
          if (kEpiWG && ok && j + 1 == J) umma2_commit(&bars.o_full, kBothCtas);  // O final: the epilogue may read it
        }
        base += J;
      }
      // drain: everything issued must complete before TMEM is released
      umma2_commit(&bars.drain, 0x1);
      mbar_wait(&bars.drain, 0, status);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax rows
    // Two warpgroups share every row: warps 4-7 take S columns 0-63 of each super-chunk and O
    // dims 0-127 (for the lazy rescale), warps 8-11 columns 64-127 and dims 128-255; they exchange
    // half-row maxima (when needed) and sums through shared memory.  At the end of an item they
    // hand 1/l to the epilogue warpgroup and go straight on to the next item's first super-chunk.
    __shared__ float s_xm[2][kRows];  // half-row maxima, then half-row sums
    const int wg = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane == tile row
    const int tl = r >> 2;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t p_full0 = mapa_shared(smem_u32(&bars.p_full[0]), 0);  // rank 0's p_full[0]
    bool ok = true;
    int base = 0;  // global index of the item's first super-chunk
    for (int n = 0; ok; ++n) {
    const int q = item_of(c, nC, n, n_items);
    if (q < 0) break;
    const Item it = item_at(q, plan, n_pairs, t_begin, t_end, pos0);
    const int J = it.J;
    const int t0 = it.t0p + (int)rank * kTok;         // this CTA's first token
    const int t_last = min(t0 + kTok, it.t_end) - 1;   // < t0 for an empty tile
    const int t = t0 + tl;
    const bool row_valid = t <= t_last;
    const int n_kv_row = row_valid ? it.p0 + t + 1 : 0;
    if (!kEpiWG && gate != nullptr && row_valid) {
      // the row's gate values (this warpgroup's 128 dims) go to L2 now; the write-out reads them
      const char* grow = reinterpret_cast<const char*>(
          gate + ((size_t)t * kHeads + it.g * kHPG + it.hq * kHQ + (lane & 3)) * kD + wg * 128);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(grow));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(grow + 128));
    }
    float m_run = -INFINITY, l_run = 0.f;  // m_run in log2 units; l_run: this half of the row
    for (int j = 0; j < J; ++j) {
      const int gj = base + j, b = gj % kNS;
      const bool w_ok = mbar_wait_warp(&bars.s_full[b], (gj / kNS) & 1, status, &s_abort);
      tc_fence_after();
      uint32_t sa[32], sb[32];
      tmem_ld32(lane_base + kColS + b * kKV + wg * 64, sa);
      tmem_ld32(lane_base + kColS + b * kKV + wg * 64 + 32, sb);
      tmem_wait_ld();
      // raw scores; non-causal cells (only near the diagonal) become -inf
      float s[64];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        s[i] = __uint_as_float(sa[i]);
        s[32 + i] = __uint_as_float(sb[i]);
      }
      const int lim = n_kv_row - j * kKV - wg * 64;  // cells i < lim are causal for this row
      if (lim < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = (i < lim) ? s[i] : -INFINITY;
      }
      float mx[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) mx[i] = fmaxf(s[i], s[i + 32]);
#pragma unroll
      for (int w = 16; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) mx[i] = fmaxf(mx[i], mx[i + w]);
      const float m_half = mx[0] * scale_log2;  // scale > 0 keeps the order
      const bool fail = !w_ok || !ok;
      // One barrier reduction per super-chunk (it also orders every S read of the tile before
      // the P stores, which overwrite the first half of the buffer): the half-row maxima are
      // exchanged only when some row crosses its running maximum by the threshold, and at j = 0.
      if (named_bar_any(1, 256, fail || j == 0 || m_half > m_run + kRescaleThreshold)) {
        s_xm[wg][r] = m_half;
        if (named_bar_any(1, 256, fail)) { ok = false; break; }  // both warpgroups leave together
        const float m_new = fmaxf(m_run, fmaxf(m_half, s_xm[wg ^ 1][r]));
        if (j == 0) {
          m_run = m_new;
        } else {
          const bool need = m_new > m_run + kRescaleThreshold;  // identical in both warpgroups
          if (__any_sync(0xffffffffu, need)) {
            // O must hold every PV issued so far before it is rescaled in place
            if (mbar_wait_warp(&bars.pv_done[(gj - 1) % kNS], ((gj - 1) / kNS) & 1, status, &s_abort)) {
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
              ok = false;  // reported at the next super-chunk's barrier reduction
            }
          }
        }
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      uint32_t pa[16], pb[16];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = fast_exp2(fmaf(s[2 * i], scale_log2, -m_use));
        const float p1 = fast_exp2(fmaf(s[2 * i + 1], scale_log2, -m_use));
        const float p2 = fast_exp2(fmaf(s[32 + 2 * i], scale_log2, -m_use));
        const float p3 = fast_exp2(fmaf(s[33 + 2 * i], scale_log2, -m_use));
        lsum += (p0 + p1) + (p2 + p3);
        pa[i] = pack_half2(p0, p1);
        pb[i] = pack_half2(p2, p3);
      }
      l_run += lsum;
      tmem_st16(lane_base + kColS + b * kKV + wg * 32, pa);
      tmem_st16(lane_base + kColS + b * kKV + wg * 32 + 16, pb);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&bars.p_full[b]);
        else mbar_arrive_cluster(p_full0 + 8u * (uint32_t)b);
      }
    }
    if (named_bar_any(1, 256, !ok)) {  // uniform: a failure in the last chunk is seen by all
      ok = false;
    } else {
      s_xm[wg][r] = l_run;
      named_bar_any(1, 256, false);
      if constexpr (kEpiWG) {
        if (wg == 0) {  // 1/l of the row to the epilogue warpgroup, once it has taken the previous item's
          const float l_tot = l_run + s_xm[1][r];
          if (n == 0 || mbar_wait_warp(&bars.l_empty, (n - 1) & 1, status, &s_abort)) {
            s_invl[r] = (l_tot > 0.f) ? 1.f / l_tot : 0.f;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.l_full);
          } else {
            ok = false;
          }
        }
      } else {  // this warpgroup's half of the dims, once the item's last PV is complete
        const float l_tot = l_run + s_xm[wg ^ 1][r];
        const int gl = base + J - 1;
        if (mbar_wait_warp(&bars.pv_done[gl % kNS], (gl / kNS) & 1, status, &s_abort)) {
          tc_fence_after();
          const int gq = lane & 3;
          const int tok = t0 + quarter * 8 + (lane >> 2);
          const bool tok_valid = tok <= t_last;
          const size_t orow = (size_t)(tok_valid ? tok : 0) * kHeads + it.g * kHPG + it.hq * kHQ;
          store_o_rows(lane_base, wg * 128, wg * 128 + 128, (l_tot > 0.f) ? 1.f / l_tot : 0.f,
                       out + orow * kD + 16 * gq, gate ? gate + (orow + gq) * kD : nullptr, tok_valid, lane, [&] {
                         tc_fence_before();  // O is in registers: the next item's first PV may overwrite it
                         __syncwarp();
                         if (lane == 0) {
                           if (rank == 0) mbar_arrive(&bars.o_free);
                           else mbar_arrive_cluster(mapa_shared(smem_u32(&bars.o_free), 0));
                         }
                       });
        } else {
          ok = false;
        }
      }
    }
    // all 256 threads agree before the next item's barriers
    if (named_bar_any(1, 256, !ok)) ok = false;
    base += J;
    }
  } else if (kEpiWG && warp >= 12) {
    // ------------------------------------------------------------ epilogue rows
    // One row per thread, all 256 dims: once the item's last PV is complete, O is read from TMEM
    // in 64-dim pieces, scaled by 1/l (and the gate), rounded to fp16 and stored; O is released
    // to the next item's first PV as soon as its last piece is in registers.  Meanwhile the
    // softmax warpgroups already work on the next item, so the read-out is off the tensor pipe's
    // critical path.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane == tile row
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t o_free0 = mapa_shared(smem_u32(&bars.o_free), 0);  // rank 0's o_free
    const int gq = lane & 3;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int q = item_of(c, nC, n, n_items);
      if (q < 0) break;
      const Item it = item_at(q, plan, n_pairs, t_begin, t_end, pos0);
      const int t0 = it.t0p + (int)rank * kTok;        // this CTA's first token
      const int t_last = min(t0 + kTok, it.t_end) - 1;  // < t0 for an empty tile
      const int tok = t0 + quarter * 8 + (lane >> 2);
      const bool tok_valid = tok <= t_last;
      const size_t orow = (size_t)(tok_valid ? tok : 0) * kHeads + it.g * kHPG + it.hq * kHQ;
      __half* gdst = out + orow * kD + 16 * gq;
      // this lane's own row (head it.hq * kHQ + gq of token tok) in the gate input, sent to L2 now
      const __half* grow = gate ? gate + (orow + gq) * kD : nullptr;
      if (grow && tok_valid) {
#pragma unroll
        for (int u = 0; u < 4; ++u) asm volatile("prefetch.global.L2 [%0];" ::"l"(grow + 64 * u));
      }
      if (!mbar_wait_warp(&bars.l_full, n & 1, status, &s_abort)) {
        ok = false;
        break;
      }
      const float inv_l = s_invl[r];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.l_empty);
      if (!mbar_wait_warp(&bars.o_full, n & 1, status, &s_abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      store_o_rows(lane_base, 0, kD, inv_l, gdst, grow, tok_valid, lane, [&] {
        tc_fence_before();  // O is in registers: the next item's first PV may overwrite it
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(&bars.o_free);
          else mbar_arrive_cluster(o_free0);
        }
      });
    }
  }

  tc_fence_before();
  cluster_sync_all();  // rank 0's MMAs have drained; neither CTA leaves while the other may read its memory
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, 512);
}

// 3D map over a fp16 mirror [n][2][256]: box = 64 dims x 1 group x `box_cells` cells, 128B swizzle.
bool make_mirror_map(CUtensorMap* map, const __half* base, int n, int box_cells) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kGroups, (cuuint64_t)n};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * kGroups * 2};
  const cuuint32_t box[3] = {64u, 1u, (cuuint32_t)box_cells};
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

namespace {

// Per device, set once (0 = not yet): the shared-memory attribute and how many CTA pairs fit on the
// GPU at once; threads that race here both set the same attribute and store the same count.
template <bool kEpiWG>
cudaError_t dense_clusters(int* n_clusters_max) {
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  int nc = max_clusters[dev].load(std::memory_order_acquire);
  if (nc == 0) {
    cudaError_t e =
        cudaFuncSetAttribute(flash_dense_kernel<kEpiWG>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kEpiWG ? 512 : 384, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    e = cudaOccupancyMaxActiveClusters(&nc, flash_dense_kernel<kEpiWG>, &cfg);
    if (e != cudaSuccess) return e;
    if (nc < 1) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(nc, std::memory_order_release);
  }
  *n_clusters_max = nc;
  return cudaSuccess;
}

// The plain launch takes the epilogue warpgroup; the gated one does not (see flash_dense_kernel).
template <typename... Args>
cudaError_t launch_dense(const __half* gate, int n_items, cudaStream_t stream, Args&&... args) {
  int n_clusters_max = 0;
  const bool epi = gate == nullptr;
  cudaError_t e = epi ? dense_clusters<true>(&n_clusters_max) : dense_clusters<false>(&n_clusters_max);
  if (e != cudaSuccess) return e;
  const int n_clusters = std::min(n_clusters_max, n_items);  // persistent: each takes items in snake order
  if (epi)
    return launch_pdl(flash_dense_kernel<true>, dim3(n_clusters * 2), dim3(512), kSmemAlloc, stream, args...);
  return launch_pdl(flash_dense_kernel<false>, dim3(n_clusters * 2), dim3(384), kSmemAlloc, stream, args...);
}

}  // namespace

cudaError_t launch_flash_dense(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                               cudaStream_t stream) {
  if (t_end <= t_begin) return cudaSuccess;
  const int n = a.pos0 + a.T;  // cells in the mirror
  CUtensorMap mk, mv, mq;
  if (!make_mirror_map(&mk, khat, n, kKV / 2) || !make_mirror_map(&mv, vhat, n, kKV) || !make_q_map(&mq, a.q, a.T))
    return cudaErrorInvalidValue;
  const int n_ttiles = (t_end - t_begin + kTok - 1) / kTok;
  const int n_items = (n_ttiles + 1) / 2 * 6;  // (pair of tiles, group, head quad)
  return launch_dense(a.gate, n_items, stream, mk, mv, mq, a.gate, a.out, static_cast<const int4*>(nullptr), a.pos0,
                      t_begin, t_end, a.p.sm_scale * kLog2e, a.status);
}

cudaError_t launch_flash_dense_batched(const __half* q, int n_tok, const __half* gate, __half* out, const int4* plan,
                                       int max_pairs, const __half* khat, const __half* vhat, int mirror_rows,
                                       float sm_scale, int* status, cudaStream_t stream) {
  if (max_pairs <= 0) return cudaSuccess;
  CUtensorMap mk, mv, mq;
  if (!make_mirror_map(&mk, khat, mirror_rows, kKV / 2) || !make_mirror_map(&mv, vhat, mirror_rows, kKV) ||
      !make_q_map(&mq, q, n_tok))
    return cudaErrorInvalidValue;
  const int n_items = (int)std::min<long long>(6LL * max_pairs, INT_MAX);
  return launch_dense(gate, n_items, stream, mk, mv, mq, gate, out, plan, 0, 0, 0, sm_scale * kLog2e, status);
}

}  // namespace qsa
