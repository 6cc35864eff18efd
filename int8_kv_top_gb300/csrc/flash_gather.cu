// qsa_flash_prefill, selected tokens (n_kv > identity_max): attention of one token's 12
// group heads over its own top-k cell set, on the tcgen05 tensor cores.
//
// In the pages, qsa_flash reads explicit selected ids above the budget (per token, grid
// (2, T); "round 6 track b - qsa flash", delivered change) and hoists per-cell byte offsets
// and zero scales for invalid cells ("round 14 track b: qsa metadata hoist", decision and
// correctness).  Here each (token, group) has its own 2048 cells, so no K/V tile is shared
// across tokens, while every cell of the cache is selected by many tokens (about 6% of
// 1984 tokens per layer on random data).  Two launches therefore:
//
//  1. the fp16 mirror (mirror.cu): K^ = fp16(kq * ksc) and V^ = fp16(vq * vsc) once per
//     call for the cells the call's tokens can see, in the cache's [cell][group][256] layout.
//  2. flash_gather: per (token, group), the selected fp16 rows are gathered with 16-byte
//     cp.async copies straight into 128B-swizzled UMMA operand tiles, and the MMA is swapped
//     so the gathered cells form the 128-wide M side:
//        S^T[c][h]  = K^[c] . q[h]      A = K^ (128 cells, K-major)  B = Q^T (16 rows, 12 used)
//        O^T[d][h] += V^[c][d] P[h][c]  A = V^ as MN-major (dims x cells)  B = P^T (K-major)
//
// K and V have rings of their own (three 32 KB slots each: half a tile, 128 cells x 128
// dims), each fed by a pool of three producer warp pairs that take turns, one pair per fill,
// so fills complete independently and several are in flight.  QK and PV are issued by two
// threads, each waiting only for what its own MMAs read, so neither pays for the other's
// barrier round trips; kNS S^T / P^T buffers decouple them.  Ids are ascending, so tile j of
// every item covers about the same cell range; each item starts its walk at tile (item mod
// tiles), which spreads the SMs' concurrent reads over the whole mirror (the online softmax
// does not depend on the order of the tiles).
//     warp 0        TMEM owner, QK issue (S^T = K^ . Q^T)
//     warp 1        PV issue (O^T += V^^T . P^T)
//     warps 2-3, 12-15  K producers (warp 2 also starts each item's Q^T tile by TMA)
//     warps 16-21   V producers
//     warps 4-7     softmax for heads 0-5, warps 8-11 for heads 6-11: one gathered cell per
//                   thread (TMEM lane), column-wise online softmax over the 128 cells
//                   (shuffle + shared-memory max per head, base-2 exponent), fp16 P^T into
//                   shared memory, lazy O^T rescale, epilogue (thread = dim)
// The CTA is persistent over (token, group) work items.  TMEM: S^T buffers [0, 64), O^T
// double buffer (two 16-column halves for dims 0-127 / 128-255) [64, 128).
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kCells = 128;                // gathered cells per tile (UMMA M)
constexpr int kNQ = 16;                    // UMMA N: 12 heads + 4 zero rows
constexpr int kThreads = 704;
constexpr int kPoolPairs = 3;              // warp pairs per producer pool (K: 2-3, 12-15; V: 16-21)
constexpr int kBlkBytes = kCells * 128;    // 16 KB: one 64-dim block of a tile
constexpr int kSlotBytes = 2 * kBlkBytes;  // 32 KB: one 128-dim half of a K or V tile
constexpr int kRing = 3;                   // slots per ring
constexpr int kNS = 4;                     // S^T and P^T buffers
constexpr int kQBytes = kNQ * kD * 2;      // 8 KB
constexpr int kPBytes = kNQ * kCells * 2;  // 4 KB
constexpr int kOffK = 0, kOffV = kRing * kSlotBytes, kOffQ = 2 * kRing * kSlotBytes;
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kSmemTotal = kOffP + kNS * kPBytes;
constexpr int kSmemAlloc = kSmemTotal + 1024;
constexpr uint32_t kColS = 0, kColO = kNS * 16;
constexpr int kHPW = 6;  // heads per softmax warpgroup
constexpr float kRescaleThreshold = 8.0f;
constexpr int kNoSlot = -2147483647 - 1;  // marks tile slots past the end of an id row
// A ring's empty barriers are keyed by the consumed fill mod 2 * kRing: a warp pair refilling
// the slot of fill f saw, at its previous fill (kPoolPairs earlier), fill f - kPoolPairs - kRing
// consumed, which covers the previous phase of the barrier it waits on.
static_assert(kPoolPairs <= 2 * kRing, "empty-barrier keying must cover the producer round-robin");

struct Ring {
  uint64_t full[kRing], empty[2 * kRing];
};

struct __align__(8) GBars {
  Ring k, v;
  uint64_t q_full[2], q_empty[2];
  // p_free[u mod kNS] completes when PV(u) (and every PV before it) is done: it frees P^T(u)
  // and tells the softmax O^T is up to date.  Every wait on it is at most one phase behind:
  // the softmax waits for PV(u - kNS) at tile u, and for PV(u - 1) only later.
  uint64_t s_full[kNS], s_free[kNS], p_full[kNS], p_free[kNS];
  uint64_t o_free[2];
  uint64_t drain_qk, drain_pv;
};

// 16-byte copy that writes zeros (and reads nothing) when `valid` is false.
__device__ __forceinline__ void cp_async16_sh(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(valid ? 16 : 0)
               : "memory");
}

// Position in this CTA's walk over (item, tile): k-th own item, tile jl of it, and the item's
// rotation (item mod tiles), advanced by compare-and-wrap instead of integer divisions.
struct TileIter {
  int k, jl, rot;
  __device__ __forceinline__ void advance(int n_tiles, int rot_step) {
    if (++jl == n_tiles) {
      jl = 0;
      ++k;
      rot += rot_step;
      if (rot >= n_tiles) rot -= n_tiles;
    }
  }
  __device__ __forceinline__ int tile(int n_tiles) const {  // the tile taken at step jl (rotated order)
    const int p = jl + rot;
    return p >= n_tiles ? p - n_tiles : p;
  }
};

__device__ __forceinline__ int pick4(const int (&v)[4], int x) {  // select chain: no local memory
  return x == 0 ? v[0] : x == 1 ? v[1] : x == 2 ? v[2] : v[3];
}

// This warpgroup's six head columns (wg 0: 0-5, wg 1: 6-11) of a 16-column TMEM group.
__device__ __forceinline__ void ld6(uint32_t taddr, int wg, uint32_t (&r)[kHPW]) {
  if (wg == 0) {
    tmem_ld4(taddr, r);
    tmem_ld2(taddr + 4, r + 4);
  } else {
    tmem_ld2(taddr + 6, r);
    tmem_ld4(taddr + 8, r + 2);
  }
}
__device__ __forceinline__ void st6(uint32_t taddr, int wg, const uint32_t (&r)[kHPW]) {
  if (wg == 0) {
    tmem_st4(taddr, r);
    tmem_st2(taddr + 4, r + 4);
  } else {
    tmem_st2(taddr + 6, r);
    tmem_st4(taddr + 8, r + 2);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    flash_gather_kernel(const __grid_constant__ CUtensorMap map_q, const __half* __restrict__ khat,
                        const __half* __restrict__ vhat, const int32_t* __restrict__ ids,
                        const __half* __restrict__ gate, __half* __restrict__ out, int pos0, int t_begin, int n_items,
                        int K, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ GBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_red[2][2][4][kHPW];  // [warpgroup][tile parity][quarter][head]
  __shared__ float s_l[2][4][kHPW];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (K + kCells - 1) / kCells;
  const int my_items = (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int U = my_items * n_tiles;  // tiles this CTA processes
  const int rot_step = (int)gridDim.x % n_tiles;     // item rotation step between this CTA's items
  const TileIter it0{0, 0, (int)blockIdx.x % n_tiles};

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&bars.k.full[i], 64);  // the filling warp pair's cp.async arrivals
      mbar_init(&bars.v.full[i], 64);
    }
    for (int i = 0; i < 2 * kRing; ++i) {
      mbar_init(&bars.k.empty[i], 1);
      mbar_init(&bars.v.empty[i], 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], 8);  // the softmax warps, once S^T is read
      mbar_init(&bars.p_full[i], 8);
      mbar_init(&bars.p_free[i], 1);  // PV commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.o_free[i], 8);
    }
    mbar_init(&bars.drain_qk, 1);
    mbar_init(&bars.drain_pv, 1);
    fence_mbar_init();
  }
  // zero the Q^T and P^T buffers: rows 12..15 are never written again
  for (int i = tid; i < (2 * kQBytes + kNS * kPBytes) / 16; i += kThreads)
    *reinterpret_cast<uint4*>(smem + kOffQ + i * 16) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&s_tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_begin();

  // Raw ids of tile u for a producer warp: lane l holds slots l, l+32, l+64, l+96 (kNoSlot past
  // the end of the id row).
  // Loaded a tile ahead and checked only when used, so the loads overlap the copies.
  auto load_ids = [&](const TileIter& ti, int (&dst)[4], int& g_out, int& nkv_out) {
    const int it = blockIdx.x + ti.k * gridDim.x;
    const int t = t_begin + (it >> 1), g = it & 1;
    const int32_t* idrow = ids + ((size_t)t * kGroups + g) * K;
    const int pt = ti.tile(n_tiles);  // tile order rotated per item (see above)
    g_out = g;
    nkv_out = pos0 + t + 1;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int slot = pt * kCells + 32 * x + lane;
      dst[x] = (slot < K) ? __ldg(idrow + slot) : kNoSlot;
    }
  };
  // Ids in [0, n_kv) stay, anything else becomes -1 (a zero row); a bad id in a real slot is
  // reported once per tile by the reporting warp.
  auto check_ids = [&](int (&v)[4], int n_kv, bool report) {
    bool bad = false;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const bool ok = v[x] >= 0 && v[x] < n_kv;
      bad |= !ok && v[x] != kNoSlot;
      if (!ok) v[x] = -1;
    }
    if (report && __any_sync(0xffffffffu, bad) && lane == 0) set_dev_status(status, QSA_DEV_BAD_ID);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ QK issue
    if (lane == 0) {
      const uint32_t idesc_s = idesc_f16_f32(kCells, kNQ, 0, 0);
      const uint32_t sK = smem_u32(smem + kOffK), sQ = smem_u32(smem + kOffQ);
      int f = 0;  // K fill counter
      TileIter ti = it0;
      for (int s = 0; s < U; ++s, ti.advance(n_tiles, rot_step)) {  // S^T(s) = K^(s) . Q^T: two fills of two 64-dim blocks each
        const int k = ti.k, jl = ti.jl;
        if (jl == 0 && !mbar_wait(&bars.q_full[k & 1], (k >> 1) & 1, status, &s_abort)) break;
        if (s >= kNS && !mbar_wait(&bars.s_free[s % kNS], ((s / kNS) - 1) & 1, status, &s_abort)) break;
        const uint64_t bq0 = sdesc_sw128(sQ + (k & 1) * kQBytes, 16, 1024);
        const uint32_t dS = tmem + kColS + (s % kNS) * 16;
        bool ok = true;
        for (int hf = 0; hf < 2; ++hf, ++f) {
          const int slot = f % kRing;
          if (!mbar_wait(&bars.k.full[slot], (f / kRing) & 1, status, &s_abort)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();  // the fill's cp.async writes (generic proxy) before the MMA reads them
          const uint64_t a0 = sdesc_sw128(sK + slot * kSlotBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(dS, a0 + (uint64_t)(((kk >> 2) * kBlkBytes + (kk & 3) * 32) >> 4),
                    bq0 + (uint64_t)(((2 * hf + (kk >> 2)) * (kNQ * 128) + (kk & 3) * 32) >> 4), idesc_s,
                    (hf > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars.k.empty[f % (2 * kRing)]);
        }
        if (!ok) break;
        umma_commit(&bars.s_full[s % kNS]);
        if (jl == n_tiles - 1) umma_commit(&bars.q_empty[k & 1]);
      }
      umma_commit(&bars.drain_qk);
      mbar_wait(&bars.drain_qk, 0, status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ PV issue
    if (lane == 0) {
      const uint32_t idesc_o = idesc_f16_f32(kCells, kNQ, 1, 0);
      const uint32_t sV = smem_u32(smem + kOffV), sP = smem_u32(smem + kOffP);
      int f = 0;  // V fill counter
      TileIter ti = it0;
      for (int u = 0; u < U; ++u, ti.advance(n_tiles, rot_step)) {  // O^T += V^(u)^T . P^T(u): one fill per 128-dim half
        const int k = ti.k, jl = ti.jl, ob = k & 1;
        if (jl == 0 && k >= 2 && !mbar_wait(&bars.o_free[ob], ((k >> 1) & 1) ^ 1, status, &s_abort)) break;
        if (!mbar_wait(&bars.p_full[u % kNS], (u / kNS) & 1, status, &s_abort)) break;
        const uint64_t bp0 = sdesc_sw128(sP + (u % kNS) * kPBytes, 16, 1024);
        bool ok = true;
        for (int h = 0; h < 2; ++h, ++f) {
          const int slot = f % kRing;
          if (!mbar_wait(&bars.v.full[slot], (f / kRing) & 1, status, &s_abort)) { ok = false; break; }
          tc_fence_after();
          fence_proxy_async_smem();
          // MN-major A: the half's two 64-dim atoms 16 KB apart (LBO), 8-cell groups 1 KB apart
          const uint64_t a0 = sdesc_sw128(sV + slot * kSlotBytes, kBlkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < kCells / 16; ++kk)
            umma_ss(tmem + kColO + ob * 32 + h * 16, a0 + (uint64_t)((kk * 2048) >> 4),
                    bp0 + (uint64_t)(((kk >> 2) * (kNQ * 128) + (kk & 3) * 32) >> 4), idesc_o,
                    (jl > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars.v.empty[f % (2 * kRing)]);
        }
        if (!ok) break;
        umma_commit(&bars.p_free[u % kNS]);
      }
      umma_commit(&bars.drain_pv);
      mbar_wait(&bars.drain_pv, 0, status);
    }
    __syncwarp();
  } else if ((warp >= 2 && warp <= 3) || warp >= 12) {
    // ------------------------------------------------------------ gather producers
    // Every fill is half a tile: 128 rows x 256 bytes, copied by one warp pair of the ring's
    // pool (fill f by pair f mod 3; each warp of the pair takes 64 rows).  Instruction i copies
    // rows 2i, 2i+1 (lane: row 2i + lane/16, chunk lane%16 of the half: 64-dim block
    // (lane%16)/8, 16-byte chunk lane%8).
    const bool is_v = warp >= 16;
    const int pw = is_v ? warp - 16 : (warp <= 3 ? warp - 2 : warp - 10);  // 0..5 in the pool
    const int pair = pw >> 1, half_rows = pw & 1;
    Ring& ring = is_v ? bars.v : bars.k;
    uint8_t* ring_base = smem + (is_v ? kOffV : kOffK);
    const __half* base = is_v ? vhat : khat;
    const int ch = lane & 15;
    // Byte offset of this lane's 16-byte chunk in row 2 (i0 + m) + lane / 16 of a fill, past
    // 256 (i0 + m) bytes: i0 is a multiple of 8, so the row's swizzle phase is (2 m + lane / 16) mod 8.
    uint32_t dsw[8];
#pragma unroll
    for (int m = 0; m < 8; ++m)
      dsw[m] = (uint32_t)(128 * (lane >> 4) + (((ch & 7) ^ ((2 * m + (lane >> 4)) & 7)) << 4) + 256 * m);
    int cur[4] = {-1, -1, -1, -1}, nxt[4] = {-1, -1, -1, -1};
    bool cur_valid = false;  // every id of the current tile is in [0, n_kv) (warp-uniform)
    int g_cur = 0, g_nxt = 0, nkv_nxt = 0;
    TileIter ti = it0, ta = it0;  // tile s and tile s + 1 (ids loaded one tile ahead)
    if (U > 0) load_ids(ta, nxt, g_nxt, nkv_nxt);
    ta.advance(n_tiles, rot_step);
    if (warp == 2 && lane == 0) tma_prefetch_desc(&map_q);
    auto fill = [&](int f, int h) -> bool {
      if (f % kPoolPairs != pair) return true;  // fills go round-robin over the pool's pairs
      const int slot = f % kRing;
      if (f >= kRing) {  // fill f - kRing (same slot) consumed
        const int e = f - kRing;
        if (!mbar_wait_warp(&ring.empty[e % (2 * kRing)], (e / (2 * kRing)) & 1, status, &s_abort)) return false;
      }
      const uint32_t dst = smem_u32(ring_base + slot * kSlotBytes + (ch >> 3) * kBlkBytes);
      const __half* src_g = base + (size_t)g_cur * kD + h * 128 + ch * 8;
      // instruction i copies rows 2i, 2i+1; cells are resolved eight instructions at a time
#pragma unroll 1
      for (int i0 = half_rows * (kCells / 4); i0 < (half_rows + 1) * (kCells / 4); i0 += 8) {
        const int sel = pick4(cur, (i0 >> 4) & 3);  // rows 2*i0 .. 2*i0 + 15 share one id register
        const int sbase = ((2 * i0) & 31) + (lane >> 4);  // the lane holding row 2 i0's id, + 2 m for row 2 (i0 + m)
        int cell[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) cell[m] = __shfl_sync(0xffffffffu, sel, sbase + 2 * m);
        const uint32_t d_i0 = dst + 256 * i0;
        if (cur_valid) {  // every slot of the tile holds a valid id: plain copies
#pragma unroll
          for (int m = 0; m < 8; ++m) cp_async16_sh(d_i0 + dsw[m], src_g + (uint32_t)cell[m] * (uint32_t)(kGroups * kD));
        } else {  // a ragged last tile or a bad id: those rows are zero-filled
#pragma unroll
          for (int m = 0; m < 8; ++m)
            cp_async16_zfill(d_i0 + dsw[m], src_g + (uint32_t)max(cell[m], 0) * (uint32_t)(kGroups * kD), cell[m] >= 0);
        }
      }
      cp_async_arrive_noinc(&ring.full[slot]);
      return true;
    };
    int f = 0;
    for (int s = 0; s < U; ++s, ti = ta, ta.advance(n_tiles, rot_step)) {
      check_ids(nxt, nkv_nxt, warp == 2);  // tile s: loaded during the previous step
#pragma unroll
      for (int x = 0; x < 4; ++x) cur[x] = nxt[x];
      cur_valid = __all_sync(0xffffffffu, (cur[0] | cur[1] | cur[2] | cur[3]) >= 0);
      g_cur = g_nxt;
      // the next tile's ids, if this warp's pair fills in it (fills 2 (s + 1) and 2 (s + 1) + 1 go to pairs
      // f mod 3); warp 2 always, for the item's Q tile and the bad-id report
      const int f1 = 2 * (s + 1) % kPoolPairs;
      if (s + 1 < U && (warp == 2 || f1 == pair || (f1 + 1) % kPoolPairs == pair)) load_ids(ta, nxt, g_nxt, nkv_nxt);
      const int k = ti.k, jl = ti.jl;
      if (jl == 0 && warp == 2) {
        // Q^T tile for this item by TMA: per 64-dim block the group's 12 head rows land as
        // rows 0..11 of a 128B-swizzled [16][64] block (rows 12..15 stay zero)
        const int it = blockIdx.x + k * gridDim.x;
        const int t = t_begin + (it >> 1);
        if (k >= 2 && !mbar_wait_warp(&bars.q_empty[k & 1], ((k >> 1) & 1) ^ 1, status, &s_abort)) break;
        if (lane == 0) {
          uint8_t* qb = smem + kOffQ + (k & 1) * kQBytes;
          mbar_arrive_expect_tx(&bars.q_full[k & 1], kNB * kHPG * 128);
#pragma unroll
          for (int b = 0; b < kNB; ++b)
            tma_load_2d(qb + b * (kNQ * 128), &map_q, &bars.q_full[k & 1], b * 64, t * kHeads + g_cur * kHPG);
        }
        __syncwarp();
      }
      if (!fill(f++, 0) || !fill(f++, 1)) break;
    }
    cp_async_wait_all();  // nothing of ours may land after the CTA exits
  } else if (warp >= 4 && warp <= 11) {
    // ------------------------------------------------------------ softmax (thread = cell)
    const int wg = warp >= 8 ? 1 : 0;
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;  // cell slot in the tile == TMEM lane
    const int h0 = wg * kHPW;           // this warpgroup's first head
    const uint32_t bar_id = 1 + wg;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t sP = smem_u32(smem + kOffP);
    // this cell's byte offsets in a P^T buffer for the warpgroup's six heads (K-major SW128: 64-cell
    // blocks of [16 rows][128 B]; head row h, chunk (cell mod 64) / 8 swizzled by h mod 8)
    uint32_t poff[kHPW];
#pragma unroll
    for (int j = 0; j < kHPW; ++j) {
      const int h = h0 + j;
      poff[j] = (uint32_t)((i >> 6) * (kNQ * 128) + h * 128 + ((((i & 63) >> 3) ^ (h & 7)) << 4) + (i & 7) * 2);
    }
    int u = 0;
    bool ok = true;
    for (int it = blockIdx.x, k = 0; ok && it < n_items; it += gridDim.x, ++k) {
      const int t = t_begin + (it >> 1), g = it & 1;
      const int n_kv = pos0 + t + 1;
      const int32_t* idrow = ids + ((size_t)t * kGroups + g) * K;
      float m_run[kHPW], l_part[kHPW];
#pragma unroll
      for (int j = 0; j < kHPW; ++j) {
        m_run[j] = -INFINITY;
        l_part[j] = 0.f;
      }
      int last_v = -1;
      // the item's tiles are taken in rotated order, as the producers fill them
      const int rot = it % n_tiles;
      auto slot_of = [&](int jl) {
        const int p = jl + rot;
        return (p >= n_tiles ? p - n_tiles : p) * kCells + i;
      };
      int c_next = (slot_of(0) < K) ? idrow[slot_of(0)] : -1;  // this lane's id, one tile ahead
      for (int jl = 0; jl < n_tiles; ++jl, ++u) {
        const int c_cur = c_next;
        const bool valid = slot_of(jl) < K && c_cur >= 0 && c_cur < n_kv;
        const int slot_next = slot_of(jl + 1);
        c_next = (jl + 1 < n_tiles && slot_next < K) ? idrow[slot_next] : -1;
        const bool w_ok = mbar_wait_warp(&bars.s_full[u % kNS], (u / kNS) & 1, status, &s_abort);
        if (named_bar_any(bar_id, 128, !w_ok)) { ok = false; break; }  // the warpgroup leaves together
        tc_fence_after();
        uint32_t sr[kHPW];
        ld6(lane_base + kColS + (u % kNS) * 16, wg, sr);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_free[u % kNS]);  // QK(u + kNS) may overwrite S^T(u)
        float s[kHPW];
        bool high = jl == 0;  // the item's first tile always sets the running maxima
#pragma unroll
        for (int j = 0; j < kHPW; ++j) {
          s[j] = valid ? __uint_as_float(sr[j]) * scale_log2 : -INFINITY;
          high |= s[j] > m_run[j] + kRescaleThreshold;
        }
        // The column maxima are needed only when some score of the tile exceeds its head's running
        // maximum by more than the rescale threshold: otherwise P = exp2(s - m_run) <= 2^8 as
        // with any lazily rescaled tile, and one barrier-reduction replaces the shuffle maxima.
        bool need_any = false;
        float alpha[kHPW];
#pragma unroll
        for (int j = 0; j < kHPW; ++j) alpha[j] = 1.f;
        if (named_bar_any(bar_id, 128, high)) {  // uniform over the warpgroup
#pragma unroll
          for (int j = 0; j < kHPW; ++j) {
            float m = s[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            if (lane == 0) s_red[wg][u & 1][quarter][j] = m;
          }
          named_bar_any(bar_id, 128, false);
#pragma unroll
          for (int j = 0; j < kHPW; ++j) {
            const float mt = fmaxf(fmaxf(s_red[wg][u & 1][0][j], s_red[wg][u & 1][1][j]),
                                   fmaxf(s_red[wg][u & 1][2][j], s_red[wg][u & 1][3][j]));
            const float mn = fmaxf(m_run[j], mt);
            if (jl == 0) {
              m_run[j] = mn;
            } else if (mn > m_run[j] + kRescaleThreshold) {
              alpha[j] = fast_exp2(m_run[j] - mn);
              m_run[j] = mn;
              need_any = true;
            }
          }
        }
        if (need_any) {  // uniform over the warpgroup: derived from the same shared maxima
          const bool r_ok = mbar_wait_warp(&bars.p_free[(u - 1) % kNS], ((u - 1) / kNS) & 1, status, &s_abort);
          if (named_bar_any(bar_id, 128, !r_ok)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[kHPW];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t col = kColO + (k & 1) * 32 + half * 16;
            ld6(lane_base + col, wg, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < kHPW; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha[j]);
            st6(lane_base + col, wg, o);
          }
          tmem_wait_st();
#pragma unroll
          for (int j = 0; j < kHPW; ++j) l_part[j] *= alpha[j];
        }
        // P^T(u) reuses the buffer of P^T(u - kNS): PV(u - kNS) must be done with it
        if (u >= kNS) {
          const bool f_ok = mbar_wait_warp(&bars.p_free[u % kNS], ((u / kNS) - 1) & 1, status, &s_abort);
          if (named_bar_any(bar_id, 128, !f_ok)) { ok = false; break; }
        }
        // P^T[h][i] (K-major SW128: 64-cell blocks of [16 rows][128 B])
        const uint32_t pb = sP + (u % kNS) * kPBytes;
#pragma unroll
        for (int j = 0; j < kHPW; ++j) {
          const float p = fast_exp2(s[j] - ((m_run[j] == -INFINITY) ? 0.f : m_run[j]));
          l_part[j] += p;
          const __half hp = __float2half_rn(p);
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(pb + poff[j]), "h"(__half_as_ushort(hp)) : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[u % kNS]);
        last_v = u;
      }
      if (!ok) break;
      // row sums over the 128 cell lanes
#pragma unroll
      for (int j = 0; j < kHPW; ++j) {
        float l = l_part[j];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) s_l[wg][quarter][j] = l;
      }
      named_bar_any(bar_id, 128, false);
      float inv_l[kHPW];
#pragma unroll
      for (int j = 0; j < kHPW; ++j) {
        const float l = s_l[wg][0][j] + s_l[wg][1][j] + s_l[wg][2][j] + s_l[wg][3][j];
        inv_l[j] = l > 0.f ? 1.f / l : 0.f;
      }
      const bool e_ok = mbar_wait_warp(&bars.p_free[last_v % kNS], (last_v / kNS) & 1, status, &s_abort);
      if (named_bar_any(bar_id, 128, !e_ok)) { ok = false; break; }
      tc_fence_after();
      // epilogue: thread = dim i (half 0) and 128 + i (half 1)
      __half* orow = out + ((size_t)t * kHeads + g * kHPG + h0) * kD;
      const __half* grow = gate ? gate + ((size_t)t * kHeads + g * kHPG + h0) * kD : nullptr;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[kHPW];
        ld6(lane_base + kColO + (k & 1) * 32 + half * 16, wg, o);
        float gs[kHPW];  // output gate: sigmoid(gate) per element, 1 without a gate
#pragma unroll
        for (int j = 0; j < kHPW; ++j) gs[j] = grow ? gate_sigmoid(__half2float(grow[j * kD + half * 128 + i])) : 1.f;
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kHPW; ++j)
          orow[j * kD + half * 128 + i] = __float2half_rn(__uint_as_float(o[j]) * inv_l[j] * gs[j]);
      }
      tc_fence_before();
      named_bar_any(bar_id, 128, false);  // s_l may be rewritten by the next item only after everyone read it
      if (lane == 0) mbar_arrive(&bars.o_free[k & 1]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

// q as rows (token * 24 + head) x 256 halves; boxes of 64 halves x 12 rows (one group's heads),
// 128B swizzle.
bool make_q_map(CUtensorMap* map, const __half* q, int T) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)T * kHeads};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)kHPG};
  const cuuint32_t estr[2] = {1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_flash_gather(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                                cudaStream_t stream) {
  if (t_end <= t_begin) return cudaSuccess;
  // per device, set once (0 = not yet): the shared-memory attribute is set and the SM count read;
  // threads that race here both set the same attribute and store the same count
  static std::atomic<int> n_sms[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return cudaErrorInvalidDevice;
  int sms = n_sms[dev].load(std::memory_order_acquire);
  if (sms == 0) {
    cudaError_t e = cudaFuncSetAttribute(flash_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (sms < 1) return cudaErrorInvalidConfiguration;
    n_sms[dev].store(sms, std::memory_order_release);
  }
  const int n_items = (t_end - t_begin) * kGroups;
  const int grid = n_items < sms ? n_items : sms;
  const float scale_log2 = a.p.sm_scale * kLog2e;
  CUtensorMap mq;
  if (!make_q_map(&mq, a.q, a.T)) return cudaErrorInvalidValue;
  return launch_pdl(flash_gather_kernel, dim3(grid), dim3(kThreads), kSmemAlloc, stream, mq, khat, vhat, a.ids, a.gate,
                    a.out, a.pos0, t_begin, n_items, a.p.topk, scale_log2, a.status);
}

}  // namespace qsa
