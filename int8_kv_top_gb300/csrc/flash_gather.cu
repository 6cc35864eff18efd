// qsa_flash_prefill, selected tokens (n_kv > identity_max): attention of one token's 12
// group heads over its own top-k cell set, on the tcgen05 tensor cores.
//
// In the pages, qsa_flash reads explicit selected ids above the budget (per token, grid
// (2, T); "round 6 track b - qsa flash", delivered change) and hoists per-cell byte offsets
// and zero scales for invalid cells ("round 14 track b: qsa metadata hoist", decision and
// correctness).  Here each (token, group) has its own 2048 cells, so there is no K/V tile
// shared across tokens; the MMA is swapped so the gathered cells form the 128-wide M side:
//
//   S^T[c][h]  = K^[c] . q[h]      A = K^ (128 cells, K-major)  B = Q^T (16 rows, 12 used)
//   O^T[d][h] += V^[c][d] P[h][c]  A = V^ as MN-major (dims x cells)  B = P^T (K-major)
//
//   warps 1, 2  gather producers: 16-byte cp.async copies of the selected cell rows (256
//               code bytes; each warp instruction moves two rows) and scale rows into K and
//               V staging rings of two 64-cell half-tiles; V runs one tile behind K, in the
//               order the MMAs need them (row-sized TMA bulk copies were issue-bound)
//   warps 8-11  dequantise staged K rows with their fp16 scales into the 128B-swizzled K^
//               tile (and load each item's Q^T tile); warps 12-15 do the same for V^
//   warp 0      TMEM owner and single-thread UMMA issue
//   warps 4-7   one gathered cell per thread (TMEM lane): column-wise online softmax over
//               the 128 cells (shuffle + shared-memory max per head, base-2 exponent),
//               fp16 P^T into shared memory, lazy O^T rescale, epilogue (thread = dim)
//
// The CTA is persistent over (token, group) work items.  TMEM: S^T double buffer [0,32),
// O^T double buffer (two 16-column halves for dims 0-127 / 128-255) [32,96).
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kCells = 128;                  // gathered cells per tile (UMMA M)
constexpr int kNQ = 16;                      // UMMA N: 12 heads + 4 zero rows
constexpr int kThreads = 512;
constexpr int kTileHalf = kCells * kD * 2;   // 64 KB fp16 tile
constexpr int kQBytes = kNQ * kD * 2;        // 8 KB
constexpr int kPBytes = kNQ * kCells * 2;    // 4 KB
constexpr int kHalfCells = 64;                               // cells per staging half-tile
constexpr int kStageCodes = kHalfCells * kD;                   // 16 KB of int8 codes
constexpr int kStageIds = kStageCodes + kHalfCells * 16;       // after one 16-byte scale row per cell
constexpr int kStageBytes = kStageIds + kHalfCells * 4;        // + the half-tile's cell ids
constexpr int kOffK = 0, kOffV = kTileHalf, kOffQ = 2 * kTileHalf, kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffKSt = kOffP + 2 * kPBytes, kOffVSt = kOffKSt + 2 * kStageBytes;
constexpr int kSmemTotal = kOffVSt + 2 * kStageBytes;
constexpr int kSmemAlloc = kSmemTotal + 1024;
constexpr uint32_t kColS = 0, kColO = 32;
constexpr float kRescaleThreshold = 8.0f;

struct __align__(8) GBars {
  uint64_t kst_full[2], kst_empty[2], vst_full[2], vst_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t kh_full, kh_empty, vh_full, vh_empty;
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t drain;
};

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    flash_gather_kernel(const __half* __restrict__ q, const int8_t* __restrict__ kq, const int8_t* __restrict__ vq,
                        const __half* __restrict__ ksc, const __half* __restrict__ vsc,
                        const int32_t* __restrict__ ids, __half* __restrict__ out, int pos0, int t_begin, int n_items,
                        int K, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ GBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_red[2][4][kHPG];
  __shared__ float s_l[4][kHPG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (K + kCells - 1) / kCells;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.kst_full[i], 33);  // 32 cp.async completions + the ids' release
      mbar_init(&bars.kst_empty[i], 4);
      mbar_init(&bars.vst_full[i], 33);
      mbar_init(&bars.vst_empty[i], 4);
      mbar_init(&bars.q_full[i], 4);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.o_done[i], 1);
      mbar_init(&bars.o_free[i], 4);
    }
    mbar_init(&bars.kh_full, 4);
    mbar_init(&bars.kh_empty, 1);
    mbar_init(&bars.vh_full, 4);
    mbar_init(&bars.vh_empty, 1);
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  // zero Q^T rows 12..15 and P^T rows 12..15 of both buffers (never written again)
  for (int i = tid; i < 2 * (kQBytes + kPBytes) / 16; i += kThreads) {
    const int qi = 2 * kQBytes / 16;
    uint8_t* p = (i < qi) ? smem + kOffQ + i * 16 : smem + kOffP + (i - qi) * 16;
    *reinterpret_cast<uint4*>(p) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&s_tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ------------------------------------------------------------ UMMA issue
    if (lane == 0) {
      const uint32_t idesc_s = idesc_f16_f32(kCells, kNQ, 0, 0);
      const uint32_t idesc_o = idesc_f16_f32(kCells, kNQ, 1, 0);
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP);
      bool ok = true;
      int u = 0;  // global tile counter of this CTA
      auto issue_pv = [&](int v, int jl, int k) -> bool {
        const int b = v & 1, ob = k & 1;
        if (jl == 0 && k >= 2 && !mbar_wait(&bars.o_free[ob], ((k >> 1) & 1) ^ 1, status, &s_abort)) return false;
        if (!mbar_wait(&bars.p_full[b], (v >> 1) & 1, status, &s_abort)) return false;
        if (!mbar_wait(&bars.vh_full, v & 1, status, &s_abort)) return false;
        tc_fence_after();
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int kk = 0; kk < kCells / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sV + half * 2 * (kCells * 128) + kk * 2048, kCells * 128, 1024);
            const uint64_t bd = sdesc_sw128(sP + b * kPBytes + (kk >> 2) * (kNQ * 128) + (kk & 3) * 32, 16, 1024);
            umma_ss(tmem + kColO + ob * 32 + half * 16, ad, bd, idesc_o, (jl > 0 || kk > 0) ? 1u : 0u);
          }
        umma_commit(&bars.vh_empty);
        umma_commit(&bars.o_done[b]);
        return true;
      };
      int prev_v = -1, prev_jl = 0, prev_k = 0;
      for (int it = blockIdx.x, k = 0; ok && it < n_items; it += gridDim.x, ++k) {
        if (!mbar_wait(&bars.q_full[k & 1], (k >> 1) & 1, status, &s_abort)) { ok = false; break; }
        for (int jl = 0; jl < n_tiles; ++jl, ++u) {
          if (!mbar_wait(&bars.kh_full, u & 1, status, &s_abort)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sK + (kk >> 2) * (kCells * 128) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sQ + (k & 1) * kQBytes + (kk >> 2) * (kNQ * 128) + (kk & 3) * 32, 16, 1024);
            umma_ss(tmem + kColS + (u & 1) * 16, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(&bars.s_full[u & 1]);
          umma_commit(&bars.kh_empty);
          if (jl == n_tiles - 1) umma_commit(&bars.q_empty[k & 1]);
          if (prev_v >= 0 && !issue_pv(prev_v, prev_jl, prev_k)) { ok = false; break; }
          prev_v = u;
          prev_jl = jl;
          prev_k = k;
        }
      }
      if (ok && prev_v >= 0) issue_pv(prev_v, prev_jl, prev_k);
      umma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0, status);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax (thread = cell)
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;  // cell slot in the tile == TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    uint8_t* sP = smem + kOffP;
    int u = 0;
    bool ok = true;
    for (int it = blockIdx.x, k = 0; ok && it < n_items; it += gridDim.x, ++k) {
      const int t = t_begin + (it >> 1), g = it & 1;
      const int n_kv = pos0 + t + 1;
      const int32_t* idrow = ids + ((size_t)t * kGroups + g) * K;
      float m_run[kHPG], l_part[kHPG];
#pragma unroll
      for (int h = 0; h < kHPG; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
      }
      int last_v = -1;
      for (int jl = 0; jl < n_tiles; ++jl, ++u) {
        const int slot = jl * kCells + i;
        bool valid = slot < K;
        if (valid) {
          const int c = idrow[slot];
          valid = c >= 0 && c < n_kv;
        }
        const bool w_ok = mbar_wait_warp(&bars.s_full[u & 1], (u >> 1) & 1, status, &s_abort);
        if (named_bar_any(1, 128, !w_ok)) { ok = false; break; }  // all four warps leave together
        tc_fence_after();
        uint32_t sr[16];
        tmem_ld16(lane_base + kColS + (u & 1) * 16, sr);
        tmem_wait_ld();
        float s[kHPG];
#pragma unroll
        for (int h = 0; h < kHPG; ++h) {
          s[h] = valid ? __uint_as_float(sr[h]) * scale_log2 : -INFINITY;
          float m = s[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) s_red[u & 1][quarter][h] = m;
        }
        softmax_bar();
        bool need_any = false;
        float alpha[kHPG];
#pragma unroll
        for (int h = 0; h < kHPG; ++h) {
          const float mt = fmaxf(fmaxf(s_red[u & 1][0][h], s_red[u & 1][1][h]), fmaxf(s_red[u & 1][2][h], s_red[u & 1][3][h]));
          const float mn = fmaxf(m_run[h], mt);
          alpha[h] = 1.f;
          if (jl == 0) {
            m_run[h] = mn;
          } else if (mn > m_run[h] + kRescaleThreshold) {
            alpha[h] = fast_exp2(m_run[h] - mn);
            m_run[h] = mn;
            need_any = true;
          }
        }
        if (need_any) {  // uniform: every thread derived it from the same shared maxima
          const bool r_ok = mbar_wait_warp(&bars.o_done[(u - 1) & 1], ((u - 1) >> 1) & 1, status, &s_abort);
          if (named_bar_any(1, 128, !r_ok)) { ok = false; break; }
          tc_fence_after();
          uint32_t o[16];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t col = kColO + (k & 1) * 32 + half * 16;
            tmem_ld16(lane_base + col, o);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kHPG; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st16(lane_base + col, o);
          }
          tmem_wait_st();
#pragma unroll
          for (int h = 0; h < kHPG; ++h) l_part[h] *= alpha[h];
        }
        // P^T[h][i] (K-major SW128: 64-cell blocks of [16 rows][128 B])
        uint8_t* pb = sP + (u & 1) * kPBytes + (i >> 6) * (kNQ * 128);
#pragma unroll
        for (int h = 0; h < kHPG; ++h) {
          const float mu = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
          const float p = fast_exp2(s[h] - mu);
          l_part[h] += p;
          *reinterpret_cast<__half*>(pb + h * 128 + ((((i & 63) >> 3) ^ (h & 7)) << 4) + (i & 7) * 2) =
              __float2half_rn(p);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[u & 1]);
        last_v = u;
      }
      if (!ok) break;
      // row sums over the 128 cell lanes
#pragma unroll
      for (int h = 0; h < kHPG; ++h) {
        float l = l_part[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) s_l[quarter][h] = l;
      }
      softmax_bar();
      float inv_l[kHPG];
#pragma unroll
      for (int h = 0; h < kHPG; ++h) {
        const float l = s_l[0][h] + s_l[1][h] + s_l[2][h] + s_l[3][h];
        inv_l[h] = l > 0.f ? 1.f / l : 0.f;
      }
      const bool e_ok = mbar_wait_warp(&bars.o_done[last_v & 1], (last_v >> 1) & 1, status, &s_abort);
      if (named_bar_any(1, 128, !e_ok)) { ok = false; break; }
      tc_fence_after();
      // epilogue: thread = dim i (half 0) and 128 + i (half 1)
      __half* orow = out + ((size_t)t * kHeads + g * kHPG) * kD;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t o[16];
        tmem_ld16(lane_base + kColO + (k & 1) * 32 + half * 16, o);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kHPG; ++h) orow[h * kD + half * 128 + i] = __float2half_rn(__uint_as_float(o[h]) * inv_l[h]);
      }
      tc_fence_before();
      softmax_bar();  // s_l may be rewritten by the next item only after everyone read it
      if (lane == 0) mbar_arrive(&bars.o_free[k & 1]);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ gather producers
    const bool is_v = warp == 2;
    const int8_t* codes = is_v ? vq : kq;
    const __half* scales = is_v ? vsc : ksc;
    uint64_t* full = is_v ? bars.vst_full : bars.kst_full;
    uint64_t* empty = is_v ? bars.vst_empty : bars.kst_empty;
    uint8_t* st0 = smem + (is_v ? kOffVSt : kOffKSt);
    int h = 0;  // half-tile counter of this ring
    bool ok = true;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const int t = t_begin + (it >> 1), g = it & 1;
      const int n_kv = pos0 + t + 1;
      const int32_t* idrow = ids + ((size_t)t * kGroups + g) * K;
      for (int jl = 0; ok && jl < n_tiles; ++jl) {
        for (int half = 0; half < 2; ++half, ++h) {
          const int s = h & 1;
          if (h >= 2 && !mbar_wait_warp(&empty[s], ((h >> 1) & 1) ^ 1, status, &s_abort)) { ok = false; break; }
          // ids of the half-tile's 64 cells: lane holds cells lane and lane + 32; they go to the
          // stage as well (-1: past the set, -2: out of range, skipped and flagged downstream)
          int id0, id1;
          uint8_t* st = st0 + s * kStageBytes;
          {
            const int s0 = jl * kCells + half * kHalfCells + lane, s1 = s0 + 32;
            id0 = (s0 < K) ? __ldg(idrow + s0) : -1;
            id1 = (s1 < K) ? __ldg(idrow + s1) : -1;
            if (s0 < K && (id0 < 0 || id0 >= n_kv)) id0 = -2;
            if (s1 < K && (id1 < 0 || id1 >= n_kv)) id1 = -2;
            reinterpret_cast<int*>(st + kStageIds)[lane] = id0;
            reinterpret_cast<int*>(st + kStageIds)[lane + 32] = id1;
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
          }
          // codes: 64 rows x 16 chunks of 16 bytes, two rows per warp instruction
#pragma unroll 4
          for (int i = 0; i < kHalfCells / 2; ++i) {
            const int r = 2 * i + (lane >> 4), ch = lane & 15;
            const int a = __shfl_sync(0xffffffffu, id0, r & 31), b = __shfl_sync(0xffffffffu, id1, r & 31);
            const int c = (r < 32) ? a : b;
            if (c >= 0) cp_async16(st + r * kD + ch * 16, codes + ((size_t)c * kGroups + g) * kD + ch * 16);
          }
          // scale rows (both groups, 16 bytes) of cells lane and lane + 32
          if (id0 >= 0) cp_async16(st + kStageCodes + lane * 16, scales + (size_t)id0 * kGroups * kNB);
          if (id1 >= 0) cp_async16(st + kStageCodes + (lane + 32) * 16, scales + (size_t)id1 * kGroups * kNB);
          cp_async_arrive_noinc(&full[s]);
        }
      }
    }
    cp_async_wait_all();  // nothing of ours may land after the CTA exits
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dequantise staged rows
    const bool is_v = warp >= 12;
    const int dw = warp & 3;
    const int blk = lane >> 3;
    uint64_t* st_full = is_v ? bars.vst_full : bars.kst_full;
    uint64_t* st_empty = is_v ? bars.vst_empty : bars.kst_empty;
    uint64_t* t_full = is_v ? &bars.vh_full : &bars.kh_full;
    uint64_t* t_empty = is_v ? &bars.vh_empty : &bars.kh_empty;
    uint8_t* tile = smem + (is_v ? kOffV : kOffK);
    const uint8_t* st0 = smem + (is_v ? kOffVSt : kOffKSt);
    int u = 0, h = 0;
    bool ok = true;
    for (int it = blockIdx.x, k = 0; ok && it < n_items; it += gridDim.x, ++k) {
      const int t = t_begin + (it >> 1), g = it & 1;
      if (!is_v) {
        // Q^T tile for this item: rows 0..11 = the group's heads (rows 12..15 stay zero)
        if (k >= 2 && !mbar_wait_warp(&bars.q_empty[k & 1], ((k >> 1) & 1) ^ 1, status, &s_abort)) break;
        uint8_t* qb = smem + kOffQ + (k & 1) * kQBytes;
        const __half* qt = q + ((size_t)t * kHeads + g * kHPG) * kD;
        for (int x = dw * 32 + lane; x < kHPG * 32; x += 128) {
          const int hh = x >> 5, ch = x & 31;  // 16-byte chunk ch of row hh
          const uint4 v = *reinterpret_cast<const uint4*>(qt + hh * kD + ch * 8);
          *reinterpret_cast<uint4*>(qb + (ch >> 3) * (kNQ * 128) + hh * 128 + (((ch & 7) ^ (hh & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.q_full[k & 1]);
      }
      for (int jl = 0; ok && jl < n_tiles; ++jl, ++u) {
        if (u >= 1 && !mbar_wait_warp(t_empty, (u - 1) & 1, status, &s_abort)) { ok = false; break; }
        for (int half = 0; half < 2; ++half, ++h) {
          const int s = h & 1;
          if (!mbar_wait_warp(&st_full[s], (h >> 1) & 1, status, &s_abort)) { ok = false; break; }
          const uint8_t* st = st0 + s * kStageBytes;
#pragma unroll 4
          for (int x = 0; x < 16; ++x) {
            const int r = dw * 16 + x;            // row within the half-tile
            const int row = half * kHalfCells + r;  // row within the tile
            int c = reinterpret_cast<const int*>(st + kStageIds)[r];
            if (c == -2) {
              if (!is_v && lane == 0) set_dev_status(status, QSA_DEV_BAD_ID);
              c = -1;
            }
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (c >= 0) {
              const uint2 w = *reinterpret_cast<const uint2*>(st + r * kD + lane * 8);
              const __half sc = *reinterpret_cast<const __half*>(st + kStageCodes + r * 16 + (g * kNB + blk) * 2);
              dequant8(w.x, w.y, __half2half2(sc), o);
            }
            *reinterpret_cast<uint4*>(tile + blk * (kCells * 128) + row * 128 + (((lane & 7) ^ (row & 7)) << 4)) =
                make_uint4(o[0], o[1], o[2], o[3]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&st_empty[s]);
        }
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(t_full);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

cudaError_t launch_flash_gather(const FlashArgs& a, int t_begin, int t_end, cudaStream_t stream) {
  if (t_end <= t_begin) return cudaSuccess;
  static bool attr_done[64] = {};
  static int n_sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(flash_gather_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    cudaDeviceGetAttribute(&n_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    attr_done[dev] = true;
  }
  const int n_items = (t_end - t_begin) * kGroups;
  const int sms = (dev < 64 && n_sms[dev] > 0) ? n_sms[dev] : 148;
  const int grid = n_items < sms ? n_items : sms;
  const float scale_log2 = a.p.sm_scale * kLog2e;
  flash_gather_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(a.q, a.kq, a.vq, a.ksc, a.vsc, a.ids, a.out, a.pos0,
                                                              t_begin, n_items, a.p.topk, scale_log2, a.status);
  return cudaGetLastError();
}

}  // namespace qsa
