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
//     warp 0      TMEM owner and single-thread UMMA issue
//     warps 1-3, 8-11  gather producers; three 64 KB tile buffers rotate in the order the MMAs
//                 consume them (K0, K1, V0, K2, V1, ...), so each load has ~1.5 tiles of lead;
//                 warp 1 also stages each item's Q^T tile
//     warps 4-7   one gathered cell per thread (TMEM lane): column-wise online softmax over
//                 the 128 cells (shuffle + shared-memory max per head, base-2 exponent),
//                 fp16 P^T into shared memory, lazy O^T rescale, epilogue (thread = dim)
// The CTA is persistent over (token, group) work items.  TMEM: S^T double buffer [0,32),
// O^T double buffer (two 16-column halves for dims 0-127 / 128-255) [32,96).
#include "common.cuh"

namespace qsa {
namespace {

constexpr int kCells = 128;                  // gathered cells per tile (UMMA M)
constexpr int kNQ = 16;                      // UMMA N: 12 heads + 4 zero rows
constexpr int kThreads = 384;
constexpr int kProdWarps = 7;                // warps 1-3 and 8-11
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kTileBytes = kCells * kD * 2;  // 64 KB fp16 tile
constexpr int kQBytes = kNQ * kD * 2;        // 8 KB
constexpr int kPBytes = kNQ * kCells * 2;    // 4 KB
constexpr int kNBuf = 3;
constexpr int kOffX = 0, kOffQ = kNBuf * kTileBytes, kOffP = kOffQ + 2 * kQBytes;
constexpr int kSmemTotal = kOffP + 2 * kPBytes;
constexpr int kSmemAlloc = kSmemTotal + 1024;
constexpr uint32_t kColS = 0, kColO = 32;
constexpr float kRescaleThreshold = 8.0f;

struct __align__(8) GBars {
  uint64_t x_full[kNBuf], x_empty[kNBuf];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t drain;
};

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// 16-byte copy that writes zeros (and reads nothing) when `valid` is false.
__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

// Entry j of the load/consume sequence: K(0), K(1), V(0), K(2), V(1), ..., K(U-1), V(U-2), V(U-1).
__device__ __forceinline__ void seq_entry(int j, int U, int* tile, int* is_v) {
  if (j == 0) {
    *tile = 0;
    *is_v = 0;
  } else if (j == 2 * U - 1) {
    *tile = U - 1;
    *is_v = 1;
  } else if (j & 1) {  // j = 2u - 1 -> K(u), u >= 1
    *tile = (j + 1) >> 1;
    *is_v = 0;
  } else {  // j = 2u -> V(u - 1)
    *tile = (j >> 1) - 1;
    *is_v = 1;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    flash_gather_kernel(const __half* __restrict__ q, const __half* __restrict__ khat,
                        const __half* __restrict__ vhat, const int32_t* __restrict__ ids, __half* __restrict__ out,
                        int pos0, int t_begin, int n_items, int K, float scale_log2, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ GBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float s_red[2][4][kHPG];
  __shared__ float s_l[4][kHPG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (K + kCells - 1) / kCells;
  const int my_items = (n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int U = my_items * n_tiles;  // tiles this CTA processes

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kNBuf; ++i) {
      mbar_init(&bars.x_full[i], kProdThreads);  // one cp.async completion arrival per producer
      mbar_init(&bars.x_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.o_done[i], 1);
      mbar_init(&bars.o_free[i], 4);
    }
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
      const uint32_t sX = smem_u32(smem + kOffX), sQ = smem_u32(smem + kOffQ), sP = smem_u32(smem + kOffP);
      bool ok = true;
      for (int j = 0; ok && j < 2 * U; ++j) {
        int u, is_v;
        seq_entry(j, U, &u, &is_v);
        const int k = u / n_tiles, jl = u % n_tiles;  // item (local) and tile within it
        const int buf = j % kNBuf;
        const uint32_t xb = sX + buf * kTileBytes;
        if (!is_v) {
          if (jl == 0 && !mbar_wait(&bars.q_full[k & 1], (k >> 1) & 1, status, &s_abort)) { ok = false; break; }
          if (!mbar_wait(&bars.x_full[buf], (j / kNBuf) & 1, status, &s_abort)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad0 = sdesc_sw128(xb, 16, 1024), bd0 = sdesc_sw128(sQ + (k & 1) * kQBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)
            umma_ss(tmem + kColS + (u & 1) * 16, ad0 + (uint64_t)(((kk >> 2) * (kCells * 128) + (kk & 3) * 32) >> 4),
                    bd0 + (uint64_t)(((kk >> 2) * (kNQ * 128) + (kk & 3) * 32) >> 4), idesc_s, kk > 0 ? 1u : 0u);
          umma_commit(&bars.s_full[u & 1]);
          umma_commit(&bars.x_empty[buf]);
          if (jl == n_tiles - 1) umma_commit(&bars.q_empty[k & 1]);
        } else {
          const int b = u & 1, ob = k & 1;
          if (jl == 0 && k >= 2 && !mbar_wait(&bars.o_free[ob], ((k >> 1) & 1) ^ 1, status, &s_abort)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&bars.p_full[b], (u >> 1) & 1, status, &s_abort)) { ok = false; break; }
          if (!mbar_wait(&bars.x_full[buf], (j / kNBuf) & 1, status, &s_abort)) { ok = false; break; }
          tc_fence_after();
          const uint64_t av0 = sdesc_sw128(xb, kCells * 128, 1024), bp0 = sdesc_sw128(sP + b * kPBytes, 16, 1024);
#pragma unroll
          for (int half = 0; half < 2; ++half)
#pragma unroll
            for (int kk = 0; kk < kCells / 16; ++kk)
              umma_ss(tmem + kColO + ob * 32 + half * 16,
                      av0 + (uint64_t)((half * 2 * (kCells * 128) + kk * 2048) >> 4),
                      bp0 + (uint64_t)(((kk >> 2) * (kNQ * 128) + (kk & 3) * 32) >> 4), idesc_o,
                      (jl > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars.x_empty[buf]);
          umma_commit(&bars.o_done[b]);
        }
      }
      umma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0, status);
    }
    __syncwarp();
  } else if ((warp >= 1 && warp <= 3) || warp >= 8) {
    // ------------------------------------------------------------ gather producers
    const int pw = warp <= 3 ? warp - 1 : warp - 5;  // 0..6: rows pw, pw + 7, ... of every 32-row group
    // ids of entry j's tile, lane l holding rows l, l+32, l+64, l+96 (-1: none); loaded one
    // entry ahead so the copies never wait on them
    auto load_ids = [&](int j, int (&dst)[4]) {
      int u, is_v;
      seq_entry(j, U, &u, &is_v);
      const int k = u / n_tiles, jl = u % n_tiles;
      const int it = blockIdx.x + k * gridDim.x;
      const int t = t_begin + (it >> 1), g = it & 1;
      const int n_kv = pos0 + t + 1;
      const int32_t* idrow = ids + ((size_t)t * kGroups + g) * K;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int slot = jl * kCells + 32 * x + lane;
        int c = (slot < K) ? __ldg(idrow + slot) : -1;
        if (c >= n_kv || (c < 0 && slot < K)) {
          if (!is_v && pw == 0) set_dev_status(status, QSA_DEV_BAD_ID);
          c = -1;
        }
        dst[x] = c;
      }
    };
    // one entry's work, given its ids (returns false if a wait gave up)
    auto produce = [&](int j, const int (&cur)[4]) -> bool {
      int u, is_v;
      seq_entry(j, U, &u, &is_v);
      const int k = u / n_tiles, jl = u % n_tiles;
      const int it = blockIdx.x + k * gridDim.x;
      const int t = t_begin + (it >> 1), g = it & 1;
      if (!is_v && jl == 0 && warp == 1) {
        // Q^T tile for this item: rows 0..11 = the group's heads (rows 12..15 stay zero)
        if (k >= 2 && !mbar_wait_warp(&bars.q_empty[k & 1], ((k >> 1) & 1) ^ 1, status, &s_abort)) return false;
        uint8_t* qb = smem + kOffQ + (k & 1) * kQBytes;
        const __half* qt = q + ((size_t)t * kHeads + g * kHPG) * kD;
        for (int x = lane; x < kHPG * 32; x += 32) {
          const int hh = x >> 5, ch = x & 31;  // 16-byte chunk ch of row hh
          const uint4 v = *reinterpret_cast<const uint4*>(qt + hh * kD + ch * 8);
          *reinterpret_cast<uint4*>(qb + (ch >> 3) * (kNQ * 128) + hh * 128 + (((ch & 7) ^ (hh & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.q_full[k & 1]);
      }
      const int buf = j % kNBuf;
      if (j >= kNBuf && !mbar_wait_warp(&bars.x_empty[buf], ((j / kNBuf) & 1) ^ 1, status, &s_abort)) return false;
      uint8_t* xb = smem + kOffX + buf * kTileBytes;
      const __half* src = is_v ? vhat : khat;
      // lane = 16-byte chunk of the row: its k-block and swizzle-free part of the offset
      uint8_t* dst_l = xb + (lane >> 3) * (kCells * 128);
      const __half* src_l = src + (size_t)g * kD + lane * 8;
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        for (int rr = pw; rr < 32; rr += kProdWarps) {
          const int r = 32 * x + rr;
          const int cell = __shfl_sync(0xffffffffu, cur[x], rr);
          cp_async16_zfill(dst_l + r * 128 + (((lane & 7) ^ (r & 7)) << 4),
                           src_l + (size_t)(cell >= 0 ? cell : 0) * (kGroups * kD), cell >= 0);
        }
      }
      cp_async_arrive_noinc(&bars.x_full[buf]);
      return true;
    };
    // ping-pong id sets: entry j+1's ids are in flight while entry j is issued
    int ids_a[4] = {-1, -1, -1, -1}, ids_b[4] = {-1, -1, -1, -1};
    if (U > 0) load_ids(0, ids_a);
    for (int j = 0; j < 2 * U; j += 2) {
      if (j + 1 < 2 * U) load_ids(j + 1, ids_b);
      if (!produce(j, ids_a)) break;
      if (j + 1 >= 2 * U) break;
      if (j + 2 < 2 * U) load_ids(j + 2, ids_a);
      if (!produce(j + 1, ids_b)) break;
    }
    cp_async_wait_all();  // nothing of ours may land after the CTA exits
  } else if (warp >= 4 && warp <= 7) {
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
      int c_next = (i < K) ? idrow[i] : -1;  // id of this lane's cell in tile 0, then one tile ahead
      for (int jl = 0; jl < n_tiles; ++jl, ++u) {
        const int c_cur = c_next;
        const bool valid = jl * kCells + i < K && c_cur >= 0 && c_cur < n_kv;
        const int slot_next = (jl + 1) * kCells + i;
        c_next = (jl + 1 < n_tiles && slot_next < K) ? idrow[slot_next] : -1;
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
          const float mt =
              fmaxf(fmaxf(s_red[u & 1][0][h], s_red[u & 1][1][h]), fmaxf(s_red[u & 1][2][h], s_red[u & 1][3][h]));
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
        for (int h = 0; h < kHPG; ++h)
          orow[h * kD + half * 128 + i] = __float2half_rn(__uint_as_float(o[h]) * inv_l[h]);
      }
      tc_fence_before();
      softmax_bar();  // s_l may be rewritten by the next item only after everyone read it
      if (lane == 0) mbar_arrive(&bars.o_free[k & 1]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 128);
}

}  // namespace

cudaError_t launch_flash_gather(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                                cudaStream_t stream) {
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
  flash_gather_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(a.q, khat, vhat, a.ids, a.out, a.pos0, t_begin, n_items,
                                                              a.p.topk, scale_log2, a.status);
  return cudaGetLastError();
}

}  // namespace qsa
