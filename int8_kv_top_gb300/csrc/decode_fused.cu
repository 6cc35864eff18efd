// qsa_decode_layer / qsa_decode_layer_batched: a whole decode step of the layer in one launch
// (selection, attention over the selected cells and the log-sum-exp merge).
//
// What it computes is the chain select -> partial -> merge of the pages' production decode
// ("round 27 track b - qsa prep and merge", decision: qsa_score, qsa_topk, qsa_attn2 partials,
// qsa_merge2; "round 6 track b - qsa flash", experiment contract: the 2051/2052 budget
// boundary): for token t and group g, the cells are all causal cells while n_kv <= identity_max,
// else the topk cells of largest exact selection score (ties to the lower index), and
//   xp[t, h] = sum_c softmax_c(sm_scale q[t,h] . k^[c]) v^[c],   k^ = kq * ksc, v^ = fp16(vq * vsc).
// The pages split this over five dependent dispatches; on GB300 a decode token's work is a
// few megabytes, so the dispatch chain, not the bytes, set the time.  Here one thread-block
// cluster of C CTAs (C = 2, 4, 8 or 16, chosen per launch) takes one (token, group); CTA r owns the cells
// [r W, (r + 1) W) of the token's n_kv cells, W = ceil(n_kv / C) <= 8192.  The CTAs exchange data by
// PUSHING it into each other's shared memory (remote stores and adds need no round trip; a
// remote load costs hundreds of cycles) and a cluster barrier makes it visible:
//
//  1. score   (selected tokens) the CTA's cells stream through a ring of bulk copies (one
//             256-byte copy per code row); per 16 cells a warp runs mma.sync m16n8k16 with the
//             int8 codes (exact in fp16) as A and the token's Qsum split hi/lo (two fp16 columns,
//             products exact in fp32) as B, one fp32 accumulator per 64-dim scale block:
//             s~ = sm_scale sum_b ksc_b (S_hi,b + S_lo,b).  |s~ - s| <= a + b|s~| rigorously (a from
//             the hi/lo residual, the fp32 accumulation and the roundings; b from the final
//             products).  Each CTA counts its scores in a 4096-bin histogram of the top 12 bits of
//             their order keys.
//  2. threshold  each CTA adds its histogram into the owners of the bin slices (CTA r owns slice
//             r); barrier; every owner broadcasts its merged slice to all CTAs; barrier; every CTA
//             then holds the cluster's histogram and finds the bin holding the topk-th largest
//             score.  With U(f) = f + a + b|f|, L(f) = f - a - b|f| (increasing) and the bin's
//             range [f_lo, f_hi] holding tau (the topk-th largest s~), the exact topk-th score
//             lies in [L(f_lo), U(f_hi)], so cells with L(s~) > U(f_hi) are surely in, cells with
//             U(s~) < L(f_lo) surely out, and the rest are candidates.
//  3. exact   each CTA computes the EXACT 128-bit key of its candidates (every fp16 value is an
//             integer multiple of 2^-24: 2^48 score / sm_scale = sum_b ksc_b 2^24 sum_{d in b}
//             Qsum_d 2^24 kq_d) and pushes them, with its counts, to every CTA; barrier; each CTA
//             ranks its own candidates against all of them by (key desc, index asc) and keeps those
//             ranked below topk - (surely-in count).  The kept cells are exactly the exact top-k.
//             (When some CTA has more candidates than its push slot holds, which takes massive
//             exact ties, every CTA ranks from the others' shared memory instead.)
//  4. attend  the CTA's kept cells (all its cells for identity tokens) are gathered in batches of
//             64 by bulk copies (their V rows were prefetched into L2 once classified), logits by
//             mma.sync (q as A, codes as B), base-2 online softmax in fp32, P (fp16) x V^ (fp16)
//             by mma.sync into fp32 partials.
//  5. merge   each CTA pushes its (m, l) and, to CTA r, the r-th 1/C of its 12 x 256 partial
//             outputs; barrier; CTA r merges its share (M = max m, L = sum l 2^(m - M),
//             xp = sum o 2^(m - M) / L) from its own shared memory.  The ids of selected tokens are
//             written in ascending order from per-CTA offsets.  With a gate input the output is
//             multiplied by sigmoid(gate) before it is stored.
//
// No global scratch and no spin on global memory: the waits are cluster barriers and bounded
// mbarrier waits on the bulk copies.
#include "common.cuh"
#include "select_math.cuh"

namespace qsa {
namespace {

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxW = 8192;          // cells per CTA
constexpr int kOwnCap = 4096;        // a CTA's candidates with exact keys (more: flagged, see below)
constexpr int kHistBins = 4096;      // top 12 bits of the fp32 order key
constexpr int kTile = 256;           // cells per scoring tile: 16 per warp
constexpr int kBoxB = kTile * 128;   // one TMA box: 256 cells x 128 code bytes, 128B-swizzled
constexpr int kStages = 2;           // scoring ring depth
constexpr int kTileBytes = 2 * kBoxB + kTile * 16;  // codes (two boxes), then both groups' 4 K scales per cell
constexpr int kRingBytes = kStages * kTileBytes;
constexpr int kRowB = 272;           // attention: staged code row stride (256 + 16: conflict-free 32-bit reads)
constexpr int kBatch = 64;           // attention batch (cells)
constexpr int kQKWarps = kBatch / 8; // warps that form logits: 8 cells each
constexpr int kDimsPerWarp = kD / kFWarps;  // P.V output dims per warp
static_assert(kDimsPerWarp == 16, "one ldmatrix.x4.trans (two 8-dim tiles) per 16-cell step");
constexpr int kBatchBytes = kBatch * kRowB * 2 + kBatch * 32;  // K rows, V rows, K scales, V scales
constexpr int kVhStride = 264;       // halves per V^ row (528 B: conflict-free ldmatrix)
constexpr int kQStride = 264;        // halves per staged q row
constexpr int kPStride = 72;         // halves per P row
constexpr int kMinC = 2;             // the smallest cluster (largest slice of the histogram per CTA)
constexpr int kCandPush = 1792;      // candidates a CTA receives by push: kCandPush / max(C, 8) per source
constexpr int kDenseOff = 256;       // fast path: own candidates use entries [0, kDenseOff) of their arrays
constexpr int kCandStage = 768;      // remote candidates staged per round (pull fallback)

// shared-memory map (bytes from a 1024-byte aligned base)
constexpr int kOffRing = 0;                                  // scoring ring / candidates / attention
constexpr int kOffQ = kOffRing + kRingBytes;                 // fp16 [12][kQStride]
constexpr int kOffQsum = kOffQ + 12 * kQStride * 2;          // int64 [256] (exact Qsum)
constexpr int kOffHL = kOffQsum + 256 * 8;                   // fp16 hi[256] | lo[256]
constexpr int kOffScore = kOffHL + 512 * 2;                  // f32 [kMaxW]; later the received partials
constexpr int kOffStat = kOffScore + kMaxW * 4;              // u8 [kMaxW]
constexpr int kOffHist = kOffStat + kMaxW;                   // u32 [kHistBins] own, then the cluster's; later u16 kept list
constexpr int kOffSlice = kOffHist + kHistBins * 4;          // u32 [kHistBins / C] the owned bin slice, summed by the others
constexpr int kOffP = kOffSlice + kHistBins / kMinC * 4;     // fp16 [16][kPStride]
constexpr int kOffBar = kOffP + 16 * kPStride * 2;           // mbarriers of the scoring ring
constexpr int kSmemBytes = kOffBar + 8 * 8 + 1024;           // + the alignment slack
// candidates inside the ring region: own keys hi [kOwnCap] | lo [kOwnCap] | index [kOwnCap] |
// received (pushed) hi [kCandPush] | lo | index | staged copy (pull fallback) hi | lo | index
constexpr int kCandHi = kOffRing, kCandLo = kCandHi + kOwnCap * 8, kCandIdx = kCandLo + kOwnCap * 8;
constexpr int kRcvHi = kCandIdx + kOwnCap * 4, kRcvLo = kRcvHi + kCandPush * 8, kRcvIdx = kRcvLo + kCandPush * 8;
constexpr int kStgHi = kRcvIdx + kCandPush * 4, kStgLo = kStgHi + kCandStage * 8, kStgIdx = kStgLo + kCandStage * 8;
static_assert(kStgIdx + kCandStage * 4 <= kOffRing + kRingBytes, "candidates fit the ring region");
// attention inside the ring region: two batch stages, then V^
constexpr int kOffVh = kOffRing + 2 * kBatchBytes;
static_assert(kOffVh + kBatch * kVhStride * 2 <= kOffRing + kRingBytes, "attention buffers fit the ring region");
static_assert(kTileBytes % 1024 == 0 && kBoxB % 1024 == 0, "swizzled boxes start on 1024-byte boundaries");
// received partials inside the score array: o [C][12 * 256 / C], then m, l [C][12] each
static_assert(12 * 256 * 4 + 2 * 16 * 12 * 4 <= kMaxW * 4, "the received partials fit the score array");
static_assert(kMaxW * 2 <= kHistBins * 4, "the kept list fits the histogram array");
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

struct FusedArgs {
  const __half* q;
  const int8_t* kq;
  const int8_t* vq;
  const __half* ksc;
  const __half* vsc;
  const int4* seqs;  // per sequence {first pool cell, n_cells, pos0, first token}; null: one sequence
  int n_seq;
  long long n_pool;  // cells in the pool (bounds of every sequence)
  int n_cells, pos0; // the one sequence when seqs is null
  int32_t* ids;      // [n_tok][2][topk] or null
  const __half* gate;  // [n_tok][24][256] output gate, or null
  float* xp;         // [n_tok][24][256]
  Params p;
  int* status;
  __half* out16;     // [n_tok][24][256] fp16 output instead of xp (a prefill), or null
  int selected_only; // tokens at or under the identity threshold are left to another kernel
  int ids_only;      // the selection alone: ids of selected tokens, no attention (V not read)
};

// ---------------------------------------------------------------- small helpers
__device__ __forceinline__ uint32_t f32_okey(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void red_cluster_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// the two halves of a cluster barrier: arrive releases this thread's prior writes (local and
// remote), wait acquires every other thread's
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// the two 128-byte lines of a 256-byte row into L2
__device__ __forceinline__ void prefetch_l2_256(const void* src) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(src)));
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(src) + 128));
}
// four int8 codes (dims 4j .. 4j+3 of a 16-dim step) -> two half2 of the exact integer values
__device__ __forceinline__ void codes4_to_half(uint32_t w, uint32_t& lo2, uint32_t& hi2) {
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152 = 1024 + 128
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140), b = __byte_perm(u, 0x64646464u, 0x4342);
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias), hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo2 = *reinterpret_cast<uint32_t*>(&ha);
  hi2 = *reinterpret_cast<uint32_t*>(&hb);
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// better(j, i): candidate j ranks ahead of candidate i (larger exact key, then lower index)
__device__ __forceinline__ bool ranks_ahead(long long hj, unsigned long long lj, int ij, long long hi,
                                            unsigned long long li, int ii) {
  return hj != hi ? hj > hi : (lj != li ? lj > li : ij < ii);
}
// block-wide exclusive prefix sum of one int per thread (256 threads)
__device__ __forceinline__ int block_scan(int v, int* s_red, int* total) {
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
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kFWarps; ++w) {
    const int sw = s_red[w];
    base += (w < warp) ? sw : 0;
    tot += sw;
  }
  *total = tot;
  return base + x - v;
}

struct Seq {
  long long cell0;  // first pool cell of the sequence
  int n_kv, tl;     // causal cells of this token, token index within its sequence
  bool ok;
};

__device__ __forceinline__ Seq resolve_seq(const FusedArgs& a, int t) {
  Seq s{0, 0, t, true};
  if (a.seqs == nullptr) {
    s.n_kv = a.pos0 + t + 1;
    return s;
  }
  int lo = 0, hi = a.n_seq - 1;  // last sequence whose first token is <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&a.seqs[mid].w) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int4 e = __ldg(&a.seqs[lo]);
  const int next = lo + 1 < a.n_seq ? __ldg(&a.seqs[lo + 1].w) : (int)gridDim.z;
  s.cell0 = e.x;
  s.tl = t - e.w;
  s.n_kv = e.z + s.tl + 1;
  // the sequence must hold its tokens' cells inside the pool
  s.ok = e.x >= 0 && e.y >= 1 && e.z >= 0 && e.w <= t && t < next && (long long)e.z + (next - e.w) <= e.y &&
         (long long)e.x + e.y <= a.n_pool;
  return s;
}

template <int C>
__global__ void __launch_bounds__(kFThreads, 1)
    decode_fused_kernel(const FusedArgs a, const __grid_constant__ CUtensorMap tm_codes,
                        const __grid_constant__ CUtensorMap tm_scales) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (smem_u32(sm_raw) & 1023u)) & 1023u);
  __shared__ float s_eh[8];               // E_b, H_b
  __shared__ float s_kmax_all[4];         // max |ksc| per block over the cluster (pushed by every CTA)
  __shared__ int s_red[kFWarps];
  __shared__ int s_bin, s_need, s_slow, s_cnt_cand, s_nlist;
  __shared__ float s_bnd[4];              // a, b, U(f_hi), L(f_lo)
  __shared__ float s_wred[kFWarps][16];
  __shared__ int s_ccnt[16][2];           // pushed by CTA q: its surely-in count, its candidate count
  __shared__ int s_nsel_all[16];          // pushed by CTA q: its kept-cell count

  pdl_begin();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, j = lane & 3, r8 = lane >> 2;
  const int r = (int)cluster_ctarank();
  const int g = blockIdx.y, t = blockIdx.z;
  const Params p = a.p;
  const Seq sq = resolve_seq(a, t);
  const int n_kv = sq.n_kv;
  if (!sq.ok || n_kv > C * kMaxW) {  // uniform over the cluster: nobody touches another CTA
    if (tid == 0 && r == 0) set_dev_status(a.status, QSA_DEV_BAD_ID);
    return;
  }
  const bool selected = n_kv > p.identity_max;
  if (!selected && (a.selected_only || a.ids_only)) return;  // uniform over the cluster, before any cluster barrier
  const int K = p.topk;
  const int W = (n_kv + C - 1) / C;
  const int c_lo = r * W, c_hi = min(n_kv, c_lo + W), nloc = max(0, c_hi - c_lo);
  const int8_t* kq = a.kq + sq.cell0 * (kGroups * kD);
  const int8_t* vq = a.vq + sq.cell0 * (kGroups * kD);
  const __half* ksc = a.ksc + sq.cell0 * (kGroups * kNB);
  const __half* vsc = a.vsc + sq.cell0 * (kGroups * kNB);
  __half* s_q = reinterpret_cast<__half*>(sm + kOffQ);
  float* s_score = reinterpret_cast<float*>(sm + kOffScore);
  uint8_t* s_stat = sm + kOffStat;
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(sm + kOffHist);
  uint32_t* s_slice = reinterpret_cast<uint32_t*>(sm + kOffSlice);
  uint16_t* s_list = reinterpret_cast<uint16_t*>(sm + kOffHist);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  bool ok_waits = true;
  // ids of a selected token: this CTA's kept cells (ascending in s_list) at the offset of the
  // CTAs before it, once every CTA's kept count is in s_nsel_all
  auto write_ids = [&](int n_sel) {
    if (a.ids == nullptr) return;
    int off = 0, total = 0;
#pragma unroll
    for (int qq = 0; qq < C; ++qq) {
      const int c = s_nsel_all[qq];
      off += qq < r ? c : 0;
      total += c;
    }
    if (total != p.topk && r == 0 && tid == 0) set_dev_status(a.status, QSA_DEV_BAND_OVERFLOW);
    int32_t* row = a.ids + ((size_t)t * kGroups + g) * p.topk;
    for (int i = tid; i < n_sel; i += kFThreads)
      if (off + i < p.topk) row[off + i] = c_lo + (int)s_list[i];
  };
  // a copy wait that gave up: wait (bounded) for the last phase of every ring barrier used
  auto drain = [&]() {
    if (!ok_waits) {
      const int ntiles = selected ? (nloc + kTile - 1) / kTile : 0;
      for (int s = 0; s < kStages; ++s)
        if (ntiles > s) mbar_wait(&bars[s], (uint32_t)(((ntiles - 1 - s) / kStages) & 1), nullptr);
    }
  };

  // receive buffers that others add into start at zero; then the first half of barrier #0,
  // whose second half (before the first remote access) also guarantees every CTA has started
  for (int i = tid; i < kHistBins / C; i += kFThreads) s_slice[i] = 0u;
  for (int i = tid; i < kHistBins; i += kFThreads) s_hist[i] = 0u;
  if (tid < 4) s_kmax_all[tid] = 0.f;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_arrive();  // #0
  // the group's 12 query rows, fp16
  for (int i = tid; i < 12 * 32; i += kFThreads) {
    const int h = i >> 5, c16 = i & 31;
    *reinterpret_cast<uint4*>(s_q + h * kQStride + c16 * 8) =
        __ldg(reinterpret_cast<const uint4*>(a.q + ((size_t)t * kHeads + g * kHPG + h) * kD) + c16);
  }

  int n_sel = nloc;  // identity: every owned cell
  if (selected) {
    long long* s_qsum = reinterpret_cast<long long*>(sm + kOffQsum);
    __half* s_hl = reinterpret_cast<__half*>(sm + kOffHL);
    // ---- 1. scores of the owned cells: bulk copies through a ring of kStages tiles
    const int ntiles = (nloc + kTile - 1) / kTile;
    // one thread: three TMA copies per tile (the two 128-byte halves of the 128 code rows, 128B-
    // swizzled, and the 128 scale lines); cells past the pool read as zero and are not used
    auto issue = [&](int i) {
      if (i >= ntiles || tid != 0) return;
      uint8_t* base = sm + kOffRing + (i % kStages) * kTileBytes;
      uint64_t* bar = &bars[i % kStages];
      const int z = (int)(sq.cell0 + c_lo + i * kTile);
      mbar_arrive_expect_tx(bar, (uint32_t)kTileBytes);
      tma_load_3d(base, &tm_codes, bar, 0, g, z);
      tma_load_3d(base + kBoxB, &tm_codes, bar, 128, g, z);
      tma_load_2d(base + 2 * kBoxB, &tm_scales, bar, 0, z);
    };
    __syncthreads();  // barriers initialised before any copy completes on them
#pragma unroll
    for (int i = 0; i < kStages; ++i) issue(i);
    // Qsum (exact), its hi/lo split and the error terms while the first tiles land; thread = dim
    {
      __shared__ long long s_e2[16];
      if (tid < kD) {  // thread = dim
        __half hi, lo;
        long long e, habs, ex;
        qsum_split_exact(a.q, t, g, tid, hi, lo, e, habs, ex);
        s_qsum[tid] = ex;
        s_hl[tid] = hi;
        s_hl[256 + tid] = lo;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          e += __shfl_xor_sync(0xffffffffu, e, o);
          habs += __shfl_xor_sync(0xffffffffu, habs, o);
        }
        if (lane == 0) {
          s_e2[warp] = e;
          s_e2[8 + warp] = habs;
        }
      }
      __syncthreads();
      if (tid < 4) {
        constexpr float kUnit = 5.9604644775390625e-8f;  // 2^-24
        s_eh[tid] = __ll2float_ru(s_e2[2 * tid] + s_e2[2 * tid + 1]) * kUnit;
        s_eh[4 + tid] = __ll2float_ru(s_e2[8 + 2 * tid] + s_e2[8 + 2 * tid + 1]) * kUnit;
      }
    }
    // B fragments: column 0 = hi, column 1 = lo, columns 2-7 zero; k slots (2j, 2j+1, 2j+8, 2j+9)
    // of step ks carry dims 16 ks + 4j .. 4j+3 (the same order the A fragments use)
    uint32_t bq[16][2];
    {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(s_hl + (r8 == 1 ? 256 : 0));
#pragma unroll
      for (int ks = 0; ks < 16; ++ks) {
        bq[ks][0] = r8 < 2 ? src[(16 * ks + 4 * j) >> 1] : 0u;
        bq[ks][1] = r8 < 2 ? src[(16 * ks + 4 * j + 2) >> 1] : 0u;
      }
    }
    float kmx[4] = {0.f, 0.f, 0.f, 0.f};
    const float sms = p.sm_scale;
    for (int i = 0; i < ntiles; ++i) {
      ok_waits &= mbar_wait(&bars[i % kStages], (uint32_t)((i / kStages) & 1), a.status);
      const uint8_t* base = sm + kOffRing + (i % kStages) * kTileBytes;
      const int cell0 = i * kTile + 16 * warp;  // first local cell of this warp's 16
      if (cell0 < nloc) {
        float acc[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[b][u] = 0.f;
        // rows R = 16 warp + r8 (+8) of the tile; dims 16 ks + 4j .. +3 sit in box ks / 8, 16-byte
        // chunk (ks % 8) ^ (R % 8) of the row (the 128B swizzle), so the eight rows a step reads
        // fall in distinct banks
        const uint8_t* row0 = base + (16 * warp + r8) * 128 + 4 * j;
        const uint8_t* row1 = row0 + 8 * 128;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const int off = (ks >> 3) * kBoxB + (((ks & 7) ^ r8) << 4);
          uint32_t a0, a1, a2, a3;
          codes4_to_half(*reinterpret_cast<const uint32_t*>(row0 + off), a0, a2);
          codes4_to_half(*reinterpret_cast<const uint32_t*>(row1 + off), a1, a3);
          mma16816(acc[ks >> 2], a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
        }
        if (j == 0) {
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int lc = cell0 + r8 + 8 * hr;  // local cell
            if (lc < nloc) {
              const uint2 sw = *reinterpret_cast<const uint2*>(base + 2 * kBoxB + (16 * warp + r8 + 8 * hr) * 16 + 8 * g);
              const float s0 = __half2float(__ushort_as_half((unsigned short)(sw.x & 0xFFFFu)));
              const float s1 = __half2float(__ushort_as_half((unsigned short)(sw.x >> 16)));
              const float s2 = __half2float(__ushort_as_half((unsigned short)(sw.y & 0xFFFFu)));
              const float s3 = __half2float(__ushort_as_half((unsigned short)(sw.y >> 16)));
              kmx[0] = fmaxf(kmx[0], fabsf(s0));
              kmx[1] = fmaxf(kmx[1], fabsf(s1));
              kmx[2] = fmaxf(kmx[2], fabsf(s2));
              kmx[3] = fmaxf(kmx[3], fabsf(s3));
              float v = s0 * (acc[0][2 * hr] + acc[0][2 * hr + 1]);
              v = fmaf(s1, acc[1][2 * hr] + acc[1][2 * hr + 1], v);
              v = fmaf(s2, acc[2][2 * hr] + acc[2][2 * hr + 1], v);
              v = fmaf(s3, acc[3][2 * hr] + acc[3][2 * hr + 1], v);
              v *= sms;
              s_score[lc] = v;
              atomicAdd(&s_hist[f32_okey(v) >> 20], 1u);
            }
          }
        }
      }
      __syncthreads();  // the stage is free
      issue(i + kStages);
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float m = kmx[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) s_wred[warp][b] = m;
    }
    __syncthreads();
    cluster_wait();  // #0: every CTA has started and zeroed its receive buffers
    // ---- 2. histogram: add the own counts into the owners of the slices; kmax to everyone
    constexpr int kSlice = kHistBins / C;
    for (int i = tid; i < kHistBins; i += kFThreads) {
      const uint32_t v = s_hist[i];
      if (v) red_cluster_add_u32(mapa_shared(smem_u32(s_slice + (i % kSlice)), i / kSlice), v);
    }
    if (tid < 4 * C) {
      float m = 0.f;
#pragma unroll
      for (int w = 0; w < kFWarps; ++w) m = fmaxf(m, s_wred[w][tid & 3]);
      // kmax >= 0, so the float order is the int order
      asm volatile("red.shared::cluster.max.s32 [%0], %1;" ::"r"(mapa_shared(smem_u32(&s_kmax_all[tid & 3]), tid >> 2)),
                   "r"(__float_as_int(m))
                   : "memory");
    }
    cluster_arrive();
    cluster_wait();  // #1: every slice holds the cluster's counts
    // broadcast the owned slice to every CTA's full histogram
    for (int i = tid; i < kSlice * C; i += kFThreads) {
      const int qq = i / kSlice, b = i % kSlice;
      st_cluster_u32(mapa_shared(smem_u32(s_hist + r * kSlice + b), qq), s_slice[b]);
    }
    cluster_arrive();
    cluster_wait();  // #2: every CTA holds the cluster's histogram
    // the bin holding the K-th largest score: thread tid sums the kPerB bins from 4095 - kPerB tid down
    {
      constexpr int kPerB = kHistBins / kFThreads;
      static_assert(kPerB == 8, "two 16-byte reads per thread");
      const uint4* hp = reinterpret_cast<const uint4*>(s_hist + kHistBins - kPerB * (tid + 1));
      const uint4 h0 = hp[0], h1 = hp[1];
      const unsigned cnt = h0.x + h0.y + h0.z + h0.w + h1.x + h1.y + h1.z + h1.w;
      int tot;
      const int before = block_scan((int)cnt, s_red, &tot);  // counts in higher bins
      if (before < K && before + (int)cnt >= K) {
        int run = before, bin = kHistBins - kPerB * tid - 1;
        for (; bin >= kHistBins - kPerB * (tid + 1); --bin) {
          run += (int)s_hist[bin];
          if (run >= K) break;
        }
        s_bin = bin;
      }
      if (tid == 0 && tot < K) {  // cannot happen: the histogram holds n_kv >= K scores
        set_dev_status(a.status, QSA_DEV_BAND_OVERFLOW);
        s_bin = 0;
      }
    }
    __syncthreads();
    // ---- 3. classify the owned cells; exact keys of the candidates
    if (tid == 0) {
      // |s~ - s| <= a + b|s~|: a covers the Qsum residual after the hi + lo split (E_b), the
      // fp32 accumulation of 128 exact products per block (128 * 2^-23 relative to their
      // absolute sum, |kq| <= 128: the H_b * 2^-16 term) and the roundings of the scale
      // products (2^-21 of the absolute sum); b covers the final product by sm_scale.  Both are
      // doubled for margin.
      float acc = 0.f;
      for (int b = 0; b < kNB; ++b) acc += s_kmax_all[b] * (s_eh[b] + s_eh[kNB + b] * (1.5258789e-05f + 4.7683716e-07f));
      const float ea = 2.f * (p.sm_scale * 128.f * acc + 1.2e-7f), eb = 2.f * 9.5367432e-07f;
      const uint32_t klo = (uint32_t)s_bin << 20, khi = klo | 0xFFFFFu;
      float f_lo = okey_f32(klo), f_hi = okey_f32(khi);
      if (!(f_lo >= -3.0e38f)) f_lo = -3.0e38f;
      if (!(f_hi <= 3.0e38f)) f_hi = 3.0e38f;
      s_bnd[0] = ea;
      s_bnd[1] = eb;
      s_bnd[2] = f_hi + ea + eb * fabsf(f_hi);  // U(f_hi)
      s_bnd[3] = f_lo - ea - eb * fabsf(f_lo);  // L(f_lo)
      s_cnt_cand = 0;
    }
    __syncthreads();
    long long* c_hi_key = reinterpret_cast<long long*>(sm + kCandHi);
    unsigned long long* c_lo_key = reinterpret_cast<unsigned long long*>(sm + kCandLo);
    int* c_idx = reinterpret_cast<int*>(sm + kCandIdx);
    int n_in = 0;
    {
      const float ea = s_bnd[0], eb = s_bnd[1], Uhi = s_bnd[2], Llo = s_bnd[3];
      for (int base = 0; base < nloc; base += kFThreads) {
        const int i = base + tid;
        int st = 0;
        if (i < nloc) {
          const float f = s_score[i];
          const float Lf = f - ea - eb * fabsf(f), Uf = f + ea + eb * fabsf(f);
          st = Lf > Uhi ? 1 : (Uf < Llo ? 0 : 2);
          s_stat[i] = (uint8_t)st;
          n_in += st == 1;
          // the V rows of the cells that may be kept go to L2 now, for the attention phase
          if (st != 0 && !a.ids_only) prefetch_l2_256(vq + ((size_t)(c_lo + i) * kGroups + g) * kD);
        }
        const unsigned m = __ballot_sync(0xffffffffu, st == 2);
        int slot0 = 0;
        if (lane == 0 && m) slot0 = atomicAdd(&s_cnt_cand, __popc(m));
        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
        const int slot = slot0 + __popc(m & ((1u << lane) - 1u));
        if (st == 2 && slot < kOwnCap) c_idx[slot] = c_lo + i;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) n_in += __shfl_xor_sync(0xffffffffu, n_in, o);
      if (lane == 0) s_red[warp] = n_in;
      __syncthreads();
      n_in = 0;
#pragma unroll
      for (int w = 0; w < kFWarps; ++w) n_in += s_red[w];
    }
    // exact key of each candidate: a warp per candidate, lane = 8 dims; a warp loads the rows
    // of up to four candidates before it uses any
    const int nc = s_cnt_cand;               // may exceed kOwnCap (then the cluster flags and stops ranking)
    const int nc_st = min(nc, kOwnCap);      // candidates stored with their keys
    for (int c4 = 4 * warp; c4 < nc_st; c4 += 4 * kFWarps) {
      uint2 w[4], sw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c4 + u < nc_st ? c_idx[c4 + u] : c_lo;
        w[u] = __ldg(reinterpret_cast<const uint2*>(kq + ((size_t)c * kGroups + g) * kD + lane * 8));
        sw[u] = __ldg(reinterpret_cast<const uint2*>(ksc + ((size_t)c * kGroups + g) * kNB));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c4 + u >= nc_st) break;  // warp-uniform
        long long part = 0;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const int code = (int)(int8_t)((v < 4 ? w[u].x : w[u].y) >> (8 * (v & 3)));
          part += s_qsum[lane * 8 + v] * (long long)code;
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        part += __shfl_xor_sync(0xffffffffu, part, 4);  // block sum B_b on lanes 8b .. 8b+7
        const long long B0 = __shfl_sync(0xffffffffu, part, 0), B1 = __shfl_sync(0xffffffffu, part, 8);
        const long long B2 = __shfl_sync(0xffffffffu, part, 16), B3 = __shfl_sync(0xffffffffu, part, 24);
        if (lane == 0) {
          __int128 key = (__int128)half_int24((uint16_t)(sw[u].x & 0xFFFFu)) * B0;
          key += (__int128)half_int24((uint16_t)(sw[u].x >> 16)) * B1;
          key += (__int128)half_int24((uint16_t)(sw[u].y & 0xFFFFu)) * B2;
          key += (__int128)half_int24((uint16_t)(sw[u].y >> 16)) * B3;
          c_hi_key[c4 + u] = (long long)(key >> 64);
          c_lo_key[c4 + u] = (unsigned long long)key;
        }
      }
    }
    __syncthreads();
    // push the counts, and the candidates when they fit this CTA's slot, to every CTA
    constexpr int kSlot = kCandPush / (C < 8 ? 8 : C);  // a source's slot in every receiver
    long long* r_hi = reinterpret_cast<long long*>(sm + kRcvHi);
    unsigned long long* r_lo = reinterpret_cast<unsigned long long*>(sm + kRcvLo);
    int* r_idx = reinterpret_cast<int*>(sm + kRcvIdx);
    if (tid < C) {
      st_cluster_u32(mapa_shared(smem_u32(&s_ccnt[r][0]), tid), (uint32_t)n_in);
      st_cluster_u32(mapa_shared(smem_u32(&s_ccnt[r][1]), tid), (uint32_t)nc);
    }
    if (nc <= kSlot) {
      for (int i = tid; i < nc * C; i += kFThreads) {
        const int qq = i / nc, e = i % nc, slot = r * kSlot + e;
        st_cluster_u64(mapa_shared(smem_u32(r_hi + slot), qq), (unsigned long long)c_hi_key[e]);
        st_cluster_u64(mapa_shared(smem_u32(r_lo + slot), qq), c_lo_key[e]);
        st_cluster_u32(mapa_shared(smem_u32(r_idx + slot), qq), (uint32_t)c_idx[e]);
      }
    }
    cluster_arrive();
    cluster_wait();  // #3: counts and candidates delivered
    __shared__ int s_coff[17];  // exclusive prefix of the sources' candidate counts
    if (warp == 0) {  // lane q: source CTA q's counts; sums and prefix by shuffles
      const int in_q = lane < C ? s_ccnt[lane][0] : 0, nq = lane < C ? s_ccnt[lane][1] : 0;
      int in = in_q, pre = nq;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, pre, o);
        if (lane >= o) pre += y;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) in += __shfl_xor_sync(0xffffffffu, in, o);
      const bool over = __any_sync(0xffffffffu, nq > kSlot);
      // more candidates in one CTA than it keeps keys for (kOwnCap: only massive exact ties among
      // more than 65,536 cells do that): the ranking would be incomplete, so the token is flagged
      // and not ranked
      const bool beyond = __any_sync(0xffffffffu, nq > kOwnCap);
      if (lane < C) s_coff[lane] = pre - nq;
      if (lane == C - 1) s_coff[C] = pre;
      if (lane == 0) {
        int need = K - in;
        if (need < 0) {  // cannot happen: surely-in cells lie strictly above the k-th score
          set_dev_status(a.status, QSA_DEV_BAND_OVERFLOW);
          need = 0;
        }
        s_need = need;
        s_slow = beyond ? 2 : over;
        if (beyond && r == 0) set_dev_status(a.status, QSA_DEV_BAND_OVERFLOW);
      }
    }
    __syncthreads();
    const bool slow = s_slow == 1;  // uniform over the cluster: every CTA sees the same counts
    const int need = s_need;
    if (s_slow == 2) {
      // flagged above; the kept set is left at the surely-in cells
    } else if (!slow) {
      // the received candidates compacted into dense arrays (source-major) in one pass, then a
      // warp per own candidate with its lanes over consecutive entries.  The dense arrays use the
      // tails of the own-candidate arrays (here nc <= kSlot <= kDenseOff); a key is one 16-byte
      // word (lo, hi).
      static_assert(kCandPush / 8 <= kDenseOff, "own candidates (at most kSlot) stay below the dense arrays");
      static_assert((kDenseOff + kCandPush) * 16 <= kOwnCap * 8, "dense 16-byte keys fit the own hi-key array");
      static_assert(kDenseOff + kCandPush <= kOwnCap, "dense indices fit the own index array");
      ulonglong2* d_key = reinterpret_cast<ulonglong2*>(c_hi_key) + kDenseOff;  // bytes 16 kDenseOff ..
      int* d_idx = c_idx + kDenseOff;
      const int total = s_coff[C];
      for (int slot = tid; slot < C * kSlot; slot += kFThreads) {
        const int qq = slot / kSlot, e = slot - qq * kSlot;
        if (e < s_ccnt[qq][1]) {
          const int at = s_coff[qq] + e;
          d_key[at] = make_ulonglong2(r_lo[slot], (unsigned long long)r_hi[slot]);
          d_idx[at] = r_idx[slot];
        }
      }
      __syncthreads();
      for (int i = warp; i < nc; i += kFWarps) {
        const long long mh = c_hi_key[i];
        const unsigned long long ml = c_lo_key[i];
        const int mi = c_idx[i];
        int rank = 0;
#pragma unroll 4
        for (int e = lane; e < total; e += 32) {
          const ulonglong2 kk = d_key[e];
          rank += ranks_ahead((long long)kk.y, kk.x, d_idx[e], mh, ml, mi);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (lane == 0 && rank < need) s_stat[mi - c_lo] = 1;
      }
    } else {
      for (int base = 0; base < nc; base += kFThreads) {  // own candidates, one per thread per round
        const int i = base + tid;
        const bool mine = i < nc;
        const long long mh = mine ? c_hi_key[i] : 0;
        const unsigned long long ml = mine ? c_lo_key[i] : 0ull;
        const int mi = mine ? c_idx[i] : 0;
        int rank = 0;
        {
          // some CTA had more candidates than its slot: read them from its shared memory
          long long* st_hi = reinterpret_cast<long long*>(sm + kStgHi);
          unsigned long long* st_lo = reinterpret_cast<unsigned long long*>(sm + kStgLo);
          int* st_idx = reinterpret_cast<int*>(sm + kStgIdx);
          for (int qq = 0; qq < C; ++qq) {
            const int nq = s_ccnt[qq][1];
            for (int s0 = 0; s0 < nq; s0 += kCandStage) {
              const int len = min(kCandStage, nq - s0);
              __syncthreads();  // the stage is free
              for (int e = tid; e < len; e += kFThreads) {
                st_hi[e] = (long long)ld_cluster_u64(mapa_shared(smem_u32(c_hi_key + s0 + e), qq));
                st_lo[e] = ld_cluster_u64(mapa_shared(smem_u32(c_lo_key + s0 + e), qq));
                st_idx[e] = (int)ld_cluster_u32(mapa_shared(smem_u32(c_idx + s0 + e), qq));
              }
              __syncthreads();
              if (mine)
                for (int e = 0; e < len; ++e) rank += ranks_ahead(st_hi[e], st_lo[e], st_idx[e], mh, ml, mi);
            }
          }
        }
        if (mine && rank < need) s_stat[mi - c_lo] = 1;
      }
    }
    if (slow) {  // the candidate arrays stay readable until every CTA has ranked
      cluster_arrive();
      cluster_wait();
    }
    __syncthreads();
    // ---- ascending list of the kept owned cells
    {
      constexpr int kPerT = kMaxW / kFThreads;  // 16 consecutive cells per thread
      static_assert(kPerT == 16, "one 16-byte status read per thread");
      const int i0 = tid * kPerT;
      uint32_t keep = 0;  // bit u: cell i0 + u is kept
      if (i0 < nloc) {
        const uint4 w = *reinterpret_cast<const uint4*>(s_stat + i0);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < kPerT; ++u)
          if (i0 + u < nloc && ((ww[u >> 2] >> (8 * (u & 3))) & 0xFFu) == 1u) keep |= 1u << u;
      }
      int total;
      int off = block_scan(__popc(keep), s_red, &total);
      while (keep) {
        const int u = __ffs(keep) - 1;
        keep &= keep - 1;
        s_list[off++] = (uint16_t)(i0 + u);
      }
      if (tid == 0) s_nlist = total;
      __syncthreads();
      n_sel = s_nlist;
    }
    if (a.ids_only) {  // uniform: the kept counts to every CTA, then the ids; no attention
      if (tid < C) st_cluster_u32(mapa_shared(smem_u32(&s_nsel_all[r]), tid), (uint32_t)n_sel);
      cluster_arrive();
      cluster_wait();  // #4 of this form: every CTA's kept count delivered
      write_ids(n_sel);
      drain();
      return;
    }
  } else {
    // identity: the V rows to L2 while the first batch is set up
    for (int i = tid; i < nloc; i += kFThreads) prefetch_l2_256(vq + ((size_t)(c_lo + i) * kGroups + g) * kD);
  }

  // ---- 4. attention over the kept owned cells, batches of 64 (bulk copies, two stages)
  float o_acc[2][4];  // O rows r8, r8 + 8 x this warp's 16 dims
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int u = 0; u < 4; ++u) o_acc[nt][u] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // heads r8 and r8 + 8 (log2 units)
  {
    const int nb = (n_sel + kBatch - 1) / kBatch;
    __half* s_vh = reinterpret_cast<__half*>(sm + kOffVh);
    __half* s_p = reinterpret_cast<__half*>(sm + kOffP);
    auto cell_of = [&](int i) -> int { return c_lo + (selected ? (int)s_list[i] : i); };
    // cp.async of the batch's K and V rows (16 bytes a piece, 16 pieces a row) and scale lines
    auto issue = [&](int bi) {
      if (bi < nb) {
        uint8_t* base = sm + kOffRing + (bi & 1) * kBatchBytes;
        const int i0 = bi * kBatch, cnt = min(kBatch, n_sel - i0);
        for (int pce = tid; pce < kBatch * 32; pce += kFThreads) {
          const int cell = pce >> 5, piece = pce & 31;
          if (cell < cnt) {
            const int c = cell_of(i0 + cell);
            const int8_t* src = (piece < 16 ? kq : vq) + ((size_t)c * kGroups + g) * kD + (piece & 15) * 16;
            cp_async16(base + (piece < 16 ? 0 : kBatch * kRowB) + cell * kRowB + (piece & 15) * 16, src);
          }
        }
        if (tid < 2 * kBatch) {
          const int cell = tid & (kBatch - 1);
          if (cell < cnt) {
            const int c = cell_of(i0 + cell);
            cp_async16(base + 2 * kBatch * kRowB + (tid < kBatch ? 0 : kBatch * 16) + cell * 16,
                       (tid < kBatch ? ksc : vsc) + (size_t)c * kGroups * kNB);
          }
        }
      }
      cp_async_commit();
    };
    __syncthreads();  // the ring region is free (scoring and candidates are done) and the list is set
    issue(0);
    issue(1);
    const float sl2 = p.sm_scale * kLog2e;
    for (int bi = 0; bi < nb; ++bi) {
      cp_async_wait<1>();
      __syncthreads();
      const uint8_t* base = sm + kOffRing + (bi & 1) * kBatchBytes;
      const int cnt = min(kBatch, n_sel - bi * kBatch);
      // V^ = fp16(vq * vsc) for the batch (rows past cnt are zero)
      for (int e = tid; e < kBatch * 32; e += kFThreads) {
        const int cell = e >> 5, c8 = e & 31;
        uint4 outw = make_uint4(0, 0, 0, 0);
        if (cell < cnt) {
          const uint2 w = *reinterpret_cast<const uint2*>(base + kBatch * kRowB + cell * kRowB + c8 * 8);
          const __half s =
              *reinterpret_cast<const __half*>(base + 2 * kBatch * kRowB + kBatch * 16 + cell * 16 + 8 * g + (c8 >> 3) * 2);
          uint32_t o4[4];
          dequant8(w.x, w.y, __half2half2(s), o4);
          outw = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        *reinterpret_cast<uint4*>(s_vh + cell * kVhStride + c8 * 8) = outw;
      }
      // logits of this warp's 8 cells for the 12 heads (rows 12-15 of A are zero); warps
      // kQKWarps and above have no cells and only take part in V^ and P.V
      float sc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // (r8, 2j), (r8, 2j+1), (r8+8, 2j), (r8+8, 2j+1)
      const bool row1 = r8 + 8 < 12;
      const bool qk = warp < kQKWarps;
      if (qk) {
        float acc[4][4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[b][u] = 0.f;
        const uint8_t* krow = base + (8 * warp + r8) * kRowB + 4 * j;  // B: cell 8 warp + r8
        const __half* q0 = s_q + r8 * kQStride + 4 * j;
        const __half* q1 = s_q + (r8 + 8) * kQStride + 4 * j;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const uint2 x0 = *reinterpret_cast<const uint2*>(q0 + 16 * ks);
          const uint2 x1 = row1 ? *reinterpret_cast<const uint2*>(q1 + 16 * ks) : make_uint2(0u, 0u);
          uint32_t b0, b1;
          codes4_to_half(*reinterpret_cast<const uint32_t*>(krow + 16 * ks), b0, b1);
          mma16816(acc[ks >> 2], x0.x, x1.x, x0.y, x1.y, b0, b1);
        }
        const int cA = 8 * warp + 2 * j;  // this thread's two cells
        const uint8_t* scb = base + 2 * kBatch * kRowB + 8 * g;
        float ks0[4], ks1[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          ks0[b] = __half2float(*reinterpret_cast<const __half*>(scb + cA * 16 + 2 * b));
          ks1[b] = __half2float(*reinterpret_cast<const __half*>(scb + (cA + 1) * 16 + 2 * b));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float* kk = (u & 1) ? ks1 : ks0;
          float v = kk[0] * acc[0][u];
          v = fmaf(kk[1], acc[1][u], v);
          v = fmaf(kk[2], acc[2][u], v);
          v = fmaf(kk[3], acc[3][u], v);
          const bool valid = (cA + (u & 1)) < cnt && (u < 2 || row1);
          sc[u] = valid ? v * sl2 : -INFINITY;
        }
      }
      // batch maxima per head row: 4 lanes per row, then across the 8 warps
      float mx0 = fmaxf(sc[0], sc[1]), mx1 = fmaxf(sc[2], sc[3]);
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      if (j == 0 && qk) {
        s_wred[warp][r8] = mx0;
        s_wred[warp][r8 + 8] = mx1;
      }
      __syncthreads();
      float Mn[2], alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float m = m_run[hr];
#pragma unroll
        for (int w = 0; w < kQKWarps; ++w) m = fmaxf(m, s_wred[w][r8 + 8 * hr]);
        Mn[hr] = m;
        alpha[hr] = (m == -INFINITY) ? 1.f : fast_exp2(m_run[hr] - m);
      }
      // P = 2^(s - M) (fp16 into shared memory, rows 12-15 zero) and its row sums
      float pr[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) pr[u] = (sc[u] == -INFINITY) ? 0.f : fast_exp2(sc[u] - Mn[u >> 1]);
      if (qk) {
        const int cA = 8 * warp + 2 * j;
        *reinterpret_cast<uint32_t*>(s_p + r8 * kPStride + cA) = pack_half2(pr[0], pr[1]);
        *reinterpret_cast<uint32_t*>(s_p + (r8 + 8) * kPStride + cA) = pack_half2(pr[2], pr[3]);
      }
      float rs0 = pr[0] + pr[1], rs1 = pr[2] + pr[3];
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        rs0 += __shfl_xor_sync(0xffffffffu, rs0, o);
        rs1 += __shfl_xor_sync(0xffffffffu, rs1, o);
      }
      __syncthreads();  // maxima read by all; P and V^ complete; this batch's stage is free
      if (j == 0 && qk) {
        s_wred[warp][r8] = rs0;
        s_wred[warp][r8 + 8] = rs1;
      }
      issue(bi + 2);
      __syncthreads();
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float rs = 0.f;
#pragma unroll
        for (int w = 0; w < kQKWarps; ++w) rs += s_wred[w][r8 + 8 * hr];
        l_run[hr] = l_run[hr] * alpha[hr] + rs;
        m_run[hr] = Mn[hr];
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        o_acc[nt][0] *= alpha[0];
        o_acc[nt][1] *= alpha[0];
        o_acc[nt][2] *= alpha[1];
        o_acc[nt][3] *= alpha[1];
      }
      // O[16 heads][16 dims of this warp] += P[16][64] x V^[64][16]
#pragma unroll
      for (int kk = 0; kk < kBatch / 16; ++kk) {
        uint32_t pa0, pa1, pa2, pa3;
        {
          const int row = (lane & 7) + ((lane >> 3) & 1) * 8, col = 16 * kk + (lane >> 4) * 8;
          ldsm_x4(smem_u32(s_p + row * kPStride + col), pa0, pa1, pa2, pa3);
        }
        uint32_t v0, v1, v2, v3;
        const int krow = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int ncol = kDimsPerWarp * warp + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(s_vh + krow * kVhStride + ncol), v0, v1, v2, v3);
        mma16816(o_acc[0], pa0, pa1, pa2, pa3, v0, v1);
        mma16816(o_acc[1], pa0, pa1, pa2, pa3, v2, v3);
      }
    }
    cp_async_wait<0>();
  }
  // ---- 5. push (m, l), the kept count and each owner's share of the partial outputs
  constexpr int kPerCta = 12 * 256 / C;
  float* r_o = s_score;                    // [C][kPerCta] received from CTA q
  float* r_m = s_score + 12 * 256;         // [C][12]
  float* r_l = r_m + 16 * 12;              // [C][12]
  if (!selected) cluster_wait();           // #0 (the selected path waited before its first push)
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int d = kDimsPerWarp * warp + 8 * nt + 2 * j;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int h = r8 + 8 * hr;
      if (h < 12) {
        const int idx = h * 256 + d, owner = idx / kPerCta;  // d and d+1 share an owner (kPerCta is even)
        st_cluster_f32x2(mapa_shared(smem_u32(r_o + r * kPerCta + (idx - owner * kPerCta)), owner),
                         o_acc[nt][2 * hr], o_acc[nt][2 * hr + 1]);
      }
    }
  }
  if (warp == 0 && j == 0) {  // m, l of heads r8 and r8 + 8 to every CTA
    for (int qq = 0; qq < C; ++qq) {
      st_cluster_u32(mapa_shared(smem_u32(r_m + r * 12 + r8), qq), __float_as_uint(m_run[0]));
      st_cluster_u32(mapa_shared(smem_u32(r_l + r * 12 + r8), qq), __float_as_uint(l_run[0]));
      if (r8 + 8 < 12) {
        st_cluster_u32(mapa_shared(smem_u32(r_m + r * 12 + r8 + 8), qq), __float_as_uint(m_run[1]));
        st_cluster_u32(mapa_shared(smem_u32(r_l + r * 12 + r8 + 8), qq), __float_as_uint(l_run[1]));
      }
    }
  }
  if (tid < C) st_cluster_u32(mapa_shared(smem_u32(&s_nsel_all[r]), tid), (uint32_t)n_sel);
  cluster_arrive();
  cluster_wait();  // #4: partials delivered; no CTA touches another after this
  for (int e = tid; e < kPerCta; e += kFThreads) {
    const int idx = r * kPerCta + e, h = idx >> 8, d = idx & 255;
    float M = -INFINITY;
#pragma unroll
    for (int qq = 0; qq < C; ++qq) M = fmaxf(M, r_m[qq * 12 + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int qq = 0; qq < C; ++qq) {
      const float mq = r_m[qq * 12 + h];
      if (mq == -INFINITY) continue;
      const float w = fast_exp2(mq - M);
      L = fmaf(r_l[qq * 12 + h], w, L);
      O = fmaf(r_o[qq * kPerCta + e], w, O);
    }
    float v = O / L;
    if (a.gate) v *= gate_sigmoid(__half2float(a.gate[((size_t)t * kHeads + g * kHPG + h) * kD + d]));
    const size_t o = ((size_t)t * kHeads + g * kHPG + h) * kD + d;
    if (a.out16) a.out16[o] = __float2half_rn(v);
    else a.xp[o] = v;
  }
  if (selected) write_ids(n_sel);
  drain();
}

cudaLaunchConfig_t launch_config(int C, int n_tok, cudaStream_t stream, cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, kGroups, n_tok);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// Per device: 0 = not set up, 1 = attributes set and clusters of 16 fit, 2 = set, only 8 fit;
// and how many clusters of 2, 4, 8 and 16 CTAs the GPU holds at once, read at set-up (a cluster
// lives inside one GPC, so large clusters fit fewer times than the SM count suggests).
std::atomic<int> g_setup[64];
std::atomic<int> g_maxc[64][4];
constexpr int kClusterSizes[4] = {2, 4, 8, 16};
int g_dev_of_setup() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev >= 0 && dev < 64 ? dev : 0;
}

template <int C>
cudaError_t set_attrs() {
  auto kern = decode_fused_kernel<C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && C > 8) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t device_setup(int* state) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int s = g_setup[dev].load(std::memory_order_acquire);
  if (s == 0) {
    if ((e = set_attrs<2>()) != cudaSuccess) return e;
    if ((e = set_attrs<4>()) != cudaSuccess) return e;
    if ((e = set_attrs<8>()) != cudaSuccess) return e;
    if ((e = set_attrs<16>()) != cudaSuccess) return e;
    int nmax[4] = {0, 0, 0, 0};
    for (int i = 0; i < 4; ++i) {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = launch_config(kClusterSizes[i], 1, nullptr, attr);
      e = i == 0   ? cudaOccupancyMaxActiveClusters(&nmax[i], decode_fused_kernel<2>, &cfg)
          : i == 1 ? cudaOccupancyMaxActiveClusters(&nmax[i], decode_fused_kernel<4>, &cfg)
          : i == 2 ? cudaOccupancyMaxActiveClusters(&nmax[i], decode_fused_kernel<8>, &cfg)
                   : cudaOccupancyMaxActiveClusters(&nmax[i], decode_fused_kernel<16>, &cfg);
      if (e != cudaSuccess) return e;
    }
    if (nmax[2] <= 0) return cudaErrorInvalidConfiguration;  // clusters of 8 are portable
    s = nmax[3] > 0 ? 1 : 2;
    for (int i = 0; i < 4; ++i) g_maxc[dev][i].store(nmax[i], std::memory_order_release);
    g_setup[dev].store(s, std::memory_order_release);
  }
  *state = s;
  return cudaSuccess;
}

template <int C>
cudaError_t launch_c(const FusedArgs& a, int n_tok, const CUtensorMap& tmc, const CUtensorMap& tms,
                     cudaStream_t stream) {
  auto kern = decode_fused_kernel<C>;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(C, n_tok, stream, attr);
  return cudaLaunchKernelEx(&cfg, kern, a, tmc, tms);
}

// Tensor maps over the pool: codes as [n_pool][2][256] bytes (128-byte boxes of 128 cells of one
// group, 128B-swizzled) and K scales as [n_pool][8] fp16 lines (both groups; 128-line boxes).
bool encode_maps(const int8_t* kq, const __half* ksc, long long n_pool, CUtensorMap* tmc, CUtensorMap* tms) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t cd[3] = {256, 2, (cuuint64_t)n_pool};
  const cuuint64_t cs[2] = {256, 512};
  const cuuint32_t cb[3] = {128, 1, kTile};
  const cuuint32_t ce[3] = {1, 1, 1};
  if (enc(tmc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<int8_t*>(kq), cd, cs, cb, ce, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return false;
  const cuuint64_t sd[2] = {8, (cuuint64_t)n_pool};
  const cuuint64_t ss[1] = {16};
  const cuuint32_t sb[2] = {8, kTile};
  const cuuint32_t se[2] = {1, 1};
  return enc(tms, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<__half*>(ksc), sd, ss, sb, se,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

int decode_layer_cells_per_cta() { return kMaxW; }

cudaError_t decode_layer_max_cluster(int* c) {
  int state = 0;
  cudaError_t e = device_setup(&state);
  if (e != cudaSuccess) return e;
  *c = state == 1 ? 16 : 8;
  return cudaSuccess;
}

cudaError_t launch_decode_layer(const __half* q, const int8_t* kq, const int8_t* vq, const __half* ksc,
                                const __half* vsc, const int4* seqs, int n_seq, long long n_pool, int n_cells, int pos0,
                                int n_tok, int max_n_kv, int32_t* ids, const __half* gate, float* xp, Params p,
                                int* status, cudaStream_t stream, __half* out16, bool selected_only,
                                bool ids_only) {
  FusedArgs a{q, kq, vq, ksc, vsc, seqs, n_seq, n_pool, n_cells, pos0, ids, gate, xp, p, status, out16,
              selected_only ? 1 : 0, ids_only ? 1 : 0};
  int state = 0;
  cudaError_t e = device_setup(&state);
  if (e != cudaSuccess) return e;
  // 16 CTAs per (token, group) for a few tokens (more SMs per token) or when a token's cells
  // need them; otherwise 8, which keeps twice as many clusters resident.
  CUtensorMap tmc, tms;
  if (!encode_maps(kq, ksc, n_pool, &tmc, &tms)) return cudaErrorInvalidValue;
  // The cluster size: the kernel's phases are latency bound, so a launch takes about (waves of
  // clusters) x (a fixed part + a part growing with the cells per CTA); measured on GB300 the two
  // parts match at about 2,048 cells.  Few tokens: more CTAs per token (one wave either way); many
  // tokens: fewer, larger CTAs (fewer waves).  A wave is as many clusters of that size as the GPU
  // holds at once.  C must hold max_n_kv in C x kMaxW cells.
  const int dev = g_dev_of_setup();
  const long long clusters = (long long)kGroups * n_tok;
  int best_c = 0;
  double best_t = 0.0;
  for (int i = 3; i >= 0; --i) {
    const int c = kClusterSizes[i];
    const int maxc = g_maxc[dev][i].load(std::memory_order_acquire);
    if (maxc <= 0 || (long long)max_n_kv > (long long)c * kMaxW) continue;
    const double waves = (double)((clusters + maxc - 1) / maxc);
    const double cells = (double)max_n_kv / c;
    const double t = waves * (1.0 + cells / 2048.0);
    if (best_c == 0 || t < best_t) {
      best_c = c;
      best_t = t;
    }
  }
  switch (best_c) {
    case 16: return launch_c<16>(a, n_tok, tmc, tms, stream);
    case 4: return launch_c<4>(a, n_tok, tmc, tms, stream);
    case 2: return launch_c<2>(a, n_tok, tmc, tms, stream);
    default: return launch_c<8>(a, n_tok, tmc, tms, stream);
  }
}

}  // namespace qsa
