// Shared constants, the int8 -> fp16 dequantisation step and the internal launcher
// interface between the C ABI (api.cu) and the kernel translation units.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <utility>

#include "ptx.cuh"

namespace qsa {

// Launch with programmatic stream serialization (see pdl_begin): the kernel may start while the
// previous kernel on `stream` finishes, and waits for it inside pdl_begin().
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kGroups = 2;         // KV heads
constexpr int kHPG = 12;           // query heads per KV head
constexpr int kHeads = 24;
constexpr int kD = 256;            // head dim
constexpr int kBlk = 64;           // elements per fp16 scale
constexpr int kNB = kD / kBlk;     // scales per row
constexpr int kChunk = 64;         // decode split size
constexpr int kPartStride = 258;   // o[256], m, l
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  int topk;
  int identity_max;
  float sm_scale;
};

// First token of a call whose cell count n_kv = pos0 + t + 1 exceeds identity_max.
__host__ __device__ inline int first_selected_token(int pos0, int identity_max) {
  const long long t = (long long)identity_max - pos0;
  return t < 0 ? 0 : (int)t;
}

// 8 int8 codes (two 32-bit words) times one fp16 scale -> 8 fp16 values, packed as four
// half2 words with the lower-indexed element in the low half.  The bytes are biased to
// unsigned, placed under an fp16 exponent of 2^10 (1024 + u is exact), the bias 1152 is
// subtracted (exact integer result) and one multiply rounds code * scale to nearest.
__device__ __forceinline__ void dequant8(uint32_t w0, uint32_t w1, __half2 s2, uint32_t (&o)[4]) {
  const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152.0
  const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
  uint32_t h[4];
  h[0] = __byte_perm(u0, 0x64646464u, 0x4140);
  h[1] = __byte_perm(u0, 0x64646464u, 0x4342);
  h[2] = __byte_perm(u1, 0x64646464u, 0x4140);
  h[3] = __byte_perm(u1, 0x64646464u, 0x4342);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = __hsub2(*reinterpret_cast<__half2*>(&h[i]), bias);
    v = __hmul2(v, s2);
    o[i] = *reinterpret_cast<uint32_t*>(&v);
  }
}

// ---------------------------------------------------------------- launchers
// All launchers enqueue on `stream`, return a cudaError_t from the launch, and assume the
// host has validated every argument.  `status` is the device status word.

struct FlashArgs {
  const __half* q;
  const int8_t* kq;
  const int8_t* vq;
  const __half* ksc;
  const __half* vsc;
  const int32_t* ids;
  const __half* gate;  // output gate [T][24][256], or null
  __half* out;
  int n_cells, T, pos0;
  Params p;
  int* status;
};

// fp16 mirror of the cache cells 0 .. n-1 (K^ and V^), written once per prefill call.
size_t prefill_workspace_bytes(int T, int pos0);
cudaError_t launch_dequant_mirror(const int8_t* kq, const int8_t* vq, const __half* ksc, const __half* vsc, int n,
                                  __half* khat, __half* vhat, cudaStream_t stream);
cudaError_t launch_flash_dense(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                               cudaStream_t stream);
cudaError_t launch_flash_gather(const FlashArgs& a, int t_begin, int t_end, const __half* khat, const __half* vhat,
                                cudaStream_t stream);

// Batched prefill (many sequences, the seqs table of the batched decode): a work list of the
// identity tokens' tiles and one fp16 mirror of rows_per_seq rows per sequence, built on the
// device (mirror.cu), then the dense kernel over that list.  Workspace: the list (plan_bytes),
// then K^ and V^ of mirror_rows rows each.
struct BatchedPrefillLayout {
  int rows_per_seq, max_pairs;
  long long mirror_rows;
  size_t plan_bytes, bytes;
};
BatchedPrefillLayout batched_prefill_layout(int n_seq, int n_tok, int max_n_kv, int identity_max);
cudaError_t launch_batched_prefill_prep(const int8_t* kq, const int8_t* vq, const __half* ksc, const __half* vsc,
                                        const int4* seqs, int n_seq, int n_tok, long long n_pool, int max_n_kv,
                                        int identity_max, const BatchedPrefillLayout& L, void* ws, int* status,
                                        cudaStream_t stream);
cudaError_t launch_flash_dense_batched(const __half* q, int n_tok, const __half* gate, __half* out, const int4* plan,
                                       int max_pairs, const __half* khat, const __half* vhat, int mirror_rows,
                                       float sm_scale, int* status, cudaStream_t stream);

cudaError_t launch_decode_partial(const __half* q, const int8_t* kq, const int8_t* vq, const __half* ksc,
                                  const __half* vsc, const int32_t* ids, float* part, int32_t* n_chunks,
                                  int chunk_cap, int n_cells, int N, int pos0, Params p, int* status,
                                  cudaStream_t stream);

// Fused decode layer (decode_fused.cu): selection, attention and merge in one launch, one
// cluster per (token, group).  seqs (device, may be null) lists {first pool cell, n_cells, pos0,
// first token} per sequence; with null the call is one sequence of n_cells cells at pos0.
int decode_layer_cells_per_cta();
cudaError_t decode_layer_max_cluster(int* c);
cudaError_t launch_decode_layer(const __half* q, const int8_t* kq, const int8_t* vq, const __half* ksc,
                                const __half* vsc, const int4* seqs, int n_seq, long long n_pool, int n_cells, int pos0,
                                int n_tok, int max_n_kv, int32_t* ids, const __half* gate, float* xp, Params p,
                                int* status, cudaStream_t stream, __half* out16 = nullptr, bool selected_only = false,
                                bool ids_only = false);

// Output gate: the elementwise logistic function of the gate input, in fp32, 1 / (1 + e^-x).  The
// exponential takes the special-function unit; the reciprocal of d = 1 + e^-x (d >= 1, and finite
// for |x| <= 80, past which the result is 0 or 1 in every output format) is formed on the FMA
// pipe, which the epilogues leave idle, so that the gate costs one special-function operation per
// element instead of two: an estimate whose float bits are 0x7EF00000 - bits(d) (the exponent
// negated and the mantissa mirrored; within 6.25% of 1/d), then three Newton-Raphson steps
// r <- r (2 - d r), each of which squares the relative error (below 1e-9 before the last
// rounding; sigmoid(0) is exactly 1/2).
__device__ __forceinline__ float gate_sigmoid(float x) {
  const float d = 1.f + __expf(-fminf(fmaxf(x, -80.f), 80.f));
  float r = __int_as_float(0x7EF00000 - __float_as_int(d));
  r = r * fmaf(-d, r, 2.f);
  r = r * fmaf(-d, r, 2.f);
  r = r * fmaf(-d, r, 2.f);
  return r;
}

cudaError_t launch_merge(const float* part, const int32_t* n_chunks, int N, int chunk_cap, const __half* gate,
                         float* xp, int* status, cudaStream_t stream);

cudaError_t launch_quantize(const __half* x, int64_t n_rows, int8_t* xq, __half* xsc, cudaStream_t stream);

// Fused prep (prep.cu): RMS norm + rotary embedding of q and k, qcur / kcur, and the int8 cache
// rows of cells pos0 .. pos0 + T - 1.
cudaError_t launch_prep(const __half* q_raw, const __half* k_raw, const __half* v_raw, const float* q_gamma,
                        const float* k_gamma, const int32_t* pos3, int T, int pos0, double base, int rotary_dim,
                        float eps, const int* sections, __half* qcur, __half* kcur, int8_t* kq, __half* ksc,
                        int8_t* vq, __half* vsc, cudaStream_t stream);

// The score-GEMM and top-k selection holds caches of up to select_max_cells() cells; longer
// caches are selected by the single-launch decode layer's cluster kernel (ids only).
int select_max_cells();
size_t select_workspace_bytes(int T, int pos0, int n_cells, Params p);
cudaError_t launch_select(const __half* q, const int8_t* kq, const __half* ksc, int n_cells, int T, int pos0,
                          int32_t* ids, void* ws, Params p, int* status, cudaStream_t stream);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

}  // namespace qsa
