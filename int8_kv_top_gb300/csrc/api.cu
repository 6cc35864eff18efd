// C ABI of the QSA layer: argument validation, the device status word, the per-thread
// last-error string, and dispatch to the kernel launchers.  Declarations and the
// contract of every entry point are in include/qsa.h.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/qsa.h"
#include "common.cuh"

namespace qsa {

// One status word per device; kernels receive its address.
__device__ int g_status_word = 0;

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace qsa

namespace {

thread_local char t_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  t_last_error[0] = '\0';
  return QSA_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(QSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Address of this device's status word (looked up once per device).
int* status_ptr(int* err) {
  static int* cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = cuda_fail(e == cudaSuccess ? cudaErrorInvalidDevice : e, "cudaGetDevice");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, qsa::g_status_word);
    if (e != cudaSuccess) {
      *err = cuda_fail(e, "cudaGetSymbolAddress(status word)");
      return nullptr;
    }
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int resolve_params(const qsa_params* in, qsa::Params* out) {
  qsa::Params p{2048, 2051, 0.0625f};
  if (in) {
    p.topk = in->topk;
    p.identity_max = in->identity_max;
    p.sm_scale = in->sm_scale;
  }
  if (p.identity_max < 1) return fail(QSA_ERR_INVALID_ARG, "identity_max must be >= 1 (got %d)", p.identity_max);
  if (p.topk < 1 || p.topk > p.identity_max + 1)
    return fail(QSA_ERR_INVALID_ARG, "topk must be in [1, identity_max + 1] (got %d)", p.topk);
  if (!(p.sm_scale > 0.f) || !(p.sm_scale < 3.0e38f))
    return fail(QSA_ERR_INVALID_ARG, "sm_scale must be positive and finite");
  *out = p;
  return QSA_OK;
}

#define CHECK_PTR(p, name)                                                                      \
  do {                                                                                          \
    if (!(p)) return fail(QSA_ERR_INVALID_ARG, "%s is NULL", name);                             \
    if (!aligned16(p)) return fail(QSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);      \
  } while (0)

int check_layer(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T, int pos0) {
  CHECK_PTR(q, "q");
  CHECK_PTR(kq, "kq");
  CHECK_PTR(ksc, "ksc");
  if (T <= 0) return fail(QSA_ERR_INVALID_ARG, "T must be positive (got %d)", T);
  if (pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "pos0 must be >= 0 (got %d)", pos0);
  if ((long long)pos0 + T > (long long)n_cells)
    return fail(QSA_ERR_INVALID_ARG, "cache too small: pos0 + T = %lld > n_cells = %d", (long long)pos0 + T, n_cells);
  return QSA_OK;
}

// Largest n_kv the fused decode takes on this device (cells per CTA x the largest cluster).
int decode_layer_limit(int* rc) {
  int c = 0;
  cudaError_t e = qsa::decode_layer_max_cluster(&c);
  if (e != cudaSuccess) {
    *rc = cuda_fail(e, "qsa_decode_layer set-up");
    return 0;
  }
  return c * qsa::decode_layer_cells_per_cta();
}

// Selection over a cache longer than the score-GEMM path holds: the single-launch decode layer's
// cluster kernel, ids only (its exact ranking; no attention, V not read, no workspace).
int select_long(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T, int pos0, int32_t* ids,
                const qsa::Params& p, void* stream, const char* who) {
  int rc = 0;
  const int limit = decode_layer_limit(&rc);
  if (!limit) return rc;
  if ((long long)pos0 + T > limit)
    return fail(QSA_ERR_UNSUPPORTED, "%s: selection over n_kv up to %lld cells is not supported (at most %d)", who,
                (long long)pos0 + T, limit);
  if (T > 65535) return fail(QSA_ERR_UNSUPPORTED, "%s: at most 65535 tokens over %d cells", who, qsa::select_max_cells());
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaError_t e = qsa::launch_decode_layer(reinterpret_cast<const __half*>(q), kq, nullptr,
                                           reinterpret_cast<const __half*>(ksc), nullptr, nullptr, 1, (long long)n_cells,
                                           n_cells, pos0, T, pos0 + T, ids, nullptr, nullptr, p, st,
                                           static_cast<cudaStream_t>(stream), nullptr, false, true);
  if (e != cudaSuccess) return cuda_fail(e, who);
  return ok();
}

}  // namespace

extern "C" {

const char* qsa_last_error(void) { return t_last_error; }

int qsa_prep_quantize(const uint16_t* x, int64_t n_rows, int8_t* xq, uint16_t* xsc, void* stream) {
  if (n_rows < 0) return fail(QSA_ERR_INVALID_ARG, "n_rows must be >= 0");
  if (n_rows == 0) return ok();
  CHECK_PTR(x, "x");
  CHECK_PTR(xq, "xq");
  CHECK_PTR(xsc, "xsc");
  cudaError_t e = qsa::launch_quantize(reinterpret_cast<const __half*>(x), n_rows, xq, reinterpret_cast<__half*>(xsc),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_prep_quantize launch");
  return ok();
}

int qsa_prep(const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v_raw, const float* q_gamma,
             const float* k_gamma, const int32_t* pos3, const qsa_rope* rope, int T, int pos0, int n_cells,
             uint16_t* qcur, uint16_t* kcur, int8_t* kq, uint16_t* ksc, int8_t* vq, uint16_t* vsc, void* stream) {
  qsa_rope r{10000.f, 256, 1e-6f, {32, 48, 48}};
  if (rope) r = *rope;
  CHECK_PTR(q_raw, "q_raw");
  CHECK_PTR(k_raw, "k_raw");
  CHECK_PTR(v_raw, "v_raw");
  CHECK_PTR(q_gamma, "q_gamma");
  CHECK_PTR(k_gamma, "k_gamma");
  CHECK_PTR(qcur, "qcur");
  CHECK_PTR(kq, "kq");
  CHECK_PTR(ksc, "ksc");
  CHECK_PTR(vq, "vq");
  CHECK_PTR(vsc, "vsc");
  if (kcur && !aligned16(kcur)) return fail(QSA_ERR_INVALID_ARG, "kcur is not 16-byte aligned");
  if (pos3 && (reinterpret_cast<uintptr_t>(pos3) & 3u)) return fail(QSA_ERR_INVALID_ARG, "pos3 is not 4-byte aligned");
  if (T <= 0) return fail(QSA_ERR_INVALID_ARG, "T must be positive (got %d)", T);
  if (pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "pos0 must be >= 0 (got %d)", pos0);
  if ((long long)pos0 + T > (long long)n_cells)
    return fail(QSA_ERR_INVALID_ARG, "cache too small: pos0 + T = %lld > n_cells = %d", (long long)pos0 + T, n_cells);
  const int rd = r.rotary_dim;
  if (rd < 16 || rd > 256 || (rd & (rd - 1)))
    return fail(QSA_ERR_UNSUPPORTED, "rotary_dim must be a power of two in [16, 256] (got %d)", rd);
  if (!(r.base > 1.f) || !(r.base < 3.0e38f)) return fail(QSA_ERR_INVALID_ARG, "rope base must be > 1 and finite");
  if (!(r.eps > 0.f) || !(r.eps < 1.f)) return fail(QSA_ERR_INVALID_ARG, "eps must be in (0, 1)");
  if (pos3 && (r.sections[0] < 0 || r.sections[1] < 0 || r.sections[2] < 0 ||
               r.sections[0] + r.sections[1] + r.sections[2] != rd / 2))
    return fail(QSA_ERR_INVALID_ARG, "mrope sections must be >= 0 and sum to rotary_dim / 2 = %d", rd / 2);
  cudaError_t e = qsa::launch_prep(
      reinterpret_cast<const __half*>(q_raw), reinterpret_cast<const __half*>(k_raw),
      reinterpret_cast<const __half*>(v_raw), q_gamma, k_gamma, pos3, T, pos0, (double)r.base, rd, r.eps, r.sections,
      reinterpret_cast<__half*>(qcur), reinterpret_cast<__half*>(kcur), kq, reinterpret_cast<__half*>(ksc), vq,
      reinterpret_cast<__half*>(vsc), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_prep launch");
  return ok();
}

size_t qsa_select_workspace_bytes(int T, int pos0, int n_cells, const qsa_params* params) {
  qsa::Params p;
  if (T <= 0 || pos0 < 0 || n_cells <= 0 || resolve_params(params, &p) != QSA_OK) return 0;
  return qsa::select_workspace_bytes(T, pos0, n_cells, p);
}

int qsa_select(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T, int pos0, int32_t* ids,
               void* ws, size_t ws_bytes, const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  if ((rc = check_layer(q, kq, ksc, n_cells, T, pos0))) return rc;
  const int t_sel = qsa::first_selected_token(pos0, p.identity_max);
  if (t_sel >= T) return ok();  // every token at or under the threshold: nothing to select
  CHECK_PTR(ids, "ids");
  if ((long long)pos0 + T > qsa::select_max_cells())
    return select_long(q, kq, ksc, n_cells, T, pos0, ids, p, stream, "qsa_select");
  const size_t need = qsa::select_workspace_bytes(T, pos0, n_cells, p);
  if (need == 0) return fail(QSA_ERR_UNSUPPORTED, "selection over n_kv up to %lld cells is not supported",
                             (long long)pos0 + T);
  // A smaller workspace takes the selected tokens in consecutive chunks of Tc tokens, each the same
  // call over its own token range (rows are independent; the ids are the same): the largest Tc whose
  // last chunk (the one with the most cells) fits.
  int Tc = T - t_sel;
  if (ws && ws_bytes < need) {
    const int T_sel = T - t_sel;
    auto fits = [&](int c) {
      const size_t nb = qsa::select_workspace_bytes(c, pos0 + T - c, n_cells, p);
      return nb != 0 && nb <= ws_bytes;
    };
    Tc = 0;
    for (int c = T_sel / 128 * 128; c >= 128 && !Tc; c -= 128)
      if (fits(c)) Tc = c;
    for (int c = 64; c >= 1 && !Tc; c >>= 1)
      if (c < T_sel && fits(c)) Tc = c;
  }
  if (!ws || Tc == 0)
    return fail(QSA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed (at least %zu in chunks of one token)",
                ws ? ws_bytes : (size_t)0, need, qsa::select_workspace_bytes(1, pos0 + T - 1, n_cells, p));
  if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int a = t_sel; a < T; a += Tc) {
    const int b = a + Tc < T ? a + Tc : T;
    cudaError_t e = qsa::launch_select(reinterpret_cast<const __half*>(q) + (size_t)a * QSA_N_HEADS * QSA_HEAD_DIM, kq,
                                       reinterpret_cast<const __half*>(ksc), n_cells, b - a, pos0 + a,
                                       ids + (size_t)a * QSA_N_GROUPS * p.topk, ws, p, st, s);
    if (e != cudaSuccess) return cuda_fail(e, "qsa_select launch");
  }
  return ok();
}

size_t qsa_flash_prefill_workspace_bytes(int T, int pos0, int n_cells, const qsa_params* params) {
  qsa::Params p;
  if (T <= 0 || pos0 < 0 || n_cells <= 0 || resolve_params(params, &p) != QSA_OK) return 0;
  return qsa::prefill_workspace_bytes(T, pos0);
}

int qsa_flash_prefill(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc, const uint16_t* vsc,
                      int n_cells, int T, int pos0, const int32_t* ids, uint16_t* out, void* ws, size_t ws_bytes,
                      const qsa_params* params, void* stream) {
  return qsa_flash_prefill_gated(q, kq, vq, ksc, vsc, n_cells, T, pos0, ids, nullptr, out, ws, ws_bytes, params,
                                 stream);
}

int qsa_flash_prefill_gated(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                            const uint16_t* vsc, int n_cells, int T, int pos0, const int32_t* ids, const uint16_t* gate,
                            uint16_t* out, void* ws, size_t ws_bytes, const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  if ((rc = check_layer(q, kq, ksc, n_cells, T, pos0))) return rc;
  CHECK_PTR(vq, "vq");
  CHECK_PTR(vsc, "vsc");
  CHECK_PTR(out, "out");
  const int t_sel = qsa::first_selected_token(pos0, p.identity_max);
  if (t_sel < T) CHECK_PTR(ids, "ids (needed: some tokens are above the identity threshold)");
  if (gate && !aligned16(gate)) return fail(QSA_ERR_INVALID_ARG, "gate is not 16-byte aligned");
  const size_t need = qsa::prefill_workspace_bytes(T, pos0);
  if (!ws || ws_bytes < need)
    return fail(QSA_ERR_WORKSPACE, "prefill workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0,
                need);
  if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  int* st = status_ptr(&rc);
  if (!st) return rc;
  qsa::FlashArgs a{reinterpret_cast<const __half*>(q), kq, vq, reinterpret_cast<const __half*>(ksc),
                   reinterpret_cast<const __half*>(vsc), ids, reinterpret_cast<const __half*>(gate),
                   reinterpret_cast<__half*>(out), n_cells, T, pos0, p, st};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = pos0 + T;
  __half* khat = static_cast<__half*>(ws);
  __half* vhat = khat + (size_t)n * QSA_N_GROUPS * QSA_HEAD_DIM;
  cudaError_t e = qsa::launch_dequant_mirror(kq, vq, a.ksc, a.vsc, n, khat, vhat, s);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill (fp16 mirror) launch");
  const int split = t_sel < T ? t_sel : T;
  e = qsa::launch_flash_dense(a, 0, split, khat, vhat, s);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill (identity tokens) launch");
  e = qsa::launch_flash_gather(a, split, T, khat, vhat, s);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill (selected tokens) launch");
  return ok();
}

int qsa_decode_partial(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc, const uint16_t* vsc,
                       int n_cells, int N, int pos0, const int32_t* ids, float* part, int32_t* n_chunks, int chunk_cap,
                       const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  if ((rc = check_layer(q, kq, ksc, n_cells, N, pos0))) return rc;
  CHECK_PTR(vq, "vq");
  CHECK_PTR(vsc, "vsc");
  CHECK_PTR(part, "part");
  CHECK_PTR(n_chunks, "n_chunks");
  const int need_cap = ((p.identity_max > p.topk ? p.identity_max : p.topk) + QSA_CHUNK - 1) / QSA_CHUNK;
  if (chunk_cap < need_cap) return fail(QSA_ERR_INVALID_ARG, "chunk_cap %d < %d", chunk_cap, need_cap);
  if (chunk_cap > 65535) return fail(QSA_ERR_UNSUPPORTED, "chunk_cap %d > 65535", chunk_cap);
  const int t_sel = qsa::first_selected_token(pos0, p.identity_max);
  if (t_sel < N) CHECK_PTR(ids, "ids (needed: some tokens are above the identity threshold)");
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaError_t e = qsa::launch_decode_partial(
      reinterpret_cast<const __half*>(q), kq, vq, reinterpret_cast<const __half*>(ksc),
      reinterpret_cast<const __half*>(vsc), ids, part, n_chunks, chunk_cap, n_cells, N, pos0, p, st,
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_decode_partial launch");
  return ok();
}

int qsa_merge(const float* part, const int32_t* n_chunks, int N, int chunk_cap, float* xp, void* stream) {
  return qsa_merge_gated(part, n_chunks, N, chunk_cap, nullptr, xp, stream);
}

int qsa_merge_gated(const float* part, const int32_t* n_chunks, int N, int chunk_cap, const uint16_t* gate, float* xp,
                    void* stream) {
  if (gate && !aligned16(gate)) return fail(QSA_ERR_INVALID_ARG, "gate is not 16-byte aligned");
  CHECK_PTR(part, "part");
  CHECK_PTR(n_chunks, "n_chunks");
  CHECK_PTR(xp, "xp");
  if (N <= 0) return fail(QSA_ERR_INVALID_ARG, "N must be positive (got %d)", N);
  if (chunk_cap < 1 || chunk_cap > 1024) return fail(QSA_ERR_UNSUPPORTED, "chunk_cap must be in [1, 1024]");
  int rc = 0;
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaError_t e = qsa::launch_merge(part, n_chunks, N, chunk_cap, reinterpret_cast<const __half*>(gate), xp, st,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_merge launch");
  return ok();
}

int qsa_decode_layer(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc, const uint16_t* vsc,
                     int n_cells, int N, int pos0, int32_t* ids, const uint16_t* gate, float* xp,
                     const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  if ((rc = check_layer(q, kq, ksc, n_cells, N, pos0))) return rc;
  CHECK_PTR(vq, "vq");
  CHECK_PTR(vsc, "vsc");
  CHECK_PTR(xp, "xp");
  if (ids && !aligned16(ids)) return fail(QSA_ERR_INVALID_ARG, "ids is not 16-byte aligned");
  if (gate && !aligned16(gate)) return fail(QSA_ERR_INVALID_ARG, "gate is not 16-byte aligned");
  if (N > 65535) return fail(QSA_ERR_UNSUPPORTED, "N must be at most 65535 (got %d)", N);
  const int limit = decode_layer_limit(&rc);
  if (!limit) return rc;
  if ((long long)pos0 + N > limit)
    return fail(QSA_ERR_UNSUPPORTED, "qsa_decode_layer takes n_kv up to %d cells (got %lld)", limit,
                (long long)pos0 + N);
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaError_t e = qsa::launch_decode_layer(
      reinterpret_cast<const __half*>(q), kq, vq, reinterpret_cast<const __half*>(ksc),
      reinterpret_cast<const __half*>(vsc), nullptr, 1, (long long)n_cells, n_cells, pos0, N, pos0 + N, ids,
      reinterpret_cast<const __half*>(gate), xp, p, st, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_decode_layer launch");
  return ok();
}

int qsa_decode_layer_batched(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                             const uint16_t* vsc, int64_t n_pool, const int32_t* seqs, int n_seq, int n_tok,
                             int max_n_kv, int32_t* ids, const uint16_t* gate, float* xp, const qsa_params* params,
                             void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  CHECK_PTR(q, "q");
  CHECK_PTR(kq, "kq");
  CHECK_PTR(vq, "vq");
  CHECK_PTR(ksc, "ksc");
  CHECK_PTR(vsc, "vsc");
  CHECK_PTR(seqs, "seqs");
  CHECK_PTR(xp, "xp");
  if (ids && !aligned16(ids)) return fail(QSA_ERR_INVALID_ARG, "ids is not 16-byte aligned");
  if (gate && !aligned16(gate)) return fail(QSA_ERR_INVALID_ARG, "gate is not 16-byte aligned");
  if (n_pool <= 0) return fail(QSA_ERR_INVALID_ARG, "n_pool must be positive");
  if (n_seq < 1 || n_tok < n_seq)
    return fail(QSA_ERR_INVALID_ARG, "need 1 <= n_seq <= n_tok (got n_seq %d, n_tok %d)", n_seq, n_tok);
  if (n_tok > 65535) return fail(QSA_ERR_UNSUPPORTED, "n_tok must be at most 65535 (got %d)", n_tok);
  const int limit = decode_layer_limit(&rc);
  if (!limit) return rc;
  if (max_n_kv < 1 || max_n_kv > limit)
    return fail(QSA_ERR_UNSUPPORTED, "max_n_kv must be in [1, %d] (got %d)", limit, max_n_kv);
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaError_t e = qsa::launch_decode_layer(
      reinterpret_cast<const __half*>(q), kq, vq, reinterpret_cast<const __half*>(ksc),
      reinterpret_cast<const __half*>(vsc), reinterpret_cast<const int4*>(seqs), n_seq, (long long)n_pool, 0, 0, n_tok,
      max_n_kv, ids, reinterpret_cast<const __half*>(gate), xp, p, st, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qsa_decode_layer_batched launch");
  return ok();
}

size_t qsa_flash_prefill_batched_workspace_bytes(int n_seq, int n_tok, int max_n_kv, const qsa_params* params) {
  qsa::Params p{};
  if (n_seq < 1 || n_tok < 1 || max_n_kv < 1 || resolve_params(params, &p) != QSA_OK) return 0;
  return qsa::batched_prefill_layout(n_seq, n_tok, max_n_kv, p.identity_max).bytes;
}

int qsa_flash_prefill_batched(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                              const uint16_t* vsc, int64_t n_pool, const int32_t* seqs, int n_seq, int n_tok,
                              int max_n_kv, int32_t* ids, const uint16_t* gate, uint16_t* out, void* ws,
                              size_t ws_bytes, const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  CHECK_PTR(q, "q");
  CHECK_PTR(kq, "kq");
  CHECK_PTR(vq, "vq");
  CHECK_PTR(ksc, "ksc");
  CHECK_PTR(vsc, "vsc");
  CHECK_PTR(seqs, "seqs");
  CHECK_PTR(out, "out");
  if (ids && !aligned16(ids)) return fail(QSA_ERR_INVALID_ARG, "ids is not 16-byte aligned");
  if (gate && !aligned16(gate)) return fail(QSA_ERR_INVALID_ARG, "gate is not 16-byte aligned");
  if (n_pool <= 0) return fail(QSA_ERR_INVALID_ARG, "n_pool must be positive");
  if (n_seq < 1 || n_tok < 1) return fail(QSA_ERR_INVALID_ARG, "need n_seq >= 1 and n_tok >= 1 (got %d, %d)", n_seq, n_tok);
  if (n_tok > 65535 || n_seq > 65535)
    return fail(QSA_ERR_UNSUPPORTED, "n_tok and n_seq must be at most 65535 (got %d, %d)", n_tok, n_seq);
  const bool any_selected = max_n_kv > p.identity_max;
  int limit = 131072;  // the dense work list counts up to 1024 super-chunks of 128 cells
  if (any_selected) {
    const int l2 = decode_layer_limit(&rc);
    if (!l2) return rc;
    limit = l2 < limit ? l2 : limit;
  }
  if (max_n_kv < 1 || max_n_kv > limit)
    return fail(QSA_ERR_UNSUPPORTED, "max_n_kv must be in [1, %d] (got %d)", limit, max_n_kv);
  const qsa::BatchedPrefillLayout L = qsa::batched_prefill_layout(n_seq, n_tok, max_n_kv, p.identity_max);
  if (L.mirror_rows > 0x7fffffffLL) return fail(QSA_ERR_UNSUPPORTED, "n_seq x mirror rows per sequence exceeds 2^31");
  if (!ws || ws_bytes < L.bytes)
    return fail(QSA_ERR_WORKSPACE, "batched prefill workspace of %zu bytes given, %zu needed", ws ? ws_bytes : (size_t)0,
                L.bytes);
  if (!aligned16(ws)) return fail(QSA_ERR_INVALID_ARG, "ws is not 16-byte aligned");
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int4* sq = reinterpret_cast<const int4*>(seqs);
  const __half* hksc = reinterpret_cast<const __half*>(ksc);
  const __half* hvsc = reinterpret_cast<const __half*>(vsc);
  cudaError_t e = qsa::launch_batched_prefill_prep(kq, vq, hksc, hvsc, sq, n_seq, n_tok, (long long)n_pool, max_n_kv,
                                                   p.identity_max, L, ws, st, s);
  if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill_batched (work list and mirror) launch");
  if (L.rows_per_seq > 0) {
    const int4* plan = static_cast<const int4*>(ws);
    const __half* khat = reinterpret_cast<const __half*>(static_cast<const uint8_t*>(ws) + L.plan_bytes);
    const __half* vhat = khat + (size_t)L.mirror_rows * QSA_N_GROUPS * QSA_HEAD_DIM;
    e = qsa::launch_flash_dense_batched(reinterpret_cast<const __half*>(q), n_tok, reinterpret_cast<const __half*>(gate),
                                        reinterpret_cast<__half*>(out), plan, L.max_pairs, khat, vhat,
                                        (int)L.mirror_rows, p.sm_scale, st, s);
    if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill_batched (identity tokens) launch");
  }
  if (any_selected) {
    e = qsa::launch_decode_layer(reinterpret_cast<const __half*>(q), kq, vq, hksc, hvsc, sq, n_seq, (long long)n_pool, 0,
                                 0, n_tok, max_n_kv, ids, reinterpret_cast<const __half*>(gate), nullptr, p, st, s,
                                 reinterpret_cast<__half*>(out), true);
    if (e != cudaSuccess) return cuda_fail(e, "qsa_flash_prefill_batched (selected tokens) launch");
  }
  return ok();
}

}  // extern "C"

namespace {
// One warp waits, with the library's bounded mbarrier wait and the given budget, for the first
// phase of a barrier that nothing arrives on; the wait can only give up, which sets the status
// word.  Nothing asynchronous is in flight, so the CTA leaves cleanly.
__global__ void wait_probe_kernel(unsigned long long budget_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    qsa::mbar_init(&bar, 1);
    qsa::fence_mbar_init();
  }
  __syncthreads();
  qsa::mbar_wait(&bar, 0u, status, nullptr, budget_ns);
}
}  // namespace

extern "C" {

int qsa_debug_wait_probe(uint64_t budget_ns, void* stream) {
  if (budget_ns < 1000ull || budget_ns > qsa::kWaitBudgetNs)
    return fail(QSA_ERR_INVALID_ARG, "budget_ns must be in [1000, %llu]", (unsigned long long)qsa::kWaitBudgetNs);
  int rc = 0;
  int* st = status_ptr(&rc);
  if (!st) return rc;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((unsigned long long)budget_ns, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "qsa_debug_wait_probe launch");
  return ok();
}

int qsa_check_device_status(void* stream) {
  int rc = 0;
  int* st = status_ptr(&rc);
  if (!st) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, qsa::g_status_word, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(qsa::g_status_word, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    if (v == qsa::QSA_DEV_WAIT_TIMEOUT) return fail(QSA_ERR_TIMEOUT, "a bounded device wait timed out");
    if (v == qsa::QSA_DEV_BAND_OVERFLOW) return fail(QSA_ERR_DEVICE, "selection refinement capacity exceeded");
    if (v == qsa::QSA_DEV_BAD_ID) return fail(QSA_ERR_DEVICE, "an id or chunk count was out of range");
    return fail(QSA_ERR_DEVICE, "device status %d", v);
  }
  return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// qsa_select_noalloc: qsa_select for callers that cannot allocate device memory.
//
// The selection kernels need scratch memory (the score matrix and its inputs).  qsa_select
// takes it from the caller; this entry point instead uses a fixed scratch array that lives
// in the library's own device memory, so the caller passes only its inputs and outputs.
// The array is kNoAllocScratchBytes on every device that loads the library and stays
// allocated until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;  // 24 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up once per device.
// In host code the array's name is only a host-side stand-in, never a device address.
void* noalloc_scratch_ptr(int* err) {
  static void* cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    *err = cuda_fail(e == cudaSuccess ? cudaErrorInvalidDevice : e, "cudaGetDevice");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *err = cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
      return nullptr;
    }
    cache[dev] = p;
  }
  return cache[dev];
}

}  // namespace

extern "C" int qsa_select_noalloc(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T,
                                  int pos0, int32_t* ids, const qsa_params* params, void* stream) {
  qsa::Params p;
  int rc = resolve_params(params, &p);
  if (rc) return rc;
  if ((rc = check_layer(q, kq, ksc, n_cells, T, pos0))) return rc;
  if (qsa::first_selected_token(pos0, p.identity_max) >= T) return ok();  // nothing to select
  if ((long long)pos0 + T > qsa::select_max_cells()) {  // needs no scratch at all
    CHECK_PTR(ids, "ids");
    return select_long(q, kq, ksc, n_cells, T, pos0, ids, p, stream, "qsa_select_noalloc");
  }
  const size_t need = qsa::select_workspace_bytes(T, pos0, n_cells, p);
  if (need == 0)
    return fail(QSA_ERR_UNSUPPORTED, "selection over n_kv up to %lld cells is not supported", (long long)pos0 + T);
  if (need > kNoAllocScratchBytes)
    return fail(QSA_ERR_UNSUPPORTED,
                "qsa_select_noalloc: this call needs %zu bytes of scratch but the built-in scratch holds %zu "
                "(about 16 selected tokens over 16384 cells); use qsa_select with a caller workspace",
                need, kNoAllocScratchBytes);
  void* ws = noalloc_scratch_ptr(&rc);
  if (!ws) return rc;
  return qsa_select(q, kq, ksc, n_cells, T, pos0, ids, ws, kNoAllocScratchBytes, params, stream);
}
