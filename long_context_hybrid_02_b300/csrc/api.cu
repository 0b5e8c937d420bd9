// C ABI of libhybridattn.so: host-side argument checks, launch planning and
// dispatch to the kernels.  Every entry point validates its arguments before any
// CUDA call, launches on the caller's stream and returns without synchronising.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "hybrid_attn.h"
#include "kernels.h"

namespace ha {

namespace {
std::atomic<unsigned long long> g_launches{0};
struct SmemGrant { const void* func; int device; size_t bytes; };
SmemGrant g_grants[256];
int g_n_grants = 0;
std::mutex g_grant_mu;
}  // namespace

cudaError_t ensure_smem(const void* func, size_t bytes) {
  // the default limit (48 KiB) covers static plus dynamic shared memory together
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, func);
  if (e != cudaSuccess) return e;
  if (bytes + fa.sharedSizeBytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_grant_mu);
  for (int i = 0; i < g_n_grants; ++i)
    if (g_grants[i].func == func && g_grants[i].device == dev) {
      if (g_grants[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
      if (e == cudaSuccess) g_grants[i].bytes = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
  if (e == cudaSuccess && g_n_grants < 256) g_grants[g_n_grants++] = {func, dev, bytes};
  return e;
}

cudaError_t launched(cudaError_t e) {
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

unsigned long long launch_count() { return g_launches.load(); }

}  // namespace ha

namespace {

thread_local char g_last_error[512] = "";

// One NVTX range per library call (host side: argument checks, planning and the
// launches), named after the entry point; a no-op unless a profiler is attached.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

ha_status fail(ha_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

ha_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return HA_OK;
  return fail(HA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

#define HA_REQUIRE(cond, code, ...) \
  do {                              \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

#define HA_PTR(ptr)                                                                 \
  do {                                                                              \
    HA_REQUIRE((ptr) != nullptr, HA_ERR_INVALID_ARG, "%s is NULL", #ptr);           \
    HA_REQUIRE(aligned16(ptr), HA_ERR_MISALIGNED, "%s is not 16-byte aligned", #ptr); \
  } while (0)

// Arrays read as scalars (positions, indices, gates, weights, scores, lse) need
// only their natural 4-byte alignment.
#define HA_PTR4(ptr)                                                                \
  do {                                                                              \
    HA_REQUIRE((ptr) != nullptr, HA_ERR_INVALID_ARG, "%s is NULL", #ptr);           \
    HA_REQUIRE((reinterpret_cast<uintptr_t>(ptr) & 3u) == 0, HA_ERR_MISALIGNED,     \
               "%s is not 4-byte aligned", #ptr);                                   \
  } while (0)

#define HA_OPT_PTR4(ptr)                                                              \
  do {                                                                                \
    if ((ptr) != nullptr)                                                             \
      HA_REQUIRE((reinterpret_cast<uintptr_t>(ptr) & 3u) == 0, HA_ERR_MISALIGNED,     \
                 "%s is not 4-byte aligned", #ptr);                                   \
  } while (0)

#define HA_OPT_PTR(ptr)                                                               \
  do {                                                                                \
    if ((ptr) != nullptr)                                                             \
      HA_REQUIRE(aligned16(ptr), HA_ERR_MISALIGNED, "%s is not 16-byte aligned", #ptr); \
  } while (0)

ha_status check_params(const ha_params* p, bool need_attn, bool need_index) {
  HA_REQUIRE(p != nullptr, HA_ERR_INVALID_ARG, "params is NULL");
  HA_REQUIRE(p->dtype == HA_F32 || p->dtype == HA_BF16, HA_ERR_INVALID_ARG, "dtype %d", p->dtype);
  HA_REQUIRE(p->elig == HA_ELIG_DISJOINT || p->elig == HA_ELIG_OVERLAP, HA_ERR_INVALID_ARG,
             "elig %d", p->elig);
  HA_REQUIRE(p->B >= 1, HA_ERR_INVALID_ARG, "B = %d", p->B);
  HA_REQUIRE(p->m >= 1 && p->m <= 1024, HA_ERR_UNSUPPORTED, "m = %d (1..1024)", p->m);
  HA_REQUIRE(p->n_win >= 1 && p->n_win <= 65536, HA_ERR_UNSUPPORTED, "n_win = %d", p->n_win);
  HA_REQUIRE(p->d >= 8 && p->d <= 1024 && p->d % 8 == 0, HA_ERR_UNSUPPORTED,
             "d = %d (8..1024, multiple of 8)", p->d);
  if (need_attn) {
    HA_REQUIRE(p->H >= 1 && p->H <= 256, HA_ERR_UNSUPPORTED, "H = %d (1..256)", p->H);
    HA_REQUIRE(isfinite(p->scale), HA_ERR_INVALID_ARG, "scale is not finite");
  }
  HA_REQUIRE((p->fmt & ~(HA_FMT_IDX4 | HA_FMT_KV8)) == 0, HA_ERR_INVALID_ARG, "fmt = %d", p->fmt);
  HA_REQUIRE(!(p->fmt & HA_FMT_KV8) || p->d == 512, HA_ERR_UNSUPPORTED,
             "the FP8 KV format needs d = 512 (d = %d)", p->d);
  HA_REQUIRE(p->fmt == 0 || p->dtype == HA_BF16, HA_ERR_UNSUPPORTED,
             "storage formats need bfloat16 (fmt = %d)", p->fmt);
  if ((p->fmt & HA_FMT_IDX4) && need_index)
    HA_REQUIRE(p->H_I == 64 && p->d_I == 128, HA_ERR_UNSUPPORTED,
               "the FP4 indexer needs H_I = 64 and d_I = 128 (got %d, %d)", p->H_I, p->d_I);
  if (need_index) {
    HA_REQUIRE(p->H_I >= 1 && p->H_I <= 128, HA_ERR_UNSUPPORTED, "H_I = %d (1..128)", p->H_I);
    HA_REQUIRE(p->d_I >= 8 && p->d_I <= 512 && p->d_I % 8 == 0, HA_ERR_UNSUPPORTED,
               "d_I = %d (8..512, multiple of 8)", p->d_I);
    HA_REQUIRE((size_t)p->H_I * p->d_I <= 32768, HA_ERR_UNSUPPORTED, "H_I * d_I = %d > 32768",
               p->H_I * p->d_I);
  }
  return HA_OK;
}

ha_status check_k(const ha_params* p) {
  HA_REQUIRE(p->k >= 1 && p->k <= 4096, HA_ERR_UNSUPPORTED, "k = %d (1..4096)", p->k);
  return HA_OK;
}

int max_keys(const ha_params* p, int n_cap, bool is_csa) {
  return (is_csa ? p->k : n_cap) + p->n_win;
}

// Launch plan of the attention calls: the tensor-core kernel where it applies (its
// workspace does not depend on tok_cap, so ha_workspace_size passes 0 for it),
// else the CUDA-core kernel.
ha::AttnPlan attention_plan(const ha_params* p, int rows, int n_cap, int tok_cap, bool is_csa,
                            bool decode) {
  if (ha::attention_tc_supported(*p, n_cap, tok_cap))
    return ha::plan_attention_tc(*p, rows, max_keys(p, n_cap, is_csa));
  return ha::plan_attention_simt(*p, rows, max_keys(p, n_cap, is_csa), decode);
}

ha_status compress_common(const ha_params* p, int n_tensors, const void* const* src,
                          void* const* dst, const int* dims, const float* gate, int32_t tok_cap,
                          const int32_t* blk_begin, int32_t n_blk, int32_t n_cap,
                          ha_stream_t stream, bool csa) {
  ha_status s = check_params(p, false, csa);
  if (s != HA_OK) return s;
  for (int i = 0; i < n_tensors; ++i) {
    HA_REQUIRE(src[i] != nullptr && dst[i] != nullptr, HA_ERR_INVALID_ARG, "tensor %d is NULL", i);
    HA_REQUIRE(aligned16(src[i]) && aligned16(dst[i]), HA_ERR_MISALIGNED,
               "tensor %d is not 16-byte aligned", i);
  }
  HA_PTR4(gate);
  HA_PTR4(blk_begin);
  HA_REQUIRE(tok_cap >= p->m, HA_ERR_INVALID_ARG, "tok_cap = %d < m = %d", tok_cap, p->m);
  HA_REQUIRE(!(csa && (p->fmt & HA_FMT_IDX4)) || p->m <= 16, HA_ERR_UNSUPPORTED,
             "FP4 indexer keys need m <= 16 (m = %d)", p->m);
  HA_REQUIRE(n_blk >= 0, HA_ERR_INVALID_ARG, "n_blk = %d", n_blk);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  HA_REQUIRE((long long)p->B * n_blk <= 0x7fffffffLL, HA_ERR_UNSUPPORTED, "B * n_blk too large");
  if (n_blk == 0) return HA_OK;
  return cuda_status(ha::launch_compress(*p, n_tensors, src, dst, dims, gate, blk_begin, n_blk,
                                         tok_cap, n_cap, (cudaStream_t)stream),
                     "compress launch");
}

}  // namespace

namespace {

size_t round_up256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace of an attention call: the plan's split partials, then, for FP8 K/V
// rows, the rows widened to bfloat16 (the selected entries of a decode selection,
// else every entry of the cache).
size_t attn_ws_bytes(const ha_params* p, const ha::AttnPlan& pl, int n_cap, bool select) {
  if (!(p->fmt & HA_FMT_KV8)) return pl.ws_bytes;
  return round_up256(pl.ws_bytes) + ha::kv8_expand_bytes(*p, n_cap, select);
}

// FP8 K/V rows: widen the rows the attention reads into the workspace (after the
// partials) and point ck, cv, n_cap and (selection) idx at the widened view.
cudaError_t kv8_view(const ha_params* p, const ha::AttnPlan& pl, const void*& ck, const void*& cv,
                     int& n_cap, const int32_t*& idx, bool select, const int32_t* ctx_len,
                     void* ws, cudaStream_t st) {
  if (!(p->fmt & HA_FMT_KV8)) return cudaSuccess;
  ha::KvExpanded ex{};
  cudaError_t e = ha::launch_kv8_expand(*p, ck, cv, n_cap, select ? idx : nullptr, ctx_len,
                                        static_cast<char*>(ws) + round_up256(pl.ws_bytes), &ex, st);
  if (e != cudaSuccess) return e;
  ck = ex.ck;
  cv = ex.cv;
  n_cap = ex.n_cap;
  if (select) idx = ex.idx;
  return cudaSuccess;
}

// Workspace of a fused decode step: the top-k part (segmented rows), then the
// attention's.
size_t step_workspace_bytes(const ha_params* p, int n_cap, int tok_cap, bool is_csa) {
  const size_t topk = is_csa ? round_up256(ha::topk_workspace_bytes(*p, 1, n_cap)) : 0;
  return topk + attn_ws_bytes(p, attention_plan(p, p->B, n_cap, tok_cap, is_csa, true), n_cap, is_csa);
}

// Checks shared by the two fused decode steps (everything but the indexer inputs).
ha_status check_step(const ha_params* p, const void* q, const void* k_tok, const void* v_tok,
                     const float* gate, int32_t tok_cap, const int32_t* ctx_len, const void* ck,
                     const void* cv, int32_t n_cap, const void* o, const float* lse) {
  HA_PTR(q);
  HA_PTR(k_tok);
  HA_PTR(v_tok);
  HA_PTR4(gate);
  HA_PTR4(ctx_len);
  HA_PTR(ck);
  HA_PTR(cv);
  HA_PTR(o);
  HA_OPT_PTR4(lse);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  HA_REQUIRE(tok_cap >= p->n_win && tok_cap >= p->m, HA_ERR_INVALID_ARG,
             "tok_cap = %d < max(n_win = %d, m = %d)", tok_cap, p->n_win, p->m);
  return HA_OK;
}

}  // namespace

size_t ha::decode_workspace_bytes(const ha_params* p, int n_cap, int tok_cap, bool is_csa) {
  return attn_ws_bytes(p, attention_plan(p, p->B, n_cap, tok_cap, is_csa, true), n_cap, is_csa);
}

void ha::set_last_error(const char* msg) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

extern "C" {

int32_t ha_abi_version(void) { return 3; }

uint64_t ha_launch_count(void) { return ha::launch_count(); }

void* ha_host_alloc(size_t bytes, int32_t write_combined) {
  g_last_error[0] = 0;
  if (bytes == 0) {
    ha::set_last_error("ha_host_alloc: bytes = 0");
    return nullptr;
  }
  void* p = nullptr;
  const cudaError_t e = cudaHostAlloc(
      &p, bytes, write_combined ? cudaHostAllocWriteCombined : cudaHostAllocDefault);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof msg, "ha_host_alloc(%zu): %s", bytes, cudaGetErrorString(e));
    ha::set_last_error(msg);
    return nullptr;
  }
  return p;
}

ha_status ha_host_free(void* p) {
  g_last_error[0] = 0;
  if (p == nullptr) return HA_OK;
  return cuda_status(cudaFreeHost(p), "ha_host_free");
}

const char* ha_last_error(void) { return g_last_error; }

const char* ha_status_string(ha_status s) {
  switch (s) {
    case HA_OK: return "ok";
    case HA_ERR_INVALID_ARG: return "invalid argument";
    case HA_ERR_MISALIGNED: return "pointer misaligned (16 bytes for tensors, 4 for scalar arrays)";
    case HA_ERR_UNSUPPORTED: return "shape outside the supported limits";
    case HA_ERR_WORKSPACE: return "workspace missing or too small";
    case HA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

ha_status hca_compress_kv(const ha_params* p, const void* k_tok, const void* v_tok,
                          const float* gate, int32_t tok_cap, const int32_t* blk_begin,
                          int32_t n_blk, void* ck, void* cv, int32_t n_cap,
                          ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("hca_compress_kv");
  if (!p) return fail(HA_ERR_INVALID_ARG, "params is NULL");
  const void* src[2] = {k_tok, v_tok};
  void* dst[2] = {ck, cv};
  const int dims[2] = {p->d, p->d};
  return compress_common(p, 2, src, dst, dims, gate, tok_cap, blk_begin, n_blk, n_cap, stream,
                         false);
}

ha_status csa_compress_kv(const ha_params* p, const void* k_tok, const void* v_tok,
                          const void* ki_tok, const float* gate, int32_t tok_cap,
                          const int32_t* blk_begin, int32_t n_blk, void* ck, void* cv,
                          void* cki, int32_t n_cap, ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("csa_compress_kv");
  if (!p) return fail(HA_ERR_INVALID_ARG, "params is NULL");
  const void* src[3] = {k_tok, v_tok, ki_tok};
  void* dst[3] = {ck, cv, cki};
  const int dims[3] = {p->d, p->d, p->d_I};
  return compress_common(p, 3, src, dst, dims, gate, tok_cap, blk_begin, n_blk, n_cap, stream,
                         true);
}

ha_status csa_index_scores(const ha_params* p, const void* q_idx, const float* w_idx,
                           const void* cki, int32_t n_cap, const int32_t* q_pos, int32_t Tq,
                           void* scores, ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("csa_index_scores");
  ha_status s = check_params(p, false, true);
  if (s != HA_OK) return s;
  HA_PTR(q_idx);
  HA_PTR4(w_idx);
  HA_PTR(cki);
  HA_PTR4(q_pos);
  HA_PTR4(scores);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  HA_REQUIRE(Tq >= 1, HA_ERR_INVALID_ARG, "Tq = %d", Tq);
  HA_REQUIRE((long long)p->B * Tq <= 0x7fffffffLL, HA_ERR_UNSUPPORTED, "B * Tq too large");
  if (ha::index_scores_tc_supported(*p, q_idx, cki)) {
    int* err = ha::device_error_word();
    HA_REQUIRE(err != nullptr, HA_ERR_CUDA, "device error word unavailable");
    return cuda_status(ha::launch_index_scores_tc(*p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores,
                                                  err, (cudaStream_t)stream),
                       "index launch (tensor cores)");
  }
  return cuda_status(ha::launch_index_scores_simt(*p, q_idx, w_idx, cki, n_cap, q_pos, Tq,
                                                  static_cast<float*>(scores), (cudaStream_t)stream),
                     "index launch");
}

ha_status csa_topk(const ha_params* p, const void* scores, int32_t n_cap, const int32_t* q_pos,
                   int32_t Tq, int32_t* idx, void* ws, size_t ws_bytes, ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("csa_topk");
  ha_status s = check_params(p, false, false);
  if (s != HA_OK) return s;
  s = check_k(p);
  if (s != HA_OK) return s;
  HA_PTR4(scores);
  HA_PTR4(q_pos);
  HA_PTR4(idx);
  HA_OPT_PTR(ws);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  HA_REQUIRE(n_cap <= ha::topk_max_row_entries(), HA_ERR_UNSUPPORTED, "n_cap = %d > %d", n_cap,
             ha::topk_max_row_entries());
  HA_REQUIRE(Tq >= 1, HA_ERR_INVALID_ARG, "Tq = %d", Tq);
  HA_REQUIRE((long long)p->B * Tq <= 0x7fffffffLL, HA_ERR_UNSUPPORTED, "B * Tq too large");
  const size_t need = ha::topk_workspace_bytes(*p, Tq, n_cap);
  HA_REQUIRE(ws_bytes >= need && (need == 0 || ws != nullptr), HA_ERR_WORKSPACE,
             "workspace %zu bytes < %zu", ws_bytes, need);
  return cuda_status(ha::launch_topk(*p, scores, n_cap, q_pos, Tq, idx, ws, ws_bytes,
                                     (cudaStream_t)stream),
                     "top-k launch");
}

ha_status hybrid_attn_decode(const ha_params* p, const void* q, const void* ck, const void* cv,
                             int32_t n_cap, const int32_t* idx, const void* k_tok,
                             const void* v_tok, int32_t tok_cap, const int32_t* ctx_len,
                             void* o, float* lse, void* ws, size_t ws_bytes,
                             ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("hybrid_attn_decode");
  ha_status s = check_params(p, true, false);
  if (s != HA_OK) return s;
  if (idx) {
    s = check_k(p);
    if (s != HA_OK) return s;
  }
  HA_PTR(q);
  HA_PTR(ck);
  HA_PTR(cv);
  HA_OPT_PTR4(idx);
  // both per-token caches NULL: no window keys (a shard without the sequence's tail)
  const bool no_window = k_tok == nullptr && v_tok == nullptr;
  if (!no_window) {
    HA_PTR(k_tok);
    HA_PTR(v_tok);
    HA_REQUIRE(tok_cap >= p->n_win, HA_ERR_INVALID_ARG, "tok_cap = %d < n_win = %d", tok_cap,
               p->n_win);
  } else {
    tok_cap = 0;
  }
  HA_PTR4(ctx_len);
  HA_PTR(o);
  HA_OPT_PTR4(lse);
  HA_OPT_PTR(ws);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  const bool tc = ha::attention_tc_supported(*p, n_cap, tok_cap);
  const ha::AttnPlan pl = attention_plan(p, p->B, n_cap, tok_cap, idx != nullptr, true);
  const size_t need = attn_ws_bytes(p, pl, n_cap, idx != nullptr);
  HA_REQUIRE(ws_bytes >= need && (need == 0 || ws != nullptr), HA_ERR_WORKSPACE,
             "workspace %zu bytes < %zu", ws_bytes, need);
  cudaError_t e = kv8_view(p, pl, ck, cv, n_cap, idx, idx != nullptr, ctx_len, ws,
                           (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "decode: FP8 K/V widening launch");
  if (tc) {
    int* err = ha::device_error_word();
    HA_REQUIRE(err != nullptr, HA_ERR_CUDA, "device error word unavailable");
    return cuda_status(ha::launch_attention_tc(*p, pl, 1, 1, q, ctx_len, ck, cv, n_cap, idx, k_tok,
                                               v_tok, tok_cap, o, lse, ws, err,
                                               (cudaStream_t)stream),
                       "decode launch (tensor cores)");
  }
  return cuda_status(ha::launch_attention_simt(*p, pl, 1, 1, q, ctx_len, ck, cv, n_cap, idx, k_tok,
                                               v_tok, tok_cap, o, lse, ws, (cudaStream_t)stream),
                     "decode launch");
}

ha_status hybrid_attn_merge(const ha_params* p, int32_t rows, int32_t S, const float* o_part,
                            const float* lse_part, void* o, float* lse, ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("hybrid_attn_merge");
  ha_status s = check_params(p, true, false);
  if (s != HA_OK) return s;
  HA_REQUIRE(rows >= 1, HA_ERR_INVALID_ARG, "rows = %d", rows);
  HA_REQUIRE(S >= 1 && S <= 4096, HA_ERR_UNSUPPORTED, "S = %d (1..4096)", S);
  HA_PTR(o_part);
  HA_PTR4(lse_part);
  HA_PTR(o);
  HA_OPT_PTR4(lse);
  return cuda_status(ha::launch_attn_merge(*p, rows, S, o_part, lse_part, o, lse,
                                           (cudaStream_t)stream),
                     "merge launch");
}

ha_status hybrid_attn_prefill(const ha_params* p, const void* q, const int32_t* q_pos,
                              int32_t Tq, const void* ck, const void* cv, int32_t n_cap,
                              const int32_t* idx, const void* k_tok, const void* v_tok,
                              int32_t tok_cap, void* o, float* lse, void* ws, size_t ws_bytes,
                              ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("hybrid_attn_prefill");
  ha_status s = check_params(p, true, false);
  if (s != HA_OK) return s;
  if (idx) {
    s = check_k(p);
    if (s != HA_OK) return s;
  }
  HA_PTR(q);
  HA_PTR4(q_pos);
  HA_PTR(ck);
  HA_PTR(cv);
  HA_OPT_PTR4(idx);
  HA_PTR(k_tok);
  HA_PTR(v_tok);
  HA_PTR(o);
  HA_OPT_PTR4(lse);
  HA_OPT_PTR(ws);
  HA_REQUIRE(n_cap >= 1, HA_ERR_INVALID_ARG, "n_cap = %d", n_cap);
  HA_REQUIRE(Tq >= 1, HA_ERR_INVALID_ARG, "Tq = %d", Tq);
  HA_REQUIRE((long long)p->B * Tq <= 0x7fffffffLL, HA_ERR_UNSUPPORTED, "B * Tq too large");
  HA_REQUIRE(tok_cap >= p->n_win, HA_ERR_INVALID_ARG, "tok_cap = %d < n_win = %d", tok_cap,
             p->n_win);
  const bool tc = ha::attention_tc_supported(*p, n_cap, tok_cap);
  const ha::AttnPlan pl = attention_plan(p, p->B * Tq, n_cap, tok_cap, idx != nullptr, false);
  const size_t need = attn_ws_bytes(p, pl, n_cap, false);
  HA_REQUIRE(ws_bytes >= need && (need == 0 || ws != nullptr), HA_ERR_WORKSPACE,
             "workspace %zu bytes < %zu", ws_bytes, need);
  // FP8 K/V: every entry widened (each query has its own selection)
  cudaError_t e = kv8_view(p, pl, ck, cv, n_cap, idx, false, q_pos, ws, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_status(e, "prefill: FP8 K/V widening launch");
  if (tc) {
    int* err = ha::device_error_word();
    HA_REQUIRE(err != nullptr, HA_ERR_CUDA, "device error word unavailable");
    return cuda_status(ha::launch_attention_tc(*p, pl, 0, Tq, q, q_pos, ck, cv, n_cap, idx, k_tok,
                                               v_tok, tok_cap, o, lse, ws, err,
                                               (cudaStream_t)stream),
                       "prefill launch (tensor cores)");
  }
  return cuda_status(ha::launch_attention_simt(*p, pl, 0, Tq, q, q_pos, ck, cv, n_cap, idx, k_tok,
                                               v_tok, tok_cap, o, lse, ws, (cudaStream_t)stream),
                     "prefill launch");
}

ha_status csa_decode_step(const ha_params* p, const void* q, const void* q_idx,
                          const float* w_idx, const void* k_tok, const void* v_tok,
                          const void* ki_tok, const float* gate, int32_t tok_cap,
                          const int32_t* ctx_len, void* ck, void* cv, void* cki, int32_t n_cap,
                          void* scores, int32_t* idx, void* o, float* lse, void* ws,
                          size_t ws_bytes, ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("csa_decode_step");
  ha_status s = check_params(p, true, true);
  if (s != HA_OK) return s;
  s = check_k(p);
  if (s != HA_OK) return s;
  s = check_step(p, q, k_tok, v_tok, gate, tok_cap, ctx_len, ck, cv, n_cap, o, lse);
  if (s != HA_OK) return s;
  HA_PTR(q_idx);
  HA_PTR4(w_idx);
  HA_PTR(ki_tok);
  HA_PTR(cki);
  HA_PTR4(scores);
  HA_PTR4(idx);
  HA_OPT_PTR(ws);
  HA_REQUIRE(n_cap <= ha::topk_max_row_entries(), HA_ERR_UNSUPPORTED, "n_cap = %d > %d", n_cap,
             ha::topk_max_row_entries());
  const size_t topk_ws = round_up256(ha::topk_workspace_bytes(*p, 1, n_cap));
  const ha::AttnPlan pl = attention_plan(p, p->B, n_cap, tok_cap, true, true);
  const size_t need = topk_ws + attn_ws_bytes(p, pl, n_cap, true);
  HA_REQUIRE(ws_bytes >= need && (need == 0 || ws != nullptr), HA_ERR_WORKSPACE,
             "workspace %zu bytes < %zu", ws_bytes, need);
  int* err = ha::device_error_word();
  HA_REQUIRE(err != nullptr, HA_ERR_CUDA, "device error word unavailable");
  const cudaStream_t st = (cudaStream_t)stream;
  // Under the disjoint rule with n_win >= m the block the newest token completes
  // ends inside the query's window, so no stage of this step reads it: scoring
  // starts while it is compressed (the indexer waits for the compressor only
  // before it exits).  Otherwise the stages run strictly in order.
  const bool overlap = p->elig == HA_ELIG_DISJOINT && p->n_win >= p->m;
  ha::StepOpts sc;
  sc.ctx_len = ctx_len;
  const void* src[3] = {k_tok, v_tok, ki_tok};
  void* dst[3] = {ck, cv, cki};
  const int dims[3] = {p->d, p->d, p->d_I};
  cudaError_t e = ha::launch_compress(*p, 3, src, dst, dims, gate, nullptr, 1, tok_cap, n_cap, st, sc);
  if (e != cudaSuccess) return cuda_status(e, "step: compress launch");
  ha::StepOpts si;
  si.pos_off = -1;
  if (ha::index_scores_tc_supported(*p, q_idx, cki)) {
    si.wait_last = overlap ? 1 : 0;
    e = ha::launch_index_scores_tc(*p, q_idx, w_idx, cki, n_cap, ctx_len, 1, scores, err, st, si);
  } else {
    e = ha::launch_index_scores_simt(*p, q_idx, w_idx, cki, n_cap, ctx_len, 1,
                                     static_cast<float*>(scores), st, si);
  }
  if (e != cudaSuccess) return cuda_status(e, "step: index launch");
  ha::StepOpts sk;
  sk.pos_off = -1;
  e = ha::launch_topk(*p, scores, n_cap, ctx_len, 1, idx, ws, topk_ws, st, sk);
  if (e != cudaSuccess) return cuda_status(e, "step: top-k launch");
  void* attn_ws = need > topk_ws ? static_cast<char*>(ws) + topk_ws : nullptr;
  const void* ck_a = ck;
  const void* cv_a = cv;
  int n_cap_a = n_cap;
  const int32_t* idx_a = idx;
  e = kv8_view(p, pl, ck_a, cv_a, n_cap_a, idx_a, true, ctx_len, attn_ws, st);
  if (e != cudaSuccess) return cuda_status(e, "step: FP8 K/V widening launch");
  if (ha::attention_tc_supported(*p, n_cap, tok_cap)) {
    ha::StepOpts sa;
    sa.early = 1;
    e = ha::launch_attention_tc(*p, pl, 1, 1, q, ctx_len, ck_a, cv_a, n_cap_a, idx_a, k_tok, v_tok,
                                tok_cap, o, lse, attn_ws, err, st, sa);
  } else {
    e = ha::launch_attention_simt(*p, pl, 1, 1, q, ctx_len, ck_a, cv_a, n_cap_a, idx_a, k_tok,
                                  v_tok, tok_cap, o, lse, attn_ws, st);
  }
  return cuda_status(e, "step: attention launch");
}

ha_status hca_decode_step(const ha_params* p, const void* q, const void* k_tok, const void* v_tok,
                          const float* gate, int32_t tok_cap, const int32_t* ctx_len, void* ck,
                          void* cv, int32_t n_cap, void* o, float* lse, void* ws, size_t ws_bytes,
                          ha_stream_t stream) {
  g_last_error[0] = 0;
  CallRange range("hca_decode_step");
  ha_status s = check_params(p, true, false);
  if (s != HA_OK) return s;
  s = check_step(p, q, k_tok, v_tok, gate, tok_cap, ctx_len, ck, cv, n_cap, o, lse);
  if (s != HA_OK) return s;
  HA_OPT_PTR(ws);
  const ha::AttnPlan pl = attention_plan(p, p->B, n_cap, tok_cap, false, true);
  const size_t need = attn_ws_bytes(p, pl, n_cap, false);
  HA_REQUIRE(ws_bytes >= need && (need == 0 || ws != nullptr), HA_ERR_WORKSPACE,
             "workspace %zu bytes < %zu", ws_bytes, need);
  const cudaStream_t st = (cudaStream_t)stream;
  // As in csa_decode_step: under the disjoint rule with n_win >= m the attention
  // reads no entry the compressor writes, so it runs beside the compression and
  // waits for it only before it exits.  (Launching the attention first and the
  // compressor beside it on the SMs it leaves was measured slower.)
  const bool overlap = p->elig == HA_ELIG_DISJOINT && p->n_win >= p->m;
  ha::StepOpts sc;
  sc.ctx_len = ctx_len;
  const void* src[2] = {k_tok, v_tok};
  void* dst[2] = {ck, cv};
  const int dims[2] = {p->d, p->d};
  cudaError_t e = ha::launch_compress(*p, 2, src, dst, dims, gate, nullptr, 1, tok_cap, n_cap, st, sc);
  if (e != cudaSuccess) return cuda_status(e, "step: compress launch");
  // FP8 K/V: the widening (which waits for the compressor) comes first, and the
  // attention, reading the widened rows, then waits for it as usual
  const void* ck_a = ck;
  const void* cv_a = cv;
  int n_cap_a = n_cap;
  const int32_t* no_idx = nullptr;
  e = kv8_view(p, pl, ck_a, cv_a, n_cap_a, no_idx, false, ctx_len, ws, st);
  if (e != cudaSuccess) return cuda_status(e, "step: FP8 K/V widening launch");
  if (ha::attention_tc_supported(*p, n_cap, tok_cap)) {
    int* err = ha::device_error_word();
    HA_REQUIRE(err != nullptr, HA_ERR_CUDA, "device error word unavailable");
    ha::StepOpts sa;
    sa.wait_last = overlap && !(p->fmt & HA_FMT_KV8) ? 1 : 0;
    e = ha::launch_attention_tc(*p, pl, 1, 1, q, ctx_len, ck_a, cv_a, n_cap_a, nullptr, k_tok,
                                v_tok, tok_cap, o, lse, ws, err, st, sa);
  } else {
    e = ha::launch_attention_simt(*p, pl, 1, 1, q, ctx_len, ck_a, cv_a, n_cap_a, nullptr, k_tok,
                                  v_tok, tok_cap, o, lse, ws, st);
  }
  return cuda_status(e, "step: attention launch");
}

ha_status ha_workspace_size(const ha_params* p, int32_t op, int32_t Tq, int32_t n_cap,
                            int32_t is_csa, size_t* bytes) {
  g_last_error[0] = 0;
  HA_REQUIRE(bytes != nullptr, HA_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;
  ha_status s = check_params(p, op != HA_OP_TOPK, false);
  if (s != HA_OK) return s;
  HA_REQUIRE(Tq >= 1 && n_cap >= 1, HA_ERR_INVALID_ARG, "Tq = %d, n_cap = %d", Tq, n_cap);
  switch (op) {
    case HA_OP_TOPK: *bytes = ha::topk_workspace_bytes(*p, Tq, n_cap); return HA_OK;
    case HA_OP_DECODE:
      *bytes = attn_ws_bytes(p, attention_plan(p, p->B, n_cap, 0, is_csa != 0, true), n_cap,
                             is_csa != 0);
      return HA_OK;
    case HA_OP_PREFILL:
      *bytes = attn_ws_bytes(p, attention_plan(p, p->B * Tq, n_cap, 0, is_csa != 0, false), n_cap,
                             false);
      return HA_OK;
    case HA_OP_DECODE_STEP:
      *bytes = step_workspace_bytes(p, n_cap, 0, is_csa != 0);
      return HA_OK;
  }
  return fail(HA_ERR_INVALID_ARG, "op = %d", op);
}

}  // extern "C"
