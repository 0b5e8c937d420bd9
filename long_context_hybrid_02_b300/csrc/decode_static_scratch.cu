// hybrid_attn_decode_static: the decode attention call for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: plugins of an
// inference engine that only receive the input and output pointers of a layer,
// code that runs inside another runtime's memory pool where a raw cudaMalloc
// would bypass (and fragment) that pool, and latency-bound serving loops where
// cudaMalloc/cudaFree would synchronise the device.  This entry point needs no
// workspace argument: the split-KV partials live in a fixed array in device
// global memory that belongs to this file.  The array is kStaticScratchBytes
// (32 MiB) and every GPU that loads the library keeps it until the process
// exits.  Decode problems whose partials do not fit are rejected with
// HA_ERR_WORKSPACE before anything is launched.
//
// The array is shared by every call on a device and keeps whatever the last
// call wrote.  Nothing in it has to start at zero: every split writes its whole
// partial before the merge reads it.  Two calls whose kernels overlap on the GPU
// (different streams without ordering, or different host threads) race on the
// array and give wrong results; order them on one stream.
//
// The first call on each device looks up the device address of the array
// (cudaGetSymbolAddress, with that device current) and caches it; make that
// first call before any stream capture that records this entry point.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "hybrid_attn.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

ha_status hybrid_attn_decode_static(const ha_params* p, const void* q, const void* ck,
                                    const void* cv, int32_t n_cap, const int32_t* idx,
                                    const void* k_tok, const void* v_tok, int32_t tok_cap,
                                    const int32_t* ctx_len, void* o, float* lse,
                                    ha_stream_t stream) {
  // ha_workspace_size checks the parameters; the size itself comes from the plan
  // hybrid_attn_decode makes for these very arguments (tok_cap can change it)
  size_t need = 0;
  ha_status s = ha_workspace_size(p, HA_OP_DECODE, 1, n_cap, idx != nullptr ? 1 : 0, &need);
  if (s != HA_OK) return s;
  need = ha::decode_workspace_bytes(p, n_cap, tok_cap, idx != nullptr);
  char msg[256];
  if (need > kStaticScratchBytes) {
    snprintf(msg, sizeof(msg),
             "hybrid_attn_decode_static: this problem needs %zu bytes of scratch, the static "
             "scratch holds %zu; call hybrid_attn_decode with a caller-allocated workspace",
             need, kStaticScratchBytes);
    ha::set_last_error(msg);
    return HA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "hybrid_attn_decode_static: cudaGetSymbolAddress failed: %s",
             cudaGetErrorString(e));
    ha::set_last_error(msg);
    return HA_ERR_CUDA;
  }
  return hybrid_attn_decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, ctx_len, o, lse,
                            scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
