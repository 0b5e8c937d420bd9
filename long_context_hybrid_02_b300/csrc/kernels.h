// Internal launchers of the CUDA library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "hybrid_attn.h"

namespace ha {

// How a kernel of a fused decode step (csa_decode_step / hca_decode_step) is tied
// to the previous kernel of the stream; the defaults are the stand-alone calls.
struct StepOpts {
  int pos_off = 0;                   // query position = pos + pos_off (-1: pos is ctx_len)
  int wait_last = 0;                 // reads nothing the previous kernel writes: release
                                     // the next kernel at once, wait only before exiting
  int early = 0;                     // attention: q and the positions are read before the
                                     // wait (they are inputs of the step, final by then)
  const int32_t* ctx_len = nullptr;  // compressor: compress the block the newest token
                                     // completes (block ctx_len/m - 1 when ctx_len % m == 0)
};

// api.cu: replace the message returned by ha_last_error() on this thread.
void set_last_error(const char* msg);

// api.cu: workspace bytes hybrid_attn_decode needs for these arguments (the same
// plan the call itself makes, tok_cap included); p must have passed the checks of
// ha_workspace_size.
size_t decode_workspace_bytes(const ha_params* p, int n_cap, int tok_cap, bool is_csa);

// status.cu: device address of the error word of the tensor-core kernels on the
// current device (null if it cannot be looked up).
int* device_error_word();

// compress.cu: n_tensors row tensors compressed with the same gates.
cudaError_t launch_compress(const ha_params& p, int n_tensors, const void* const* src,
                            void* const* dst, const int* dims, const float* gate,
                            const int32_t* blk_begin, int n_blk, int tok_cap, int n_cap,
                            cudaStream_t st, const StepOpts& so = StepOpts());

// indexer.cu: CUDA-core indexer for every shape and type.
cudaError_t launch_index_scores_simt(const ha_params& p, const void* q_idx, const float* w_idx,
                                     const void* cki, int n_cap, const int32_t* q_pos, int Tq,
                                     float* scores, cudaStream_t st,
                                     const StepOpts& so = StepOpts());

// indexer_tc.cu: tcgen05 indexer for bf16, H_I = 64, d_I = 128.
bool index_scores_tc_supported(const ha_params& p, const void* q_idx, const void* cki);
// Scores are float32, or bfloat16 when p.fmt has HA_FMT_IDX4 (the FP4 indexer).
cudaError_t launch_index_scores_tc(const ha_params& p, const void* q_idx, const float* w_idx,
                                   const void* cki, int n_cap, const int32_t* q_pos, int Tq,
                                   void* scores, int* err, cudaStream_t st,
                                   const StepOpts& so = StepOpts());

// topk.cu
size_t topk_workspace_bytes(const ha_params& p, int Tq, int n_cap);
int topk_max_row_entries();       // longest score row csa_topk supports
cudaError_t launch_topk(const ha_params& p, const void* scores, int n_cap, const int32_t* q_pos,
                        int Tq, int32_t* idx, void* ws, size_t ws_bytes, cudaStream_t st,
                        const StepOpts& so = StepOpts());

// attention.cu: split-KV CUDA-core attention (decode and prefill) + merge.
struct AttnPlan {
  int n_splits;        // key-list ranges per query row (and 64-head group, tensor cores)
  int keys_per_split;  // multiple of 32 (CUDA cores) / 16 (tensor cores)
  int tile;            // keys staged per shared-memory tile
  size_t ws_bytes;     // float32 partials when n_splits > 1
};
AttnPlan plan_attention_simt(const ha_params& p, int rows, int max_keys, bool decode);
cudaError_t launch_attention_simt(const ha_params& p, const AttnPlan& pl, int decode, int Tq,
                                  const void* q, const int32_t* pos, const void* ck,
                                  const void* cv, int n_cap, const int32_t* idx,
                                  const void* k_tok, const void* v_tok, int tok_cap, void* o,
                                  float* lse, void* ws, cudaStream_t st);
// o = merge of the S float32 partials [rows, S, H, d] + lse [rows, S, H], in split order.
cudaError_t launch_attn_merge(const ha_params& p, int rows, int S, const float* o_part,
                              const float* lse_part, void* o, float* lse, cudaStream_t st);

// kv8.cu: the FP8 KV rows (608 bytes) an attention call reads, widened to bfloat16
// rows in the workspace.  With idx (a decode selection, [B, k]) the valid selected
// entries are packed to the front of a [B, k] list and out->idx = 0, 1, .., -1;
// without, every entry of the cache [B, n_cap] is widened and out->idx is null.
struct KvExpanded {
  const void* ck;
  const void* cv;
  int n_cap;
  const int32_t* idx;
};
size_t kv8_expand_bytes(const ha_params& p, int n_cap, bool select);
cudaError_t launch_kv8_expand(const ha_params& p, const void* ck8, const void* cv8, int n_cap,
                              const int32_t* idx, const int32_t* ctx_len, void* ws,
                              KvExpanded* out, cudaStream_t st);

// attention_tc.cu: tcgen05 attention for bf16, d = 512, H a multiple of 64 (decode
// rows and prefill rows alike; each row has its own key list).
bool attention_tc_supported(const ha_params& p, int n_cap, int tok_cap);
AttnPlan plan_attention_tc(const ha_params& p, int rows, int max_keys);
cudaError_t launch_attention_tc(const ha_params& p, const AttnPlan& pl, int decode, int Tq,
                                const void* q, const int32_t* pos, const void* ck, const void* cv,
                                int n_cap, const int32_t* idx, const void* k_tok,
                                const void* v_tok, int tok_cap, void* o, float* lse, void* ws,
                                int* err, cudaStream_t st, const StepOpts& so = StepOpts());

}  // namespace ha
