/*
 * hybrid_attn.h -- C ABI of libhybridattn.so: the hot path of hybrid long-context
 * attention (sliding window + compressed sparse attention, or sliding window +
 * heavily compressed attention) for one NVIDIA B300 (sm_103a).
 *
 * Sources (web pages about DeepSeek-V4; they give the data flow and the
 * constants, not the formulas):
 *   [V4-notes] "DeepSeek-V4 深度研究剖析" (group-reading-wiki, DeepSeek-V4 research notes):
 *              §5.2 SWA keeps the last n_win = 128 uncompressed KV; §5.3 CSA
 *              compresses every m = 4 tokens' KV into one entry, a Lightning
 *              Indexer scores the entries and the top-k (512 / 1024) are attended;
 *              §5.4 HCA compresses every m' = 128 tokens into one entry and attends
 *              to all of them; §11.4 the cache kinds (compressed KV, indexer KV,
 *              window state, tail tokens of unfinished blocks).
 *   [LateTalk] "163: DeepSeek V4 Explained ..." (zjai.club) §14: every layer is the
 *              window plus one of CSA / HCA, fixed per layer, on one shared
 *              (MQA-style) KV head.
 *   [EP95]     "EP 95 解读 DeepSeek-V4 论文" (aifrontier.kr), the Lightning Indexer /
 *              top-k segment and the attention-block figure (window keys and
 *              compressed entries concatenated before one MQA).
 * Formulas the pages leave open and this library fixes:
 *   compressor  C_j = sum_{i<m} alpha_i X[j*m+i], alpha = softmax(gate[j*m .. j*m+m-1])
 *   indexer     s_{t,j} = sum_h w_{t,h} * max(0, qI_{t,h} . CI_j)
 *   eligibility n_elig(t) = floor(max(0, t+1-n_win)/m)   (HA_ELIG_DISJOINT, default)
 *               n_elig(t) = floor((t+1)/m)               (HA_ELIG_OVERLAP)
 *   attention   one softmax over {selected (CSA) or all eligible (HCA) entries}
 *               plus the window positions max(0,t-n_win+1) .. t, scale 1/sqrt(d).
 *
 * Conventions shared by every call
 *   - Every pointer argument except `p` is DEVICE memory owned by the caller.
 *     The library allocates nothing and never synchronises the host (except
 *     ha_device_error, which reads a device word); all work is ordered on
 *     `stream` (0 = legacy default).  Nothing carries from one call to the next
 *     but the device error word (ha_device_error) and the fixed scratch of
 *     hybrid_attn_decode_static.
 *   - Arrays are row-major with the last dimension contiguous.  "T" is the
 *     storage type selected by p->dtype (float for HA_F32, bfloat16 for
 *     HA_BF16).  Gates, indexer weights, scores and lse are always float32;
 *     indices and positions are int32.
 *   - Per-token caches are [B, tok_cap, dim]; token position u of sequence b is
 *     at slot (u % tok_cap).  tok_cap = context length gives a flat cache, a
 *     smaller tok_cap a ring (the caller keeps the window and the tail tokens of
 *     blocks not yet compressed resident).
 *   - Compressed caches are [B, n_cap, dim]; entry j of sequence b is at row j.
 *   - T arrays and workspaces must be 16-byte aligned; float32 / int32 arrays
 *     4-byte aligned; d and d_I multiples of 8 (HA_ERR_MISALIGNED /
 *     HA_ERR_UNSUPPORTED otherwise).
 *   - Arguments are checked on the host before any launch; on error nothing is
 *     launched and ha_last_error() describes the failure.  A failed launch
 *     returns HA_ERR_CUDA.  Faults of the caller's memory surface at the
 *     caller's next synchronisation.  Nothing aborts or throws across the ABI.
 *   - Results are deterministic: fixed reduction orders, no atomics on data.
 *   - Device-side positions (blk_begin, q_pos, ctx_len, idx) are range-checked by
 *     the kernels: a block or entry outside [0, n_cap) is skipped, never read or
 *     written.
 */
#ifndef HYBRID_ATTN_H_
#define HYBRID_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ha_stream_t; /* same handle as cudaStream_t */

typedef enum {
  HA_OK = 0,
  HA_ERR_INVALID_ARG = 1, /* a size or pointer is out of range / NULL        */
  HA_ERR_MISALIGNED = 2,  /* a pointer breaks its alignment rule (16 / 4 B)  */
  HA_ERR_UNSUPPORTED = 3, /* a shape outside the limits below                */
  HA_ERR_WORKSPACE = 4,   /* ws is NULL or smaller than ha_workspace_size()  */
  HA_ERR_CUDA = 5         /* a CUDA runtime call or a launch failed          */
} ha_status;

typedef enum { HA_F32 = 0, HA_BF16 = 1 } ha_dtype;

/* Storage formats of the deployed model ([V4-notes] §8), bit flags of
 * ha_params.fmt; both need dtype HA_BF16.
 *   HA_FMT_KV8: the compressed K/V caches keep their RoPE dims in BF16 and the
 *     other dims in FP8.  With d = 512 a row of ck or cv is 608 bytes: dims
 *     0..63 as bfloat16, dims 64..511 as e4m3fn codes, one float32 scale per 64
 *     dims (7), 4 unused bytes; element value = code * scale, scale = amax / 448
 *     of its group, code = e4m3(x / scale) nearest even, the divisions in
 *     float32 (an all-zero group has scale 0 and codes 0).  ck and cv are then
 *     [B, n_cap, 608] bytes; the per-token caches stay bfloat16.  The attention
 *     calls widen the rows they read to bfloat16 (code * scale rounded to nearest
 *     even) in their workspace first.  Needs d = 512.
 *   HA_FMT_IDX4: the Lightning Indexer computes in FP4 and keeps its scores in
 *     BF16.  Compressed indexer keys (cki) are rows of 80 bytes: d_I = 128
 *     e2m1 codes, two per byte (element 2i in the low nibble), then 8 e4m3fn
 *     scales (one per 16 consecutive elements), then 8 unused bytes; element
 *     value = code * scale.  scale = e4m3(amax / 6) of its 16 elements, code =
 *     e2m1(x / scale), both rounded to nearest even (codes saturate at 6), the
 *     divisions in float32; an all-zero group has scale 0 and codes 0.  The
 *     indexer's queries (q_idx, still given in bfloat16) are quantized the
 *     same way inside the indexer.  Index scores are bfloat16 (the float32 sum
 *     rounded to nearest even): csa_index_scores writes them and csa_topk reads
 *     them.  Needs H_I = 64 and d_I = 128. */
enum { HA_FMT_KV8 = 1, HA_FMT_IDX4 = 2 };
typedef enum { HA_ELIG_DISJOINT = 0, HA_ELIG_OVERLAP = 1 } ha_elig;
typedef enum { HA_OP_TOPK = 0, HA_OP_DECODE = 1, HA_OP_PREFILL = 2, HA_OP_DECODE_STEP = 3 } ha_op;

/* Layer description.  Limits: 1 <= B; 1 <= H <= 256; 8 <= d <= 1024, d % 8 == 0;
 * 1 <= n_win <= 65536; 1 <= m <= 1024; 1 <= k <= 4096 (CSA); 1 <= H_I <= 128;
 * 8 <= d_I <= 512, d_I % 8 == 0.  scale <= 0 selects 1/sqrt(d). */
typedef struct {
  int32_t B;     /* sequences in the batch                                   */
  int32_t H;     /* query heads sharing the single K/V head                  */
  int32_t d;     /* head dim of q, K, V and of the compressed entries        */
  int32_t n_win; /* sliding-window length ([V4-notes] §5.2: 128)             */
  int32_t m;     /* tokens per compressed entry (CSA 4, HCA 128)             */
  int32_t k;     /* entries selected per query (CSA; 512 / 1024)             */
  int32_t H_I;   /* indexer heads                                            */
  int32_t d_I;   /* indexer head dim (also the indexer-key dim)              */
  int32_t dtype; /* ha_dtype of every T array                                */
  int32_t elig;  /* ha_elig                                                  */
  float scale;   /* softmax scale of the attention                           */
  int32_t fmt;   /* storage-format bits (HA_FMT_*), 0 = plain dtype storage  */
} ha_params;

/* ---------------------------------------------------------------------------
 * hca_compress_kv -- HCA token compressor ([V4-notes] §5.4: every m' = 128
 * tokens' KV becomes one entry; formula: per-block softmax-gated sum).
 *   k_tok, v_tok : T [B, tok_cap, d]      per-token K and V
 *   gate         : float [B, tok_cap]     one gate logit per token
 *   blk_begin    : int32 [B]              first block to compress per sequence
 *                                         (negative: none of its blocks)
 *   n_blk        : blocks per sequence (>= 0; 0 is a no-op)
 *   ck, cv       : T [B, n_cap, d]        rows blk_begin[b] .. +n_blk-1 written
 * Block j reads positions j*m .. j*m+m-1 (the caller guarantees they are
 * resident in the per-token cache).  Only K and V; p->m is the block size.
 * ------------------------------------------------------------------------- */
ha_status hca_compress_kv(const ha_params* p, const void* k_tok, const void* v_tok,
                          const float* gate, int32_t tok_cap, const int32_t* blk_begin,
                          int32_t n_blk, void* ck, void* cv, int32_t n_cap,
                          ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_compress_kv -- CSA token compressor ([V4-notes] §5.3: every m = 4 tokens'
 * KV becomes one entry; §11.4: the indexer keys are a compressed cache of their
 * own).  As hca_compress_kv, plus the indexer keys, compressed with the same
 * gates:
 *   ki_tok : T [B, tok_cap, d_I]   cki : T [B, n_cap, d_I]
 * Under HA_FMT_IDX4 cki holds the 80-byte FP4 rows [B, n_cap, 80] of the
 * compressed indexer keys (m <= 16).
 * ------------------------------------------------------------------------- */
ha_status csa_compress_kv(const ha_params* p, const void* k_tok, const void* v_tok,
                          const void* ki_tok, const float* gate, int32_t tok_cap,
                          const int32_t* blk_begin, int32_t n_blk, void* ck, void* cv,
                          void* cki, int32_t n_cap, ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_index_scores -- Lightning Indexer ([V4-notes] §5.3; [EP95]: it scores
 * every compressed entry, so it must be light):
 *   s[b,t,j] = sum_h w[b,t,h] * max(0, q_idx[b,t,h,:] . cki[b,j,:])
 *   q_idx  : T [B, Tq, H_I, d_I]      w_idx : float [B, Tq, H_I]
 *   cki    : T [B, n_cap, d_I]        q_pos : int32 [B, Tq] absolute positions
 *   scores : float [B, Tq, n_cap]     written for j < min(n_elig(q_pos), n_cap)
 *            only; the rest of each row is left untouched.  bfloat16 [B, Tq,
 *            n_cap] under HA_FMT_IDX4, where cki holds 80-byte FP4 rows
 *            [B, n_cap, 80] and q_idx is quantized to FP4 inside the call.
 * ------------------------------------------------------------------------- */
ha_status csa_index_scores(const ha_params* p, const void* q_idx, const float* w_idx,
                           const void* cki, int32_t n_cap, const int32_t* q_pos, int32_t Tq,
                           void* scores, ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_topk -- top-k selection of compressed entries ([V4-notes] §5.3: k = 512
 * for V4-Flash, 1024 for V4-Pro).  Per row (b, t) over the n = min(n_elig(t),
 * n_cap) eligible scores: the k best by (score descending, index ascending),
 * NaN ranked as -inf; all n when n <= k.  scores as written by csa_index_scores
 * (float32, or bfloat16 under HA_FMT_IDX4).  Written in ascending index order,
 * padded with -1:
 *   idx : int32 [B, Tq, k]
 *   ws  : device workspace of ha_workspace_size(p, HA_OP_TOPK, Tq, n_cap) bytes
 *         (0 bytes, ws may be NULL, for n_cap <= 40,960; longer rows are cut
 *         into segments whose candidate lists go through ws).
 * n_cap above 41,943,040 (= 40,960 x 1,024) returns HA_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
ha_status csa_topk(const ha_params* p, const void* scores, int32_t n_cap,
                   const int32_t* q_pos, int32_t Tq, int32_t* idx, void* ws, size_t ws_bytes,
                   ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * hybrid_attn_decode -- one decode query per sequence at t = ctx_len[b]-1
 * ([V4-notes] §5.2-§5.5; [EP95] figure: window and compressed entries in one
 * MQA softmax).
 *   q          : T [B, H, d]
 *   ck, cv     : T [B, n_cap, d]       compressed K / V
 *   idx        : int32 [B, k]  CSA: attended entries (any order; entries < 0 or
 *                >= min(n_elig(t), n_cap) are ignored)
 *                NULL         HCA: every entry j < min(n_elig(t), n_cap)
 *   k_tok,v_tok: T [B, tok_cap, d]     window source, tok_cap >= n_win; both
 *                NULL: no window keys (a shard of a sequence that does not hold the
 *                sequence's tail; tok_cap is then ignored)
 *   ctx_len    : int32 [B]   context length including the query token;
 *                <= 0 gives o = 0, lse = -inf for that sequence
 *   o          : T [B, H, d]           lse : float [B, H] or NULL
 *   ws         : ha_workspace_size(p, HA_OP_DECODE, 1, n_cap) bytes (split
 *                partials: when the sequences are too few to fill the GPU, each
 *                key list is cut into splits whose float32 results (o and lse)
 *                go through ws and are merged in split order by a second
 *                launch; 0 bytes, ws may be NULL, when there is one split).
 * ------------------------------------------------------------------------- */
ha_status hybrid_attn_decode(const ha_params* p, const void* q, const void* ck, const void* cv,
                             int32_t n_cap, const int32_t* idx, const void* k_tok,
                             const void* v_tok, int32_t tok_cap, const int32_t* ctx_len,
                             void* o, float* lse, void* ws, size_t ws_bytes,
                             ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * hybrid_attn_merge -- combine attention results over disjoint key sets into the
 * result over their union ([EP95] figure: one softmax over all keys; this is that
 * softmax assembled from parts, e.g. from the shards of a sequence whose
 * compressed entries are spread over several GPUs).  Per row and head:
 *   LSE = log sum_s exp(lse_s),  o = sum_s exp(lse_s - LSE) o_s,
 * parts with lse_s = -inf carry no weight; no part with a key gives o = 0,
 * LSE = -inf.  The parts are added in part order (deterministic).
 *   o_part : float [rows, S, H, d]     lse_part : float [rows, S, H]
 *   o      : T [rows, H, d]            lse : float [rows, H] or NULL
 * p supplies H, d and the type of o; 1 <= S <= 4096.
 * ------------------------------------------------------------------------- */
ha_status hybrid_attn_merge(const ha_params* p, int32_t rows, int32_t S, const float* o_part,
                            const float* lse_part, void* o, float* lse, ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * hybrid_attn_prefill -- Tq queries per sequence at absolute positions q_pos,
 * each with its own selected set and its own causal window (the chunk's own
 * tokens must already be in the per-token cache).  Same definitions as decode:
 *   q   : T [B, Tq, H, d]        q_pos : int32 [B, Tq]
 *   idx : int32 [B, Tq, k] (CSA) or NULL (HCA)
 *   o   : T [B, Tq, H, d]        lse   : float [B, Tq, H] or NULL
 *   ws  : ha_workspace_size(p, HA_OP_PREFILL, Tq, n_cap) bytes
 * ------------------------------------------------------------------------- */
ha_status hybrid_attn_prefill(const ha_params* p, const void* q, const int32_t* q_pos,
                              int32_t Tq, const void* ck, const void* cv, int32_t n_cap,
                              const int32_t* idx, const void* k_tok, const void* v_tok,
                              int32_t tok_cap, void* o, float* lse, void* ws, size_t ws_bytes,
                              ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * csa_decode_step -- one decode token per sequence through a whole SWA + CSA
 * layer in one call, in the pages' order ([V4-notes] §5.3: compress, score every
 * compressed entry with the Lightning Indexer, select the top k, attend to them
 * and to the window; §11.4: the tail tokens of an unfinished block stay in the
 * per-token cache until the block completes):
 *   1. if the newest token completes a block (ctx_len % m == 0), that block,
 *      (ctx_len / m) - 1, is compressed into ck, cv, cki;
 *   2. csa_index_scores, 3. csa_topk and 4. hybrid_attn_decode for the query at
 *      t = ctx_len - 1.
 * The results are those of the four calls issued in that order (the same
 * kernels): scores, idx, o and lse as documented there.  The caller writes the
 * newest token's rows (k_tok, v_tok, ki_tok, gate at slot (ctx_len-1) % tok_cap)
 * before the call.  The kernels are chained with programmatic dependent launch;
 * under the disjoint rule with n_win >= m no stage reads the block the step
 * compresses, so scoring runs beside the compression and the attention requests
 * q before the selection is final.
 *   q      : T [B, H, d]         q_idx : T [B, H_I, d_I]     w_idx : float [B, H_I]
 *   k_tok, v_tok : T [B, tok_cap, d]    ki_tok : T [B, tok_cap, d_I]
 *   gate   : float [B, tok_cap]  ctx_len : int32 [B]  (tok_cap >= max(n_win, m))
 *   ck, cv : T [B, n_cap, d]     cki : T [B, n_cap, d_I]
 *   scores : float [B, n_cap] (bfloat16 under HA_FMT_IDX4)    idx : int32 [B, k]
 *   o      : T [B, H, d]         lse : float [B, H] or NULL
 *   ws     : ha_workspace_size(p, HA_OP_DECODE_STEP, 1, n_cap, 1) bytes
 * ------------------------------------------------------------------------- */
ha_status csa_decode_step(const ha_params* p, const void* q, const void* q_idx,
                          const float* w_idx, const void* k_tok, const void* v_tok,
                          const void* ki_tok, const float* gate, int32_t tok_cap,
                          const int32_t* ctx_len, void* ck, void* cv, void* cki, int32_t n_cap,
                          void* scores, int32_t* idx, void* o, float* lse, void* ws,
                          size_t ws_bytes, ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * hca_decode_step -- one decode token per sequence through a whole SWA + HCA
 * layer ([V4-notes] §5.4): the block completed by the newest token (if any) is
 * compressed into ck, cv, then hybrid_attn_decode attends to every eligible
 * entry and the window.  Arguments as csa_decode_step; ws is
 * ha_workspace_size(p, HA_OP_DECODE_STEP, 1, n_cap, 0) bytes.  Under the disjoint
 * rule with n_win >= m the attention runs beside the compression.
 * ------------------------------------------------------------------------- */
ha_status hca_decode_step(const ha_params* p, const void* q, const void* k_tok, const void* v_tok,
                          const float* gate, int32_t tok_cap, const int32_t* ctx_len, void* ck,
                          void* cv, int32_t n_cap, void* o, float* lse, void* ws, size_t ws_bytes,
                          ha_stream_t stream);

/* ---------------------------------------------------------------------------
 * hybrid_attn_decode_static -- hybrid_attn_decode without a workspace argument,
 * for callers that cannot allocate device memory (an engine plugin that only
 * gets its layer's input and output pointers, code living in another runtime's
 * memory pool, serving loops that must not call cudaMalloc because it
 * synchronises the device).  The pages have no counterpart: this is a calling
 * convention of this library, not part of the method.
 * Same arguments, results and checks as hybrid_attn_decode.  The split-KV
 * partials go to a fixed 32 MiB array in device global memory owned by the
 * library; each device that loads the library holds that array until the
 * process exits.  Problems whose partials need more than 32 MiB (the workspace
 * hybrid_attn_decode would need for the same arguments, tok_cap included; this is
 * ha_workspace_size(p, HA_OP_DECODE, 1, n_cap, idx != NULL) unless B * tok_cap
 * reaches 2^30) return HA_ERR_WORKSPACE without launching, with a message naming
 * the static scratch.  Allocates nothing.
 * Every call on a device shares the array and leaves its last contents behind
 * (no part of it needs to start at zero); calls whose kernels overlap on the GPU
 * race on it, so order them on one stream.  The first call on a device looks up
 * the array's device address once (with that device current); make that first
 * call before any stream capture that records this entry point.
 * ------------------------------------------------------------------------- */
ha_status hybrid_attn_decode_static(const ha_params* p, const void* q, const void* ck,
                                    const void* cv, int32_t n_cap, const int32_t* idx,
                                    const void* k_tok, const void* v_tok, int32_t tok_cap,
                                    const int32_t* ctx_len, void* o, float* lse,
                                    ha_stream_t stream);

/* Workspace bytes for `op` (ha_op) with Tq queries per sequence and n_cap
 * compressed entries; `is_csa` = idx will be non-NULL (decode / prefill). */
ha_status ha_workspace_size(const ha_params* p, int32_t op, int32_t Tq, int32_t n_cap,
                            int32_t is_csa, size_t* bytes);

/* First error code recorded on the current device by a tensor-core kernel whose
 * pipeline wait ran out of time (0 = none); such a kernel returns early instead
 * of hanging and its outputs are incomplete.  While a code is set, a wait of a
 * later tensor-core kernel that would block gives up at once, so the outputs of
 * later calls are incomplete too until the code is cleared.  Blocks until the
 * device's prior work is done.  `clear` != 0 resets the code. */
ha_status ha_device_error(int32_t* code, int32_t clear);

/* Test of the error path above without a fault: launches on `stream` one CTA
 * that waits on a barrier nothing arrives at, through the same bounded wait as
 * the tensor-core pipelines; after the wait limit (2 s) it records `code` (> 0)
 * in the device error word, unless a code is already set, and returns.  Not part
 * of the method; the device stays usable.  HA_ERR_INVALID_ARG for code <= 0. */
ha_status ha_selftest_wait_timeout(int32_t code, ha_stream_t stream);

/* Static description of a status code. */
const char* ha_status_string(ha_status s);

/* Detail of the last failed call on this host thread ("" if none). */
const char* ha_last_error(void);

/* ABI version of this header (bumped on any signature change). */
int32_t ha_abi_version(void);

/* Kernel launches issued by this library in this process so far (accounting;
 * launches recorded into a CUDA graph count once, at capture). */
uint64_t ha_launch_count(void);

/* Page-locked host memory for staging a step's inputs and outputs (not part of
 * the method): `bytes` (> 0) bytes from cudaHostAlloc, owned by the caller and
 * released with ha_host_free.  write_combined != 0 asks for write-combined memory
 * (fast host writes and device reads; host reads are slow: use it for inputs
 * only).  Copies from this memory to the device reach the link's bandwidth,
 * which memory registered after allocation may not.  Returns NULL on failure
 * (ha_last_error says why). */
void* ha_host_alloc(size_t bytes, int32_t write_combined);

/* Release memory from ha_host_alloc (NULL is a no-op).  HA_ERR_CUDA when the
 * runtime refuses. */
ha_status ha_host_free(void* p);

#ifdef __cplusplus
}
#endif
#endif /* HYBRID_ATTN_H_ */
