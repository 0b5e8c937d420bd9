// Joint attention of 64-head query groups over the selected (CSA) or all eligible
// (HCA) compressed entries plus the uncompressed window, on the tcgen05 tensor
// cores ("DeepSeek-V4 深度研究剖析" §5.2 SWA, §5.3 CSA, §5.4 HCA; "EP 95 解读
// DeepSeek-V4 论文": window keys and compressed entries are concatenated before
// one multi-query attention, so they share one softmax).  bfloat16 storage,
// head dim 512, H a multiple of 64; fp32 accumulation.
//
// One shared K/V head serves every query head (MQA), so for one query row the
// scores of a 64-head group are a GEMM with the keys as the M dimension:
//   S^T[key, h] = sum_c K[key, c] q[h, c]            (M = 128 keys, N = 64, K = 512)
//   O^T[c, h]  += sum_key V[key, c] P[key, h]         (M = 128 dims x 4, N = 64, K = 128)
// Both MMAs read 128-byte-swizzled shared-memory tiles: K and q are K-major, V
// and P are MN-major (the row of 64 dims / 64 heads is contiguous), so the very
// same gathered key rows serve as the A operand of both products.
//
// Work item = (query row, 64-head group, key split): a range of slots of the
// row's key list, in tiles of 128 slots,
//   slots [0, n_c)          compressed entries idx[slot] (CSA) or slot (HCA),
//   slots [n_c, n_c + n_w)  window positions t-n_w+1 .. t.
// The softmax is streamed over the tiles: per head a reference maximum m (log2
// units) is kept and raised only when a tile's maximum exceeds it by more than
// kRescaleLog2; then O^T (in tensor memory) and the running sums are scaled by
// exp2(m_old - m_new) before the tile's P.V is added.  P = exp2(c*s - m) <= 2^8
// is stored as bfloat16; o = O / l with l the sum of the stored P values, which
// is the exact softmax whatever m is.
//
// Warp-specialised CTA (9 warps):
//   warps 0-3  producer: q of the item into a resident buffer, then the key rows
//              of each tile, K one tile ahead of V, with 16-byte cp.async into a
//              ring of kRing 32 KiB stages (warp w fills every stage g with
//              g % kRing == w and blocks only on its own copies; empty slots are
//              zero-filled; a tile of R <= 32 or <= 64 used rows takes R/32
//              stages per operand, each holding R rows x 16384/R dims);
//   warp 4     MMA issuer (one thread): S(t+1) into the second score buffer while
//              the softmax works on S(t), then P(t).V(t);
//   warps 5-8  softmax of each tile (TMEM lane = key), O^T rescaling, and at the
//              end of the item the epilogue (TMEM lane = head dim).
// Persistent grid (at most one CTA per SM) looping over items.  Rows with one
// split write o directly.  When the rows are too few to fill the GPU, each row's
// key list is cut into S splits (one item per CTA); every split writes its
// normalised o and its lse (float32) to the workspace straight from tensor
// memory, and attn_merge, chained by programmatic dependent launch, combines the
// splits of a row in split order.
// Every wait is bounded (tc::kWaitLimitNs); on timeout the kernel records an error
// code in the library's device error word and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace ha {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kD = 512;                          // head dim handled
constexpr int kHG = 64;                          // heads per item (N of both MMAs)
constexpr int kTile = 128;                       // key slots per tile (M of the score MMA)
constexpr int kRing = 4;                         // shared-memory stages (one per producer warp)
constexpr int kStageBytes = 32768;               // 128 key rows x 128 dims
constexpr int kHalfBytes = kTile * 128;          // 128 key rows x 64 dims
constexpr int kQBytes = kHG * kD * 2;            // 64 heads x 512 dims
constexpr int kPBytes = kTile * kHG * 2;         // 128 keys x 64 heads
constexpr int kThreads = 9 * 32;
constexpr int kTmemCols = 512;
constexpr int kSCol = 0;                         // two S buffers: columns [0, 128)
constexpr int kOCol = 2 * kHG;                   // O^T: 4 x 64 columns [128, 384)
constexpr int kTokFlag = 1 << 30;                // slot code: per-token row
constexpr int kMinSplitKeys = 32;                // fewest keys per split the plan makes
constexpr float kRescaleLog2 = 8.f;              // P <= 2^8 before the reference moves

constexpr size_t kSmemRing = size_t(kRing) * kStageBytes;
constexpr size_t kSmemTbl = size_t(4) * 2 * kTile * 4;           // [warp][tile parity][128]
constexpr size_t kSmemMisc = (4 * 64 + 64 + 64 + 2 * 64) * 4 + 32 * 8 + 16;
constexpr size_t kSmem = 1024 + kQBytes + kSmemRing + kPBytes + kSmemTbl + kSmemMisc;
static_assert(kSmem <= 232448, "shared-memory budget");

struct TcArgs {
  const bf16* q;         // [rows, H, 512]
  const bf16* ck;        // [B, n_cap, 512]
  const bf16* cv;
  const int32_t* idx;    // [rows, k] or null (HCA)
  const bf16* k_tok;     // [B, tok_cap, 512]
  const bf16* v_tok;
  const int32_t* pos;    // decode: ctx_len [B]; prefill: q_pos [rows]
  int decode, Tq, H, n_cap, tok_cap, n_win, m, k, elig;
  float c;               // softmax scale * log2(e)
  int S, kps, HG;       // splits per (row, head group), keys per split, head groups
  long long n_items;     // rows * HG * S
  bf16* o;               // [rows, H, 512]        (S == 1)
  float* lse;            // [rows, H] or null     (S == 1)
  float* o_part;         // S > 1: float32 [rows, S, H, 512], merged by attn_merge
  float* lse_part;       // S > 1: [rows, S, H]
  int* err;
  int early;             // fused step: q and positions are read before the wait, idx after it
  int wait_last;         // fused step: nothing read comes from the previous kernel
};

struct Item {
  int r, b, hg, split;
  int t;          // query position
  int ne;         // eligible compressed entries
  int n_c, n_w;   // compressed / window slots of the row's key list
  int lo, hi;     // this item's slots [lo, hi)
  int nt;         // tiles (>= 1 even when the range is empty)
};

// The fields of item `it` that need no global read (row, head group, split, lo).
__device__ __forceinline__ Item item_head(const TcArgs& a, long long it) {
  Item x;
  x.split = int(it % a.S);
  const long long rest = it / a.S;
  x.hg = int(rest % a.HG);
  x.r = int(rest / a.HG);
  x.b = x.r / a.Tq;
  x.lo = x.split * a.kps;
  return x;
}

// The rest, from the query position.
__device__ __forceinline__ void item_tail(const TcArgs& a, Item& x) {
  x.t = a.decode ? a.pos[x.b] - 1 : a.pos[x.r];
  x.ne = x.t >= 0 ? n_eligible(x.t, a.n_win, a.m, a.elig, a.n_cap) : 0;
  x.n_c = a.idx ? a.k : x.ne;
  x.n_w = (x.t >= 0 && a.k_tok != nullptr) ? min(a.n_win, x.t + 1) : 0;   // null: no window
  x.hi = min(x.n_c + x.n_w, x.lo + a.kps);
  const int n = x.hi - x.lo;
  x.nt = n > 0 ? (n + kTile - 1) / kTile : 1;
}

__device__ __forceinline__ Item item_of(const TcArgs& a, long long it) {
  Item x = item_head(a, it);
  item_tail(a, x);
  return x;
}

// Key rows a tile's stages hold: the tile's slots rounded up to 32, 64 or 128.  A
// 32 KiB stage holds R rows x 16384/R dims (256/R swizzled 64-dim halves of R x
// 128 B), so a tile takes R/32 stages for K and as many for V.
__device__ __forceinline__ int tile_rows(const Item& x, int t) {
  const int n = x.hi - x.lo - t * kTile;
  return n <= 32 ? 32 : (n <= 64 ? 64 : kTile);
}

// Entry named by compressed slot `slot` (< n_c): idx[r, slot] (CSA) or slot (HCA).
// The load is unconditional on a clamped address, so that a loop over slots
// issues all of its loads before the first use.
__device__ __forceinline__ int slot_entry(const TcArgs& a, const Item& x, int slot) {
  if (!a.idx) return slot;
  const int s = min(max(slot, 0), a.k - 1);
  return __ldg(a.idx + (long long)x.r * a.k + s);
}

// Row of the key in `slot` given its entry j (ignored for window slots): -1 none;
// else b*n_cap + j (compressed entry j) or (b*tok_cap + token slot) | kTokFlag.
__device__ __forceinline__ int slot_code(const TcArgs& a, const Item& x, int slot, int j) {
  if (slot < x.lo || slot >= x.hi) return -1;
  if (slot < x.n_c) return (j >= 0 && j < x.ne) ? x.b * a.n_cap + j : -1;
  const int u = x.t - x.n_w + 1 + (slot - x.n_c);
  return (x.b * a.tok_cap + u % a.tok_cap) | kTokFlag;
}

__device__ __forceinline__ const bf16* key_row(const bf16* comp, const bf16* tok, int code) {
  return (code & kTokFlag) ? tok + (long long)(code & ~kTokFlag) * kD
                           : comp + (long long)code * kD;
}

// All `count` threads of barrier `id` vote; true iff every vote is true.
__device__ __forceinline__ bool named_barrier_all(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// 32 values per lane -> the op-reduction over the warp of value L, returned to lane L
// (31 shuffles: each step exchanges half of the remaining values).
template <typename Op>
__device__ __forceinline__ float warp_transpose_reduce32(const float (&v)[32], Op op) {
  const int lane = threadIdx.x & 31;
  float a[16], b[8], c[4], d[2];
  bool hi = lane & 16;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float send = hi ? v[i] : v[i + 16], keep = hi ? v[i + 16] : v[i];
    a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  hi = lane & 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = hi ? a[i] : a[i + 8], keep = hi ? a[i + 8] : a[i];
    b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  hi = lane & 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = hi ? b[i] : b[i + 4], keep = hi ? b[i + 4] : b[i];
    c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  hi = lane & 2;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = hi ? c[i] : c[i + 2], keep = hi ? c[i + 2] : c[i];
    d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  hi = lane & 1;
  const float send = hi ? d[0] : d[1], keep = hi ? d[1] : d[0];
  return op(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

struct MaxOp { __device__ float operator()(float x, float y) const { return fmaxf(x, y); } };

struct AddOp { __device__ float operator()(float x, float y) const { return x + y; } };

__global__ void __launch_bounds__(kThreads, 1) attn_decode_tc(const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sQ = base;                                  // 8 blocks x (64 heads x 128 B)
  unsigned char* ring = sQ + kQBytes;
  unsigned char* sP = ring + kSmemRing;
  int* tbl_all = reinterpret_cast<int*>(sP + kPBytes);       // [4 warps][2][128]
  float* red = reinterpret_cast<float*>(tbl_all + 4 * 2 * kTile);   // [4 warps][64]
  float* mref = red + 4 * 64;                                // [64] reference max (log2 units)
  float* alpha = mref + 64;                                  // [64] rescale of this tile
  float* stats = alpha + 64;                                 // [inv_l 64 | lse 64]
  uint64_t* full = reinterpret_cast<uint64_t*>(stats + 2 * 64);
  uint64_t* empty = full + kRing;
  uint64_t* q_full = empty + kRing;
  uint64_t* q_empty = q_full + 1;
  uint64_t* s_full = q_empty + 1;     // [2]
  uint64_t* s_empty = s_full + 2;     // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* pv_done = p_full + 1;
  uint64_t* o_empty = pv_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_empty + 1);
  int* rescale_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) { tc::mbar_init(&full[s], 32); tc::mbar_init(&empty[s], 1); }
    tc::mbar_init(q_full, 128);
    tc::mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) { tc::mbar_init(&s_full[i], 1); tc::mbar_init(&s_empty[i], 128); }
    tc::mbar_init(p_full, 128);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(o_empty, 128);
    tc::fence_mbar_init();
  }
  if (warp == 4) { tc::tmem_alloc(tmem_slot, kTmemCols); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // The set-up above touched no global memory.  Stand-alone calls wait for the
  // previous kernel here.  Inside a fused decode step q and the positions are
  // inputs of the step (final before its first kernel passed its own wait), so in
  // the CSA step the producer requests q first and waits only before it reads the
  // selection, the softmax warps before their first selection read; in the HCA
  // step nothing the kernel reads comes from the previous kernel (the compressor,
  // which writes a block no query of the step sees), so it waits only before it
  // exits.
  if (a.early || a.wait_last) pdl_release();
  else pdl_wait_then_release();

  if (warp < 4) {
    // ------------------------------------------------------------------ producer
    static_assert(kRing == 4, "one producer warp per ring stage");
    const int w = warp;                       // fills the stages g with g % kRing == w
    const int pt = threadIdx.x;               // 0..127
    const int rsub = lane >> 3, ch = lane & 7;   // rows rsub + 4 i, 16-byte chunk ch
    const uint32_t stage = tc::smem_u32(ring + size_t(w) * kStageBytes);
    const uint32_t q_base = tc::smem_u32(sQ);
    long long g = 0, n = 0;
    bool ok = true;
    auto put = [&](uint32_t dst, int code, const bf16* comp, const bf16* tok, int col) {
      if (code >= 0)
        tc::cp_async16(dst, key_row(comp, tok, code) + col);
      else
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0) : "memory");
    };
    bool q_pending = false;                   // q copies committed, not yet published
    auto publish = [&](uint64_t* bar) {
      tc::cp_async_commit();
      if (q_pending) {                        // the q group is the older one
        tc::cp_async_wait<1>();
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(q_full);
        q_pending = false;
      }
      tc::cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar);
    };
    for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, ++n) {
      // q of the item: every warp copies a quarter, once the previous item's score
      // MMAs are done with the buffer; its copies stay in flight (their own group)
      // while the first tile's table is built, and are published with this warp's
      // first stage.  q and the first tile's entries need no query position, so
      // they are requested before it is read.
      Item x = item_head(a, it);
      if (!(ok = tc::mbar_wait(q_empty, uint32_t((n & 1) ^ 1), a.err, 40))) break;
      const bf16* qrow = a.q + ((long long)x.r * a.H + x.hg * kHG) * kD;
#pragma unroll
      for (int i = 0; i < kQBytes / 16 / 128; ++i) {   // 32 chunks per thread
        const int c = pt + 128 * i;
        const int kb = c >> 9, h = (c >> 3) & 63;
        tc::cp_async16(q_base + kb * (kHG * 128) + h * 128 + ((ch ^ (h & 7)) << 4),
                       qrow + (long long)h * kD + kb * 64 + ch * 8);
      }
      tc::cp_async_commit();
      q_pending = true;
      if (a.early && n == 0) pdl_wait();      // the selection comes from the previous kernel
      int ent0[kTile / 32];
#pragma unroll
      for (int j = 0; j < kTile / 32; ++j) ent0[j] = slot_entry(a, x, x.lo + lane + 32 * j);
      item_tail(a, x);
      // stages: K(0); then per tile t: K(t+1), V(t).  Every warp keeps its own copy
      // of the row table of the tiles in flight, whether or not it fills a stage.
      // stage j of a tile with R rows: rows 0..R-1, 64-dim halves [j*hbs, (j+1)*hbs)
      auto fill = [&](int t, const bf16* comp, const bf16* tok, int err_code) -> bool {
        const int* tbl = tbl_all + (w * 2 + (t & 1)) * kTile;
        const int R = tile_rows(x, t), hbs = 256 / R;
        for (int j = 0; j < R / 32; ++j, ++g) {
          if (int(g % kRing) != w) continue;
          if (!tc::mbar_wait(&empty[w], uint32_t(((g / kRing) & 1) ^ 1), a.err, err_code)) return false;
          // 8 rows at a time: their codes in registers first (the copies are asm
          // statements with a memory clobber; table reads between them would be
          // serialised), then the copies of every half
#pragma unroll 1
          for (int i0 = 0; i0 < R / 4; i0 += 8) {
            int cd[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) cd[u] = tbl[rsub + 4 * (i0 + u)];
#pragma unroll 1
            for (int hb = 0; hb < hbs; ++hb) {
              const int col = (j * hbs + hb) * 64 + ch * 8;
              const uint32_t half_base = stage + hb * (R * 128);
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int row = rsub + 4 * (i0 + u);
                put(half_base + row * 128 + ((ch ^ (row & 7)) << 4), cd[u], comp, tok, col);
              }
            }
          }
          publish(&full[w]);
        }
        return true;
      };
      // K stages of tile t: the warp's copy of the tile's row table first
      auto k_stages = [&](int t) -> bool {
        int* tbl = tbl_all + (w * 2 + (t & 1)) * kTile;
        __syncwarp();
        int ent[kTile / 32];
#pragma unroll
        for (int j = 0; j < kTile / 32; ++j)
          ent[j] = t == 0 ? ent0[j] : slot_entry(a, x, x.lo + t * kTile + lane + 32 * j);
#pragma unroll
        for (int j = 0; j < kTile / 32; ++j)
          tbl[lane + 32 * j] = slot_code(a, x, x.lo + t * kTile + lane + 32 * j, ent[j]);
        __syncwarp();
        return fill(t, a.ck, a.k_tok, 41);
      };
      auto v_stages = [&](int t) -> bool { return fill(t, a.cv, a.v_tok, 42); };
      if (!(ok = k_stages(0))) break;
      for (int t = 0; t < x.nt && ok; ++t) {
        if (t + 1 < x.nt && !(ok = k_stages(t + 1))) break;
        ok = v_stages(t);
      }
      // an item of fewer than kRing stages leaves some warps without a stage of
      // their own: they publish their quarter of q here (no wait of theirs depends
      // on this item's MMAs, so this cannot hold up the score MMA)
      if (ok && q_pending) {
        tc::cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(q_full);
        q_pending = false;
      }
    }
    tc::cp_async_wait<0>();
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kHG);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, kHG, true, true);
      const uint32_t q_base = tc::smem_u32(sQ), p_base = tc::smem_u32(sP);
      long long g = 0, n = 0, G = 0;   // stage, item and global tile counters
      bool ok = true;
      // S(tile Gt, R key rows) from its R/32 K stages into score buffer Gt & 1.  The
      // MMA reads 128 rows from each half; rows R..127 belong to the next half or
      // stage (any values): their scores are never used.
      auto s_mma = [&](long long Gt, int R) -> bool {
        const int buf = int(Gt & 1), hbs = 256 / R;
        if (!tc::mbar_wait(&s_empty[buf], uint32_t(((Gt >> 1) & 1) ^ 1), a.err, 43)) return false;
        tc::fence_after_sync();
        for (int j = 0; j < R / 32; ++j, ++g) {
          const int s = int(g % kRing);
          if (!tc::mbar_wait(&full[s], uint32_t((g / kRing) & 1), a.err, 44)) return false;
          tc::fence_after_sync();
          const uint32_t sa = tc::smem_u32(ring + size_t(s) * kStageBytes);
          for (int hb = 0; hb < hbs; ++hb) {
            const int kb = j * hbs + hb;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_bf16(tmem + kSCol + buf * kHG,
                           tc::sdesc_kmajor_sw128(sa + hb * (R * 128) + kk * 32),
                           tc::sdesc_kmajor_sw128(q_base + kb * (kHG * 128) + kk * 32), idesc_s,
                           (kb | kk) != 0 ? 1u : 0u);
          }
          tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(&s_full[buf]);
        return true;
      };
      for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, ++n) {
        const Item x = item_of(a, it);
        if (!(ok = tc::mbar_wait(q_full, uint32_t(n & 1), a.err, 45))) break;
        tc::fence_after_sync();
        if (!(ok = s_mma(G, tile_rows(x, 0)))) break;
        if (x.nt == 1) tc::mma_commit(q_empty);
        for (int t = 0; t < x.nt && ok; ++t, ++G) {
          if (t + 1 < x.nt) {
            if (!(ok = s_mma(G + 1, tile_rows(x, t + 1)))) break;
            if (t + 2 == x.nt) tc::mma_commit(q_empty);
          }
          if (!(ok = tc::mbar_wait(p_full, uint32_t(G & 1), a.err, 46))) break;
          if (t == 0 && !(ok = tc::mbar_wait(o_empty, uint32_t((n & 1) ^ 1), a.err, 47))) break;
          tc::fence_after_sync();
          // V stage j holds dims [64*j*hbs, 64*(j+1)*hbs) of the tile's R keys, i.e.
          // the 128-dim O^T blocks j*hbs/2 .. (j+1)*hbs/2 - 1; R/16 K steps per block
          const int R = tile_rows(x, t), hbs = 256 / R;
          for (int j = 0; j < R / 32 && ok; ++j, ++g) {
            const int s = int(g % kRing);
            if (!(ok = tc::mbar_wait(&full[s], uint32_t((g / kRing) & 1), a.err, 48))) break;
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(ring + size_t(s) * kStageBytes);
            for (int mbl = 0; mbl < hbs / 2; ++mbl) {
              const int mb = j * (hbs / 2) + mbl;
              for (int kk = 0; kk < R / 16; ++kk)
                tc::mma_bf16(tmem + kOCol + mb * kHG,
                             tc::sdesc_sw128(sa + 2 * mbl * (R * 128) + kk * 2048, R * 128, 1024),
                             tc::sdesc_sw128(p_base + kk * 2048, kHalfBytes, 1024), idesc_o,
                             (t | kk) != 0 ? 1u : 0u);
            }
            tc::mma_commit(&empty[s]);
          }
          if (ok) tc::mma_commit(pv_done);
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int sw = warp - 5;                  // 0..3
    const int quarter = warp & 3;             // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;      // key slot within a tile / head dim within 128
    const uint32_t t_lane = uint32_t(quarter * 32) << 16;
    unsigned char* prow = sP + row * 128;
    const int rsw = row & 7;
    long long n = 0, G = 0;
    bool ok = true;
    if (a.early) pdl_wait();                  // slot_entry reads the selection
    for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, ++n) {
      const Item x = item_of(a, it);
      // this warp's share of the per-head sums of P: heads lane and 32 + lane
      float lw[2] = {0.f, 0.f};
      for (int t = 0; t < x.nt; ++t, ++G) {
        const int ent = slot_entry(a, x, x.lo + t * kTile + row);
        const bool valid = slot_code(a, x, x.lo + t * kTile + row, ent) >= 0;
        const int buf = int(G & 1);
        bool wok = tc::mbar_wait(&s_full[buf], uint32_t((G >> 1) & 1), a.err, 51);
        if (!(ok = named_barrier_all(1, 128, wok))) break;
        tc::fence_after_sync();
        // tile maximum per head
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kSCol + buf * kHG + half * 32, v);
          if (!valid) {
#pragma unroll
            for (int h = 0; h < 32; ++h) v[h] = -INFINITY;
          }
          red[sw * 64 + half * 32 + lane] = warp_transpose_reduce32(v, MaxOp());
        }
        tc::named_barrier(1, 128);
        if (sw == 0) {
          bool moved = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * lane + e;
            const float tm = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
            const float cand = tm == -INFINITY ? -INFINITY : tm * a.c;
            const float old = t == 0 ? -INFINITY : mref[h];
            float al = 1.f;
            if (old == -INFINITY) {
              mref[h] = cand;                 // nothing accumulated yet for this head
            } else if (cand > old + kRescaleLog2) {
              mref[h] = cand;
              al = tc::ex2_approx(old - cand);
              moved = true;
            }
            alpha[h] = al;
          }
          moved = __any_sync(0xffffffffu, moved);
          if (lane == 0) *rescale_flag = moved ? 1 : 0;
        }
        tc::named_barrier(1, 128);
        // P of the previous tile must be consumed (and O final) before P / O change
        if (G > 0) {
          wok = tc::mbar_wait(pv_done, uint32_t((G - 1) & 1), a.err, 52);
          if (!(ok = named_barrier_all(1, 128, wok))) break;
          tc::fence_after_sync();
        }
        if (*rescale_flag) {
          // O^T lane = head dim, column = head: scale column h by alpha[h]
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            float al[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) al[h] = alpha[half * 32 + h];
#pragma unroll 1
            for (int mb = 0; mb < kD / 128; ++mb) {
              float v[32];
              const uint32_t col = tmem + t_lane + kOCol + mb * kHG + half * 32;
              tc::tmem_ld32(col, v);
#pragma unroll
              for (int h = 0; h < 32; ++h) v[h] *= al[h];
              tc::tmem_st32(col, v);
            }
          }
          tc::tmem_wait_st();
          lw[0] *= alpha[lane];
          lw[1] *= alpha[32 + lane];
        }
        // P = exp2(c * s - m) as bfloat16, sums of the rounded values
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kSCol + buf * kHG + half * 32, v);
          uint32_t pk[16];
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const float p0 = valid ? tc::ex2_approx(v[h] * a.c - mref[half * 32 + h]) : 0.f;
            const float p1 = valid ? tc::ex2_approx(v[h + 1] * a.c - mref[half * 32 + h + 1]) : 0.f;
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            v[h] = __low2float(b2);           // the rounded values are the ones summed
            v[h + 1] = __high2float(b2);
            pk[h / 2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(prow + (((half * 4 + j) ^ rsw) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          lw[half] += warp_transpose_reduce32(v, AddOp());
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&s_empty[buf]);
        tc::mbar_arrive(p_full);
      }
      if (!ok) break;
      // ---- epilogue of the item: sums over the four warps, then O^T / l
      red[sw * 64 + lane] = lw[0];
      red[sw * 64 + 32 + lane] = lw[1];
      bool wok = tc::mbar_wait(pv_done, uint32_t((G - 1) & 1), a.err, 53);
      if (!(ok = named_barrier_all(1, 128, wok))) break;
      tc::fence_after_sync();
      if (sw == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          const float sum = (red[h] + red[64 + h]) + (red[128 + h] + red[192 + h]);
          stats[h] = sum > 0.f ? 1.f / sum : 0.f;
          stats[64 + h] = sum > 0.f ? (mref[h] + log2f(sum)) * 0.69314718055994531f : -INFINITY;
        }
      }
      tc::named_barrier(1, 128);
      if (a.S > 1) {
        // one split of the row: o = O^T / l and lse as float32 partials, merged by
        // attn_merge (lane = head dim: a warp stores 128 contiguous bytes per head)
        const long long prow = ((long long)x.r * a.S + x.split) * a.H + x.hg * kHG;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float sc[32];
#pragma unroll
          for (int h = 0; h < 32; ++h) sc[h] = stats[half * 32 + h];
#pragma unroll 1
          for (int mb = 0; mb < kD / 128; ++mb) {
            float v[32];
            tc::tmem_ld32(tmem + t_lane + kOCol + mb * kHG + half * 32, v);
            float* dst = a.o_part + (prow + half * 32) * kD + mb * 128 + row;
#pragma unroll
            for (int h = 0; h < 32; ++h) dst[(long long)h * kD] = v[h] * sc[h];
          }
        }
        if (sw < 2) a.lse_part[prow + sw * 32 + lane] = stats[64 + sw * 32 + lane];
        tc::fence_before_sync();
        tc::mbar_arrive(o_empty);
        tc::named_barrier(1, 128);
        continue;
      }
      const long long hrow = (long long)x.r * a.H + x.hg * kHG;   // first head of the group
      // 1/l of the 32 heads of a half in registers before any store (the stores
      // could otherwise alias them and serialise every load)
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float sc[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) sc[h] = stats[half * 32 + h];
#pragma unroll 1
        for (int mb = 0; mb < kD / 128; ++mb) {
          const int dd = mb * 128 + row;
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kOCol + mb * kHG + half * 32, v);
          bf16* dst = a.o + (hrow + half * 32) * kD + dd;
#pragma unroll
          for (int h = 0; h < 32; ++h) dst[(long long)h * kD] = __float2bfloat16_rn(v[h] * sc[h]);
        }
      }
      if (sw < 2 && a.lse) a.lse[hrow + sw * 32 + lane] = stats[64 + sw * 32 + lane];
      tc::fence_before_sync();
      tc::mbar_arrive(o_empty);
      tc::named_barrier(1, 128);              // stats and mref are rewritten by the next item
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
  if (a.wait_last) pdl_wait();
}

int g_num_sms[64] = {};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (g_num_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

}  // namespace

bool attention_tc_supported(const ha_params& p, int n_cap, int tok_cap) {
  return p.dtype == HA_BF16 && p.d == kD && p.H % kHG == 0 &&
         (long long)p.B * n_cap < kTokFlag && (long long)p.B * tok_cap < kTokFlag;
}

AttnPlan plan_attention_tc(const ha_params& p, int rows, int max_keys) {
  AttnPlan pl{};
  const long long units = (long long)rows * (p.H / kHG);
  const int sms = num_sms();
  // Enough splits per (row, head group) that the items cover the SMs in one wave,
  // but at least kMinSplitKeys keys per split (every split also loads q, 64 KiB).
  int S = units >= sms ? 1 : int(sms / units);
  const int by_keys = max_keys / kMinSplitKeys;
  if (S > by_keys) S = by_keys;
  if (S < 1) S = 1;
  int kps = (max_keys + S - 1) / S;
  kps = (kps + 15) / 16 * 16;
  if (kps < 16) kps = 16;
  S = (max_keys + kps - 1) / kps;
  if (S < 1) S = 1;
  pl.n_splits = S;
  pl.keys_per_split = kps;
  pl.tile = kTile;
  pl.ws_bytes = S > 1 ? size_t(rows) * S * p.H * (kD + 1) * sizeof(float) : 0;
  return pl;
}

cudaError_t launch_attention_tc(const ha_params& p, const AttnPlan& pl, int decode, int Tq,
                                const void* q, const int32_t* pos, const void* ck, const void* cv,
                                int n_cap, const int32_t* idx, const void* k_tok,
                                const void* v_tok, int tok_cap, void* o, float* lse, void* ws,
                                int* err, cudaStream_t st, const StepOpts& so) {
  TcArgs a{};
  a.early = so.early;
  a.wait_last = so.wait_last;
  a.q = static_cast<const bf16*>(q);
  a.ck = static_cast<const bf16*>(ck);
  a.cv = static_cast<const bf16*>(cv);
  a.idx = idx;
  a.k_tok = static_cast<const bf16*>(k_tok);
  a.v_tok = static_cast<const bf16*>(v_tok);
  a.pos = pos;
  a.decode = decode;
  a.Tq = Tq;
  a.H = p.H;
  a.n_cap = n_cap;
  a.tok_cap = tok_cap;
  a.n_win = p.n_win;
  a.m = p.m;
  a.k = p.k;
  a.elig = p.elig;
  const float scale = p.scale > 0.f ? p.scale : 1.f / sqrtf(float(p.d));
  a.c = scale * 1.4426950408889634f;
  a.S = pl.n_splits;
  a.kps = pl.keys_per_split;
  a.HG = p.H / kHG;
  const int rows = p.B * Tq;
  a.n_items = (long long)rows * a.S * a.HG;
  a.o = static_cast<bf16*>(o);
  a.lse = lse;
  a.err = err;
  if (a.S > 1) {
    if (ws == nullptr) return cudaErrorInvalidValue;
    a.o_part = static_cast<float*>(ws);
    a.lse_part = a.o_part + (long long)rows * a.S * p.H * kD;
  }
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(attn_decode_tc), kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = a.n_items < num_sms() ? a.n_items : num_sms();
  e = launch_pdl(attn_decode_tc, dim3(unsigned(grid)), dim3(kThreads), kSmem, st, 1u, a);
  if (e != cudaSuccess || a.S == 1) return e;
  return launch_attn_merge(p, rows, a.S, a.o_part, a.lse_part, o, lse, st);
}

}  // namespace ha
