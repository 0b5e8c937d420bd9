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
//   O^T[c, h]  += sum_key V[key, c] P[key, h]         (M = 128 dims x 4, N = 64, K = keys)
// Both MMAs read 128-byte-swizzled shared-memory tiles: K and q are K-major, V
// and P are MN-major (the row of 64 dims / 64 heads is contiguous), so the very
// same gathered key rows serve as the A operand of both products.
//
// Work item = (query row, 64-head group, key split): at most kMaxTiles tiles of
// 128 slots of the row's key list
//   slots [0, n_c)          compressed entries idx[slot] (CSA) or slot (HCA),
//   slots [n_c, n_c + n_w)  window positions t-n_w+1 .. t,
// so the exact softmax of the split is taken over scores held in tensor memory
// (no online rescaling).  A split writes its normalised output and log-sum-exp
// as a float32 partial that attn_merge combines in split order, or the final
// bfloat16 output when the row has one split.
//
// Persistent CTA (one per SM), warp-specialised:
//   warps 0-3  producer: gathers each tile's key rows with 16-byte cp.async into a
//              ring of kRing 32 KiB stages (per 64-dim block: 128 K rows + the 64
//              q rows; then per 128-dim block: 128 V rows), warming L2 with every
//              gathered row first;
//   warp 4     MMA issuer (one thread): S tiles, then O^T 128 dims at a time into
//              one of two tensor-memory accumulators;
//   warps 5-8  softmax: per-head max and sum over every tile of the item (TMEM
//              lane = key), P written as bfloat16 into shared memory;
//   warps 9-12 epilogue: O^T from tensor memory, scaled by 1/l, to global memory.
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
constexpr int kMaxTiles = 5;                     // tiles per item
constexpr int kRing = 4;                         // shared-memory stages
constexpr int kStageBytes = 32768;
constexpr int kKBlockBytes = kTile * 128;        // 128 key rows x 64 dims
constexpr int kPTileBytes = kTile * kHG * 2;     // 128 keys x 64 heads
constexpr int kThreads = 13 * 32;
constexpr int kTmemCols = 512;
constexpr int kSCol = 0;                         // S tiles: columns [0, 64 * kMaxTiles)
constexpr int kOCol = 64 * kMaxTiles;            // O^T double buffer: 2 x 64 columns
static_assert(kOCol + 2 * kHG <= kTmemCols, "tensor memory budget");
constexpr int kTokFlag = 1 << 30;                // slot code: per-token row

constexpr size_t kSmemRing = size_t(kRing) * kStageBytes;
constexpr size_t kSmemP = size_t(kMaxTiles) * kPTileBytes;
constexpr size_t kSmemMisc = 4 * 64 * 4 + 64 * 4 + 2 * 128 * 4 + 32 * 8 + 16;
constexpr size_t kSmemUsed = 1024 + kSmemRing + kSmemP + kSmemMisc;
// The whole 227 KiB is requested (one CTA per SM either way): every operand read
// the descriptors can address, even with the leading / stride offsets exchanged,
// then stays inside the CTA's shared memory.
constexpr size_t kSmem = 232448;
static_assert(kSmemUsed <= kSmem, "shared-memory budget");
// farthest byte of the last P tile's last K step if LBO (16 KiB) were taken as SBO
static_assert(1023 + kSmemRing + (kMaxTiles - 1) * kPTileBytes + 7 * 2048 + kKBlockBytes + 1024 <=
                  kSmem, "descriptor reach");

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
  int S, kps, HG;
  long long n_items;     // rows * S * HG
  bf16* o;               // [rows, H, 512]         (S == 1)
  float* lse;            // [rows, H] or null      (S == 1)
  float* o_part;         // [rows, S, H, 512]      (S > 1)
  float* lse_part;       // [rows, S, H]
  int* err;
};

struct Item {
  int r, b, hg, split;
  int t;          // query position
  int ne;         // eligible compressed entries
  int n_c, n_w;   // compressed / window slots of the row's key list
  int lo, hi;     // this item's slots [lo, hi)
  int nt;         // tiles (>= 1 even when the range is empty)
};

__device__ __forceinline__ Item item_of(const TcArgs& a, long long it) {
  Item x;
  x.hg = int(it % a.HG);
  const long long rest = it / a.HG;
  x.split = int(rest % a.S);
  x.r = int(rest / a.S);
  x.b = x.r / a.Tq;
  x.t = a.decode ? a.pos[x.b] - 1 : a.pos[x.r];
  x.ne = x.t >= 0 ? n_eligible(x.t, a.n_win, a.m, a.elig, a.n_cap) : 0;
  x.n_c = a.idx ? a.k : x.ne;
  x.n_w = x.t >= 0 ? min(a.n_win, x.t + 1) : 0;
  x.lo = x.split * a.kps;
  x.hi = min(x.n_c + x.n_w, x.lo + a.kps);
  const int n = x.hi - x.lo;
  x.nt = n > 0 ? (n + kTile - 1) / kTile : 1;
  return x;
}

// Row of the key in `slot`: -1 none; else b*n_cap + j (compressed entry j) or
// (b*tok_cap + token slot) | kTokFlag (window position).
__device__ __forceinline__ int slot_code(const TcArgs& a, const Item& x, int slot) {
  if (slot < x.lo || slot >= x.hi) return -1;
  if (slot < x.n_c) {
    const int j = a.idx ? __ldg(a.idx + (long long)x.r * a.k + slot) : slot;
    return (j >= 0 && j < x.ne) ? x.b * a.n_cap + j : -1;
  }
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

// 64 values per lane -> lane L holds op-reductions over the warp of values 2L, 2L+1.
template <typename Op>
__device__ __forceinline__ void warp_transpose_reduce64(const float (&v)[64], float& r0,
                                                        float& r1, Op op) {
  const int lane = threadIdx.x & 31;
  float a[32], b[16], c[8], d[4];
  bool hi = lane & 16;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float send = hi ? v[i] : v[i + 32], keep = hi ? v[i + 32] : v[i];
    a[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
  hi = lane & 8;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float send = hi ? a[i] : a[i + 16], keep = hi ? a[i + 16] : a[i];
    b[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
  hi = lane & 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = hi ? b[i] : b[i + 8], keep = hi ? b[i + 8] : b[i];
    c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  hi = lane & 2;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = hi ? c[i] : c[i + 4], keep = hi ? c[i + 4] : c[i];
    d[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  }
  hi = lane & 1;
  {
    const float send0 = hi ? d[0] : d[2], keep0 = hi ? d[2] : d[0];
    const float send1 = hi ? d[1] : d[3], keep1 = hi ? d[3] : d[1];
    r0 = op(keep0, __shfl_xor_sync(0xffffffffu, send0, 1));
    r1 = op(keep1, __shfl_xor_sync(0xffffffffu, send1, 1));
  }
}

struct MaxOp { __device__ float operator()(float x, float y) const { return fmaxf(x, y); } };
struct AddOp { __device__ float operator()(float x, float y) const { return x + y; } };

__global__ void __launch_bounds__(kThreads, 1) attn_decode_tc(const TcArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ring = base;
  unsigned char* sP = ring + kSmemRing;
  float* red = reinterpret_cast<float*>(sP + kSmemP);   // [4 warps][64]
  float* fin = red + 4 * 64;                             // [64] log2-scaled max
  float* stats = fin + 64;                               // [2 items][inv_l 64 | lse 64]
  uint64_t* full = reinterpret_cast<uint64_t*>(stats + 2 * 128);
  uint64_t* empty = full + kRing;
  uint64_t* s_full = empty + kRing;
  uint64_t* p_full = s_full + 1;
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_full = p_empty + 1;     // [2]
  uint64_t* o_empty = o_full + 2;     // [2]
  uint64_t* st_full = o_empty + 2;    // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(st_full + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) { tc::mbar_init(&full[s], 128); tc::mbar_init(&empty[s], 1); }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_full, 128);
    tc::mbar_init(p_empty, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&o_full[i], 1);
      tc::mbar_init(&o_empty[i], 128);
      tc::mbar_init(&st_full[i], 32);
    }
    tc::fence_mbar_init();
  }
  // Rows a tile does not load keep their previous (finite) contents; start from zeros.
  for (int i = threadIdx.x; i < int((kSmemRing + kSmemP) / 16); i += kThreads)
    reinterpret_cast<uint4*>(ring)[i] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (warp == 4) { tc::tmem_alloc(tmem_slot, kTmemCols); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------------ producer
    const int pt = threadIdx.x;               // 0..127
    const int rbase = pt >> 3, ch = pt & 7;   // rows rbase + 16 i, 16-byte chunk ch
    const uint32_t swz = uint32_t((ch ^ (rbase & 7)) << 4);
    long long g = 0, arrived = 0;
    bool ok = true;
    auto acquire = [&](uint32_t& sa) -> bool {
      const int s = int(g % kRing);
      if (!tc::mbar_wait(&empty[s], uint32_t(((g / kRing) & 1) ^ 1), a.err, 41)) return false;
      sa = tc::smem_u32(ring + size_t(s) * kStageBytes);
      return true;
    };
    auto release = [&]() {
      tc::cp_async_commit();
      ++g;
      if (g - arrived > kRing - 1) {
        tc::cp_async_wait<kRing - 1>();
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&full[arrived % kRing]);
        ++arrived;
      }
    };
    for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x) {
      const Item x = item_of(a, it);
      int code[kMaxTiles][8];
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          code[t][i] = t < x.nt ? slot_code(a, x, x.lo + t * kTile + rbase + 16 * i) : -1;
      const bf16* qrow = a.q + ((long long)x.r * a.H + x.hg * kHG) * kD;
      // scores: per tile, 8 blocks of 64 dims (K rows + q rows)
      for (int t = 0; t < x.nt && ok; ++t) {
        if (ch == 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (code[t][i] >= 0) {
              tc::prefetch_l2(key_row(a.ck, a.k_tok, code[t][i]), kD * 2);
              tc::prefetch_l2(key_row(a.cv, a.v_tok, code[t][i]), kD * 2);
            }
        }
        for (int kb = 0; kb < kD / 64; ++kb) {
          uint32_t sa;
          if (!(ok = acquire(sa))) break;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (code[t][i] >= 0)
              tc::cp_async16(sa + (rbase + 16 * i) * 128 + swz,
                             key_row(a.ck, a.k_tok, code[t][i]) + kb * 64 + ch * 8);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            tc::cp_async16(sa + kKBlockBytes + (rbase + 16 * i) * 128 + swz,
                           qrow + (long long)(rbase + 16 * i) * kD + kb * 64 + ch * 8);
          release();
        }
      }
      // values: per 128-dim block, every tile
      for (int mb = 0; mb < kD / 128 && ok; ++mb) {
        for (int t = 0; t < x.nt; ++t) {
          uint32_t sa;
          if (!(ok = acquire(sa))) break;
#pragma unroll
          for (int cb = 0; cb < 2; ++cb)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (code[t][i] >= 0)
                tc::cp_async16(sa + cb * kKBlockBytes + (rbase + 16 * i) * 128 + swz,
                               key_row(a.cv, a.v_tok, code[t][i]) + mb * 128 + cb * 64 + ch * 8);
          release();
        }
      }
    }
    tc::cp_async_wait<0>();
    tc::fence_proxy_async_smem();
    if (ok)
      while (arrived < g) { tc::mbar_arrive(&full[arrived % kRing]); ++arrived; }
  } else if (warp == 4) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kTile, kHG);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, kHG, true, true);
      const uint32_t p_base = tc::smem_u32(sP);
      long long g = 0, n = 0, ob = 0;
      bool ok = true;
      for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, ++n) {
        const Item x = item_of(a, it);
        for (int t = 0; t < x.nt && ok; ++t)
          for (int kb = 0; kb < kD / 64; ++kb, ++g) {
            const int s = int(g % kRing);
            if (!(ok = tc::mbar_wait(&full[s], uint32_t((g / kRing) & 1), a.err, 42))) break;
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(ring + size_t(s) * kStageBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_bf16(tmem + kSCol + t * kHG, tc::sdesc_kmajor_sw128(sa + kk * 32),
                           tc::sdesc_kmajor_sw128(sa + kKBlockBytes + kk * 32), idesc_s,
                           (kb | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&empty[s]);
          }
        if (!ok) break;
        tc::mma_commit(s_full);
        if (!(ok = tc::mbar_wait(p_full, uint32_t(n & 1), a.err, 43))) break;
        tc::fence_after_sync();
        for (int mb = 0; mb < kD / 128 && ok; ++mb, ++ob) {
          const int buf = int(ob & 1);
          if (!(ok = tc::mbar_wait(&o_empty[buf], uint32_t(((ob >> 1) & 1) ^ 1), a.err, 44))) break;
          tc::fence_after_sync();
          for (int t = 0; t < x.nt; ++t, ++g) {
            const int s = int(g % kRing);
            if (!(ok = tc::mbar_wait(&full[s], uint32_t((g / kRing) & 1), a.err, 45))) break;
            tc::fence_after_sync();
            const uint32_t sa = tc::smem_u32(ring + size_t(s) * kStageBytes);
            const uint32_t pa = p_base + t * kPTileBytes;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              tc::mma_bf16(tmem + kOCol + buf * kHG,
                           tc::sdesc_sw128(sa + kk * 2048, kKBlockBytes, 1024),
                           tc::sdesc_sw128(pa + kk * 2048, kKBlockBytes, 1024), idesc_o,
                           (t | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&empty[s]);
          }
          if (ok) tc::mma_commit(&o_full[buf]);
        }
        if (ok) tc::mma_commit(p_empty);
      }
    }
  } else if (warp < 9) {
    // ------------------------------------------------------------------ softmax
    const int sw = warp - 5;                  // 0..3
    const int quarter = warp & 3;             // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;      // key slot within a tile
    const uint32_t t_lane = uint32_t(quarter * 32) << 16;
    unsigned char* prow = sP + row * 128;
    const int rsw = row & 7;
    long long n = 0;
    for (long long it = blockIdx.x; it < a.n_items; it += gridDim.x, ++n) {
      const Item x = item_of(a, it);
      bool w = tc::mbar_wait(p_empty, uint32_t((n & 1) ^ 1), a.err, 51);
      w = w && tc::mbar_wait(s_full, uint32_t(n & 1), a.err, 52);
      if (!named_barrier_all(1, 128, w)) break;
      tc::fence_after_sync();
      unsigned vmask = 0;
      for (int t = 0; t < x.nt; ++t)
        if (slot_code(a, x, x.lo + t * kTile + row) >= 0) vmask |= 1u << t;
      // pass 1: per-head maximum over the item's keys
      float mx[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) mx[h] = -INFINITY;
      for (int t = 0; t < x.nt; ++t) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kSCol + t * kHG + half * 32, v);
          if ((vmask >> t) & 1) {
#pragma unroll
            for (int h = 0; h < 32; ++h) mx[half * 32 + h] = fmaxf(mx[half * 32 + h], v[h]);
          }
        }
      }
      {
        float r0, r1;
        warp_transpose_reduce64(mx, r0, r1, MaxOp());
        red[sw * 64 + 2 * lane] = r0;
        red[sw * 64 + 2 * lane + 1] = r1;
      }
      tc::named_barrier(1, 128);
      if (sw == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          const float m = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
          fin[h] = m == -INFINITY ? -INFINITY : m * a.c;
        }
      }
      tc::named_barrier(1, 128);
      // pass 2: P = exp2(c * s - m) as bfloat16, row sums of the rounded values
      float l[64];
#pragma unroll
      for (int h = 0; h < 64; ++h) l[h] = 0.f;
      for (int t = 0; t < x.nt; ++t) {
        const bool valid = (vmask >> t) & 1;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kSCol + t * kHG + half * 32, v);
          uint32_t pk[16];
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            const float p0 = valid ? exp2f(v[h] * a.c - fin[half * 32 + h]) : 0.f;
            const float p1 = valid ? exp2f(v[h + 1] * a.c - fin[half * 32 + h + 1]) : 0.f;
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            l[half * 32 + h] += __low2float(b2);
            l[half * 32 + h + 1] += __high2float(b2);
            pk[h / 2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(prow + t * kPTileBytes + (((half * 4 + j) ^ rsw) << 4)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      tc::mbar_arrive(p_full);
      {
        float r0, r1;
        warp_transpose_reduce64(l, r0, r1, AddOp());
        red[sw * 64 + 2 * lane] = r0;
        red[sw * 64 + 2 * lane + 1] = r1;
      }
      tc::named_barrier(1, 128);
      if (sw == 0) {
        float* st = stats + (n & 1) * 128;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * lane + e;
          const float sum = (red[h] + red[64 + h]) + (red[128 + h] + red[192 + h]);
          st[h] = sum > 0.f ? 1.f / sum : 0.f;
          st[64 + h] = sum > 0.f ? (fin[h] + log2f(sum)) * 0.69314718055994531f : -INFINITY;
        }
        tc::mbar_arrive(&st_full[n & 1]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const uint32_t t_lane = uint32_t(quarter * 32) << 16;
    const int e = (warp - 9) * 32 + lane;     // 0..127
    long long n = 0, ob = 0;
    bool ok = true;
    for (long long it = blockIdx.x; it < a.n_items && ok; it += gridDim.x, ++n) {
      const Item x = item_of(a, it);
      if (!(ok = tc::mbar_wait(&st_full[n & 1], uint32_t((n >> 1) & 1), a.err, 61))) break;
      const float* st = stats + (n & 1) * 128;
      const long long hrow = (long long)x.r * a.H + x.hg * kHG;   // first head of the group
      for (int mb = 0; mb < kD / 128; ++mb, ++ob) {
        const int buf = int(ob & 1);
        if (!(ok = tc::mbar_wait(&o_full[buf], uint32_t((ob >> 1) & 1), a.err, 62))) break;
        tc::fence_after_sync();
        const int dd = mb * 128 + quarter * 32 + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tc::tmem_ld32(tmem + t_lane + kOCol + buf * kHG + half * 32, v);
          if (a.S == 1) {
#pragma unroll
            for (int h = 0; h < 32; ++h)
              a.o[(hrow + half * 32 + h) * kD + dd] = __float2bfloat16_rn(v[h] * st[half * 32 + h]);
          } else {
            float* dst = a.o_part + (((long long)x.r * a.S + x.split) * a.H + x.hg * kHG) * kD + dd;
#pragma unroll
            for (int h = 0; h < 32; ++h) dst[(long long)(half * 32 + h) * kD] = v[h] * st[half * 32 + h];
          }
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&o_empty[buf]);
      }
      if (ok && e < kHG) {
        if (a.S == 1) {
          if (a.lse) a.lse[hrow + e] = st[64 + e];
        } else {
          a.lse_part[((long long)x.r * a.S + x.split) * a.H + x.hg * kHG + e] = st[64 + e];
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 4) tc::tmem_dealloc(tmem, kTmemCols);
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
  const int per_item = kMaxTiles * kTile;
  const int s_min = (max_keys + per_item - 1) / per_item;
  const int sms = num_sms();
  int S = units >= sms ? 1 : int(sms / units);
  if (S < s_min) S = s_min;
  if (S < 1) S = 1;
  int kps = (max_keys + S - 1) / S;
  kps = (kps + 15) / 16 * 16;
  if (kps < 16) kps = 16;
  S = (max_keys + kps - 1) / kps;
  if (S < 1) S = 1;
  pl.n_splits = S;
  pl.keys_per_split = kps;
  pl.tile = kTile;
  pl.ws_bytes = S > 1 ? size_t(rows) * S * p.H * (p.d + 1) * sizeof(float) + 256 : 0;
  return pl;
}

cudaError_t launch_attention_tc(const ha_params& p, const AttnPlan& pl, int decode, int Tq,
                                const void* q, const int32_t* pos, const void* ck, const void* cv,
                                int n_cap, const int32_t* idx, const void* k_tok,
                                const void* v_tok, int tok_cap, void* o, float* lse, void* ws,
                                int* err, cudaStream_t st) {
  TcArgs a{};
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
  if (a.S > 1) {
    a.o_part = static_cast<float*>(ws);
    a.lse_part = a.o_part + size_t(rows) * a.S * p.H * p.d;
  }
  a.err = err;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(attn_decode_tc), kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = a.n_items < num_sms() ? a.n_items : num_sms();
  attn_decode_tc<<<unsigned(grid), kThreads, kSmem, st>>>(a);
  e = launched(cudaGetLastError());
  if (e != cudaSuccess || a.S == 1) return e;
  return launch_attn_merge(p, rows, a.S, a.o_part, a.lse_part, o, lse, st);
}

}  // namespace ha
