// Lightning Indexer on the tcgen05 tensor cores ("DeepSeek-V4 深度研究剖析" §5.3:
// the indexer scores every compressed CSA entry; "EP 95 解读 DeepSeek-V4 论文": it
// must look at everything, so it must be light).  Score formula fixed by this
// library:  s[b,t,j] = sum_h w[b,t,h] * max(0, qI[b,t,h,:] . cI[b,j,:]).
//
// The scores of one query are a skinny GEMM: 64 heads x 128 dims against every
// entry (64 flop per byte of keys), far above the CUDA-core ridge, so the heads
// go on the tensor cores.  Entries are the M dimension (128 per tile), the QT
// queries x 64 heads of a query group the N dimension, d_I = 128 the K dimension:
//   D[j, (q,h)] = sum_c cI[j, c] * qI[q, h, c]      (tcgen05.mma kind::f16, fp32)
// so that the head reduction of the epilogue stays inside one TMEM lane: each
// epilogue thread owns one entry and sums w_h * ReLU(D) over its 64 columns per
// query in head order.
//
// Persistent, warp-specialised CTA (one per SM): warp 0 streams 32 KiB key
// tiles with TMA into a ring of kStages stages (the query group's operand is
// loaded once per group), warp 1 issues 8 MMAs per tile into one of two TMEM
// accumulators, warps 2-5 drain the accumulators and write the scores.  The
// work list is every (sequence, query group, 128-entry tile) with at least one
// eligible entry, split evenly across CTAs in (group, tile) order.  Decode uses
// QT = 1 (N = 64), prefill QT = 4 (N = 256).
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.h"
#include "tc.cuh"
#include "tc_host.h"

namespace ha {
namespace {

constexpr int kHeads = 64;      // H_I handled by this kernel
constexpr int kDim = 128;       // d_I handled by this kernel
constexpr int kTileM = 128;     // entries per tile
constexpr int kThreads = 192;   // 6 warps
constexpr int kTileBytes = kTileM * kDim * 2;   // 32 KiB

template <int QT> struct Cfg {
  static constexpr int N = QT * kHeads;
  static constexpr int kStages = QT == 1 ? 6 : (QT == 2 ? 5 : 4);
  static constexpr int kQBytes = N * kDim * 2;
  // decode: two query buffers, so that a CTA whose tile range crosses into the
  // next sequence loads that sequence's query while the last tiles of the
  // previous one are still in flight (one buffer stalled such CTAs by a full DRAM
  // round trip and made them the kernel's tail)
  static constexpr int kQBuf = QT == 1 ? 2 : 1;
  static constexpr int kTmemCols = 2 * N < 32 ? 32 : 2 * N;
  // epilogue warps: one per TMEM lane quarter, or two (each with half of the
  // group's queries) when four queries share a tile, so that the drain keeps up
  // with the MMAs
  static constexpr int kEpiWarps = QT == 4 ? 8 : 4;
  static constexpr int kThreadsQ = 64 + 32 * kEpiWarps;
  static constexpr size_t kSmem = 1024 + size_t(kStages) * kTileBytes + size_t(kQBuf) * kQBytes +
                                  size_t(kEpiWarps) * QT * kHeads * sizeof(float) + 256;
};

static_assert(Cfg<1>::kSmem <= 232448 && Cfg<4>::kSmem <= 232448, "shared-memory budget");

struct IdxArgs {
  const float* w;          // [B*Tq, H_I]
  const int32_t* q_pos;    // [B*Tq]; query position = q_pos + pos_off
  float* scores;           // [B*Tq, n_cap]
  int B, Tq, n_cap, n_win, m, elig;
  int* err;
  int pos_off;
  int wait_last;           // fused step: wait for the previous kernel only before exiting
};

// Tiles of group g = (b, qg): ceil(max n_elig over its queries / 128).
template <int QT>
__device__ __forceinline__ int group_tiles(const IdxArgs& a, int g) {
  const int gpb = (a.Tq + QT - 1) / QT;
  const int b = g / gpb, q0 = (g % gpb) * QT;
  int ne = 0;
#pragma unroll
  for (int q = 0; q < QT; ++q)
    if (q0 + q < a.Tq)
      ne = max(ne, n_eligible(a.q_pos[b * a.Tq + q0 + q] + a.pos_off, a.n_win, a.m, a.elig, a.n_cap));
  return (ne + kTileM - 1) / kTileM;
}

// Walk over this CTA's tiles in (group, tile) order.  Every role warp runs the
// same walk; init() scans all groups with the whole warp.
template <int QT>
struct TileWalk {
  int g, t, tiles_g, left, n_groups;
  __device__ bool init(const IdxArgs& a) {
    const int lane = threadIdx.x & 31;
    n_groups = a.B * ((a.Tq + QT - 1) / QT);
    long long total = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int gg = base + lane;
      int c = gg < n_groups ? group_tiles<QT>(a, gg) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      total += c;
    }
    const long long lo = total * blockIdx.x / gridDim.x;
    const long long hi = total * (blockIdx.x + 1) / gridDim.x;
    left = int(hi - lo);
    if (left <= 0) return false;
    // find the group holding tile `lo`
    long long run = 0;
    g = 0;
    for (int base = 0; base < n_groups; base += 32) {
      const int gg = base + lane;
      const int c = gg < n_groups ? group_tiles<QT>(a, gg) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      if (run + tot > lo) {
        const unsigned hit = __ballot_sync(0xffffffffu, run + incl > lo);
        const int l = __ffs(hit) - 1;
        const int excl = __shfl_sync(0xffffffffu, incl - c, l);
        g = base + l;
        t = int(lo - run - excl);
        tiles_g = __shfl_sync(0xffffffffu, c, l);
        return true;
      }
      run += tot;
    }
    return false;
  }
  // Advance to the next tile; returns false at the end of the range.
  __device__ bool next(const IdxArgs& a) {
    if (--left <= 0) return false;
    if (++t >= tiles_g) {
      do {
        ++g;
        tiles_g = g < n_groups ? group_tiles<QT>(a, g) : 1;
      } while (tiles_g == 0);
      t = 0;
    }
    return true;
  }
  __device__ bool last_of_group() const { return left == 1 || t + 1 >= tiles_g; }
};

template <int QT>
__global__ void __launch_bounds__(Cfg<QT>::kThreadsQ, 1)
    index_scores_tc(const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_q, IdxArgs a) {
  using C = Cfg<QT>;
  if (a.wait_last) pdl_release();
  else pdl_wait_then_release();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* s_k = base;                                   // kStages x 32 KiB
  unsigned char* s_q = s_k + size_t(C::kStages) * kTileBytes;  // kQBuf x QT x 16 KiB
  float* s_w = reinterpret_cast<float*>(s_q + size_t(C::kQBuf) * C::kQBytes);  // [epi warps][QT][64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_w + C::kEpiWarps * QT * kHeads);
  uint64_t* full = bars;                   // [kStages]
  uint64_t* empty = full + C::kStages;     // [kStages]
  uint64_t* acc_full = empty + C::kStages; // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint64_t* q_full = acc_empty + 2;        // [kQBuf]
  uint64_t* q_empty = q_full + C::kQBuf;   // [kQBuf]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + C::kQBuf);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TileWalk<QT> walk;
  const bool have = walk.init(a);      // identical in every warp
  if (!have) return;                   // CTA-uniform

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) { tc::mbar_init(&full[s], 1); tc::mbar_init(&empty[s], 1); }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_empty[i], C::kEpiWarps);
    }
    for (int i = 0; i < C::kQBuf; ++i) { tc::mbar_init(&q_full[i], 1); tc::mbar_init(&q_empty[i], 1); }
    tc::fence_mbar_init();
  }
  if (warp == 1) { tc::tmem_alloc(tmem_slot, C::kTmemCols); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int gpb = (a.Tq + QT - 1) / QT;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::tma_prefetch(&map_k);
      tc::tma_prefetch(&map_q);
      int i = 0, prev_g = -1, n_groups_seen = 0;
      do {
        if (walk.g != prev_g) {
          // group j uses buffer j % kQBuf once group j - kQBuf has released it
          const int qb = n_groups_seen % C::kQBuf, use = n_groups_seen / C::kQBuf;
          if (use > 0 && !tc::mbar_wait(&q_empty[qb], (use - 1) & 1, a.err, 11)) break;
          const int b = walk.g / gpb, q0 = (walk.g % gpb) * QT;
          const int y = (b * a.Tq + q0) * kHeads;
          unsigned char* qdst = s_q + size_t(qb) * C::kQBytes;
          tc::mbar_expect_tx(&q_full[qb], C::kQBytes);
          tc::tma_load_2d(qdst, &map_q, 0, y, &q_full[qb]);
          tc::tma_load_2d(qdst + C::kQBytes / 2, &map_q, 64, y, &q_full[qb]);
          prev_g = walk.g;
          ++n_groups_seen;
        }
        const int s = i % C::kStages;
        if (!tc::mbar_wait(&empty[s], ((i / C::kStages) & 1) ^ 1, a.err, 12)) break;
        const int b = walk.g / gpb;
        const int y = b * a.n_cap + walk.t * kTileM;
        unsigned char* dst = s_k + size_t(s) * kTileBytes;
        tc::mbar_expect_tx(&full[s], kTileBytes);
        tc::tma_load_2d(dst, &map_k, 0, y, &full[s]);
        tc::tma_load_2d(dst + kTileBytes / 2, &map_k, 64, y, &full[s]);
        ++i;
      } while (walk.next(a));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kTileM, C::N);
      const uint32_t k_base = tc::smem_u32(s_k);
      uint32_t q_base = tc::smem_u32(s_q);
      int i = 0, prev_g = -1, n_groups_seen = 0, qb = 0;
      do {
        if (walk.g != prev_g) {
          qb = n_groups_seen % C::kQBuf;
          if (!tc::mbar_wait(&q_full[qb], (n_groups_seen / C::kQBuf) & 1, a.err, 21)) break;
          q_base = tc::smem_u32(s_q + size_t(qb) * C::kQBytes);
          prev_g = walk.g;
          ++n_groups_seen;
        }
        const int s = i % C::kStages, acc = i & 1;
        if (!tc::mbar_wait(&full[s], (i / C::kStages) & 1, a.err, 22)) break;
        if (!tc::mbar_wait(&acc_empty[acc], ((i >> 1) & 1) ^ 1, a.err, 23)) break;
        tc::fence_after_sync();
        const uint32_t kb = k_base + s * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kDim / 16; ++kk) {
          const uint32_t off_k = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          const uint32_t off_q = (kk >> 2) * (C::kQBytes / 2) + (kk & 3) * 32;
          tc::mma_bf16(tmem + acc * C::N, tc::sdesc_kmajor_sw128(kb + off_k),
                       tc::sdesc_kmajor_sw128(q_base + off_q), idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[acc]);
        if (walk.last_of_group()) tc::mma_commit(&q_empty[qb]);
        ++i;
      } while (walk.next(a));
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..)
    const int quarter = warp & 3;                     // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;              // entry within the tile
    float* w_mine = s_w + (warp - 2) * QT * kHeads;   // this warp's copy of the weights
    // the group's queries this warp drains: all, or one half with two warps per quarter
    constexpr int QW = C::kEpiWarps == 8 ? QT / 2 : QT;
    const int qw0 = C::kEpiWarps == 8 ? ((warp - 2) >> 2) * QW : 0;
    int ne_q[QT];                                     // eligible entries of the group's queries
    float w_reg[QT == 1 ? kHeads : 1];                // decode: the weights stay in registers
    int i = 0, prev_g = -1;
    bool ok = true;
    do {
      const int b = walk.g / gpb, q0 = (walk.g % gpb) * QT;
      if (walk.g != prev_g) {                         // warp-private: no cross-warp barrier
        __syncwarp();
        for (int x = lane; x < QT * kHeads; x += 32) {
          const int q = x / kHeads;
          w_mine[x] = (q0 + q < a.Tq) ? a.w[(long long)(b * a.Tq + q0 + q) * kHeads + x % kHeads] : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < QT; ++q)
          ne_q[q] = q0 + q < a.Tq
                        ? n_eligible(a.q_pos[b * a.Tq + q0 + q] + a.pos_off, a.n_win, a.m, a.elig, a.n_cap)
                        : 0;
        if constexpr (QT == 1) {
#pragma unroll
          for (int h = 0; h < kHeads; ++h) w_reg[h] = w_mine[h];
        }
        prev_g = walk.g;
      }
      const int acc = i & 1;
      ok = tc::mbar_wait(&acc_full[acc], (i >> 1) & 1, a.err, 31);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc::fence_after_sync();
      const int j = walk.t * kTileM + row;
      if constexpr (QT == 1) {
        float v0[32], v1[32];
        tc::tmem_ld32x2(tmem + (uint32_t(quarter * 32) << 16) + acc * C::N,
                        tmem + (uint32_t(quarter * 32) << 16) + acc * C::N + 32, v0, v1);
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(w_reg[h], fmaxf(v0[h], 0.f), s);
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(w_reg[32 + h], fmaxf(v1[h], 0.f), s);
        if (j < ne_q[0]) a.scores[((long long)b * a.Tq + q0) * a.n_cap + j] = s;
      } else {
#pragma unroll
        for (int qq = 0; qq < QW; ++qq) {
          const int q = qw0 + qq;
          const uint32_t col = tmem + (uint32_t(quarter * 32) << 16) + acc * C::N + q * kHeads;
          float v0[32], v1[32];
          tc::tmem_ld32x2(col, col + 32, v0, v1);
          const float4* w4 = reinterpret_cast<const float4*>(w_mine + q * kHeads);
          float s = 0.f;
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wv = w4[h4];
            s = fmaf(wv.x, fmaxf(v0[4 * h4], 0.f), s);
            s = fmaf(wv.y, fmaxf(v0[4 * h4 + 1], 0.f), s);
            s = fmaf(wv.z, fmaxf(v0[4 * h4 + 2], 0.f), s);
            s = fmaf(wv.w, fmaxf(v0[4 * h4 + 3], 0.f), s);
          }
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wv = w4[8 + h4];
            s = fmaf(wv.x, fmaxf(v1[4 * h4], 0.f), s);
            s = fmaf(wv.y, fmaxf(v1[4 * h4 + 1], 0.f), s);
            s = fmaf(wv.z, fmaxf(v1[4 * h4 + 2], 0.f), s);
            s = fmaf(wv.w, fmaxf(v1[4 * h4 + 3], 0.f), s);
          }
          int ne = ne_q[0];                           // ne_q[q] without a local-memory index
#pragma unroll
          for (int x = 1; x < QT; ++x) ne = q == x ? ne_q[x] : ne;
          if (j < ne) a.scores[((long long)b * a.Tq + q0 + q) * a.n_cap + j] = s;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
      ++i;
    } while (walk.next(a));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
  if (a.wait_last) pdl_wait();
}

// ============================================================================ FP4
// The same GEMM with FP4 keys and queries ("DeepSeek-V4 深度研究剖析" §8: the
// Lightning Indexer computes in FP4; its scores are kept in BF16).  Key rows are
// 80 bytes (fp4.cuh); a tile of 128 entries is one 10 KiB bulk copy into a ring of
// raw tiles.  Eight converter warps widen every raw tile into an f16 operand tile
// (exact: code * scale has at most 6 significant bits), two threads per entry, in
// the 128-byte-swizzled K-major layout the MMA reads, and quantize each query
// group's bfloat16 query to FP4 and back to f16 in place (the keys' rule), so the
// tensor cores (kind::f16 with f16 operands) multiply exactly the FP4 values.  The
// MMA and the epilogue are those above; scores are written as bfloat16 (the
// float32 sum rounded to nearest even).
//   warp 0: bulk copies (raw key tiles) and the query's TMA loads
//   warp 1: MMA issuer          warps 2-5: epilogue          warps 6-13: converters
constexpr int kRawTileBytes = kTileM * fp4::kRowBytes;   // 10 KiB
constexpr int kConv = 256;                               // converter threads
constexpr int kThreads4 = 192 + kConv;

template <int QT> struct Cfg4 {
  static constexpr int N = QT * kHeads;
  static constexpr int kRaw = QT == 1 ? 8 : 6;     // raw tiles in flight
  static constexpr int kOp = 3;                    // bfloat16 operand tiles
  static constexpr int kQBuf = QT == 1 ? 2 : 1;
  static constexpr int kQBytes = N * kDim * 2;
  static constexpr int kTmemCols = 2 * N < 32 ? 32 : 2 * N;
  static constexpr size_t kSmem = 1024 + size_t(kOp) * kTileBytes + size_t(kRaw) * kRawTileBytes +
                                  size_t(kQBuf) * kQBytes + 4 * QT * kHeads * sizeof(float) + 512;
};
static_assert(Cfg4<1>::kSmem <= 232448 && Cfg4<4>::kSmem <= 232448, "shared-memory budget");

// Quantize one 16-element group of a bfloat16 operand row to FP4 and write it back
// in place as f16: its two 16-byte chunks sit at p0 and p1 of a swizzled tile.
__device__ __forceinline__ void requantize16(uint4* p0, uint4* p1) {
  float x[16];
  const uint4 a = *p0, b = *p1;
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  uint32_t sbyte;
  float sv;
  float lo[8], hi[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) { lo[i] = x[i]; hi[i] = x[8 + i]; }
  const uint32_t c0 = fp4::quantize8(lo, amax, sbyte, sv);
  const uint32_t c1 = fp4::quantize8(hi, amax, sbyte, sv);
  const __half h = fp4::e4m3_to_half(sbyte);
  const __half2 s2 = __halves2half2(h, h);
  *p0 = fp4::decode8_half(c0, s2);
  *p1 = fp4::decode8_half(c1, s2);
}

template <int QT>
__global__ void __launch_bounds__(kThreads4, 1)
    index_scores_fp4(const __grid_constant__ CUtensorMap map_q, const unsigned char* __restrict__ cki4,
                     IdxArgs a) {
  using C = Cfg4<QT>;
  if (a.wait_last) pdl_release();
  else pdl_wait_then_release();
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* s_op = base;                                     // kOp x 32 KiB
  unsigned char* s_q = s_op + size_t(C::kOp) * kTileBytes;        // kQBuf x QT x 16 KiB
  unsigned char* s_raw = s_q + size_t(C::kQBuf) * C::kQBytes;     // kRaw x 10 KiB
  float* s_w = reinterpret_cast<float*>(s_raw + size_t(C::kRaw) * kRawTileBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_w + 4 * QT * kHeads);
  uint64_t* raw_full = bars;                      // [kRaw]
  uint64_t* raw_empty = raw_full + C::kRaw;       // [kRaw]
  uint64_t* op_full = raw_empty + C::kRaw;        // [kOp]
  uint64_t* op_empty = op_full + C::kOp;          // [kOp]
  uint64_t* acc_full = op_empty + C::kOp;         // [2]
  uint64_t* acc_empty = acc_full + 2;             // [2]
  uint64_t* q_full = acc_empty + 2;               // [kQBuf] TMA of the bfloat16 query
  uint64_t* q_ready = q_full + C::kQBuf;          // [kQBuf] query requantized
  uint64_t* q_empty = q_ready + C::kQBuf;         // [kQBuf]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_empty + C::kQBuf);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  TileWalk<QT> walk;
  const bool have = walk.init(a);      // identical in every warp
  if (!have) {
    if (a.wait_last) pdl_wait();
    return;                            // CTA-uniform
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kRaw; ++s) { tc::mbar_init(&raw_full[s], 1); tc::mbar_init(&raw_empty[s], kConv); }
    for (int s = 0; s < C::kOp; ++s) { tc::mbar_init(&op_full[s], kConv); tc::mbar_init(&op_empty[s], 1); }
    for (int i = 0; i < 2; ++i) { tc::mbar_init(&acc_full[i], 1); tc::mbar_init(&acc_empty[i], 4); }
    for (int i = 0; i < C::kQBuf; ++i) {
      tc::mbar_init(&q_full[i], 1);
      tc::mbar_init(&q_ready[i], kConv);
      tc::mbar_init(&q_empty[i], 1);
    }
    tc::fence_mbar_init();
  }
  if (warp == 1) { tc::tmem_alloc(tmem_slot, C::kTmemCols); tc::tmem_relinquish(); }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int gpb = (a.Tq + QT - 1) / QT;

  if (warp == 0) {
    // ------------------------------------------------------------ copies
    if (lane == 0) {
      tc::tma_prefetch(&map_q);
      int i = 0, prev_g = -1, n_groups_seen = 0;
      do {
        if (walk.g != prev_g) {
          const int qb = n_groups_seen % C::kQBuf, use = n_groups_seen / C::kQBuf;
          if (use > 0 && !tc::mbar_wait(&q_empty[qb], (use - 1) & 1, a.err, 61)) break;
          const int b = walk.g / gpb, q0 = (walk.g % gpb) * QT;
          const int y = (b * a.Tq + q0) * kHeads;
          unsigned char* qdst = s_q + size_t(qb) * C::kQBytes;
          tc::mbar_expect_tx(&q_full[qb], C::kQBytes);
          tc::tma_load_2d(qdst, &map_q, 0, y, &q_full[qb]);
          tc::tma_load_2d(qdst + C::kQBytes / 2, &map_q, 64, y, &q_full[qb]);
          prev_g = walk.g;
          ++n_groups_seen;
        }
        const int s = i % C::kRaw;
        if (!tc::mbar_wait(&raw_empty[s], ((i / C::kRaw) & 1) ^ 1, a.err, 62)) break;
        const int b = walk.g / gpb;
        // rows of this sequence only (the last tile of a sequence may be partial)
        const int rows = min(kTileM, a.n_cap - walk.t * kTileM);
        const uint32_t bytes = uint32_t(rows) * fp4::kRowBytes;
        tc::mbar_expect_tx(&raw_full[s], bytes);
        tc::bulk_load(s_raw + size_t(s) * kRawTileBytes,
                      cki4 + ((long long)b * a.n_cap + (long long)walk.t * kTileM) * fp4::kRowBytes,
                      bytes, &raw_full[s]);
        ++i;
      } while (walk.next(a));
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_f16_f32(kTileM, C::N);   // keys and query both f16
      const uint32_t op_base = tc::smem_u32(s_op);
      uint32_t q_base = tc::smem_u32(s_q);
      int i = 0, prev_g = -1, n_groups_seen = 0, qb = 0;
      do {
        if (walk.g != prev_g) {
          qb = n_groups_seen % C::kQBuf;
          if (!tc::mbar_wait(&q_ready[qb], (n_groups_seen / C::kQBuf) & 1, a.err, 63)) break;
          q_base = tc::smem_u32(s_q + size_t(qb) * C::kQBytes);
          prev_g = walk.g;
          ++n_groups_seen;
        }
        const int so = i % C::kOp, acc = i & 1;
        if (!tc::mbar_wait(&op_full[so], (i / C::kOp) & 1, a.err, 64)) break;
        if (!tc::mbar_wait(&acc_empty[acc], ((i >> 1) & 1) ^ 1, a.err, 65)) break;
        tc::fence_after_sync();
        const uint32_t kb = op_base + so * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kDim / 16; ++kk) {
          const uint32_t off_k = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          const uint32_t off_q = (kk >> 2) * (C::kQBytes / 2) + (kk & 3) * 32;
          tc::mma_bf16(tmem + acc * C::N, tc::sdesc_kmajor_sw128(kb + off_k),
                       tc::sdesc_kmajor_sw128(q_base + off_q), idesc, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(&op_empty[so]);
        tc::mma_commit(&acc_full[acc]);
        if (walk.last_of_group()) tc::mma_commit(&q_empty[qb]);
        ++i;
      } while (walk.next(a));
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ converters (warps 6-13)
    const int ct = threadIdx.x - 192;                 // 0..255
    const int crow = ct >> 1, chalf = ct & 1;         // tile row, its 64-dim half
    int i = 0, prev_g = -1, n_groups_seen = 0;
    bool ok = true;
    do {
      if (walk.g != prev_g) {
        // the group's query: bfloat16 from TMA, requantized in place (N rows x 8 groups)
        const int qb = n_groups_seen % C::kQBuf;
        ok = tc::mbar_wait(&q_full[qb], (n_groups_seen / C::kQBuf) & 1, a.err, 66);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        unsigned char* q = s_q + size_t(qb) * C::kQBytes;
        for (int gi = ct; gi < C::N * (kDim / fp4::kGroup); gi += kConv) {
          const int n = gi >> 3, g = gi & 7;            // query row, 16-element group
          unsigned char* half = q + (g >> 2) * (C::kQBytes / 2) + n * 128;
          const int c0 = (g & 3) * 2;                     // 16-byte chunk within the 128 B row
          requantize16(reinterpret_cast<uint4*>(half + ((c0 ^ (n & 7)) << 4)),
                       reinterpret_cast<uint4*>(half + (((c0 + 1) ^ (n & 7)) << 4)));
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&q_ready[qb]);
        prev_g = walk.g;
        ++n_groups_seen;
      }
      const int s = i % C::kRaw, so = i % C::kOp;
      ok = tc::mbar_wait(&raw_full[s], (i / C::kRaw) & 1, a.err, 67) &&
           tc::mbar_wait(&op_empty[so], ((i / C::kOp) & 1) ^ 1, a.err, 68);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc::fence_after_sync();
      // half chalf of row crow of the raw tile (rows past the sequence's end hold
      // stale bytes: their scores are never written) -> 128 bytes of f16 in the
      // swizzled tile
      const unsigned char* src = s_raw + size_t(s) * kRawTileBytes + crow * fp4::kRowBytes;
      const uint4 ca = *reinterpret_cast<const uint4*>(src + 32 * chalf);        // 32 dims
      const uint4 cb = *reinterpret_cast<const uint4*>(src + 32 * chalf + 16);   // 32 dims
      const uint32_t sw = *reinterpret_cast<const uint32_t*>(src + 64 + 4 * chalf);  // 4 scales
      const uint32_t codes[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
      unsigned char* dst = s_op + size_t(so) * kTileBytes + chalf * (kTileBytes / 2) + crow * 128;
#pragma unroll
      for (int g = 0; g < 4; ++g) {                   // 16-element groups of this half
        const __half h = fp4::e4m3_to_half((sw >> (8 * g)) & 0xffu);
        const __half2 s2 = __halves2half2(h, h);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int cc = 2 * g + e;                   // 16-byte chunk within the 128 B row
          *reinterpret_cast<uint4*>(dst + ((cc ^ (crow & 7)) << 4)) = fp4::decode8_half(codes[cc], s2);
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&op_full[so]);
      tc::mbar_arrive(&raw_empty[s]);
      ++i;
    } while (walk.next(a));
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    float* w_mine = s_w + (warp - 2) * QT * kHeads;
    int ne_q[QT];
    float w_reg[QT == 1 ? kHeads : 1];
    __nv_bfloat16* scores = reinterpret_cast<__nv_bfloat16*>(a.scores);
    int i = 0, prev_g = -1;
    bool ok = true;
    do {
      const int b = walk.g / gpb, q0 = (walk.g % gpb) * QT;
      if (walk.g != prev_g) {
        __syncwarp();
        for (int x = lane; x < QT * kHeads; x += 32) {
          const int q = x / kHeads;
          w_mine[x] = (q0 + q < a.Tq) ? a.w[(long long)(b * a.Tq + q0 + q) * kHeads + x % kHeads] : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int q = 0; q < QT; ++q)
          ne_q[q] = q0 + q < a.Tq
                        ? n_eligible(a.q_pos[b * a.Tq + q0 + q] + a.pos_off, a.n_win, a.m, a.elig, a.n_cap)
                        : 0;
        if constexpr (QT == 1) {
#pragma unroll
          for (int h = 0; h < kHeads; ++h) w_reg[h] = w_mine[h];
        }
        prev_g = walk.g;
      }
      const int acc = i & 1;
      ok = tc::mbar_wait(&acc_full[acc], (i >> 1) & 1, a.err, 69);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc::fence_after_sync();
      const int j = walk.t * kTileM + row;
      if constexpr (QT == 1) {
        float v0[32], v1[32];
        tc::tmem_ld32x2(tmem + (uint32_t(quarter * 32) << 16) + acc * C::N,
                        tmem + (uint32_t(quarter * 32) << 16) + acc * C::N + 32, v0, v1);
        float s = 0.f;
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(w_reg[h], fmaxf(v0[h], 0.f), s);
#pragma unroll
        for (int h = 0; h < 32; ++h) s = fmaf(w_reg[32 + h], fmaxf(v1[h], 0.f), s);
        if (j < ne_q[0]) scores[((long long)b * a.Tq + q0) * a.n_cap + j] = __float2bfloat16_rn(s);
      } else {
#pragma unroll
        for (int q = 0; q < QT; ++q) {
          float s = 0.f;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float v[32];
            tc::tmem_ld32(tmem + (uint32_t(quarter * 32) << 16) + acc * C::N + q * kHeads + half * 32, v);
#pragma unroll
            for (int h = 0; h < 32; ++h) s = fmaf(w_mine[q * kHeads + half * 32 + h], fmaxf(v[h], 0.f), s);
          }
          if (j < ne_q[q])
            scores[((long long)b * a.Tq + q0 + q) * a.n_cap + j] = __float2bfloat16_rn(s);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
      ++i;
    } while (walk.next(a));
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, C::kTmemCols);
  if (a.wait_last) pdl_wait();
}

int g_num_sms = 0;

template <int QT>
cudaError_t launch_qt(const ha_params& p, const void* q_idx, const float* w_idx, const void* cki,
                      int n_cap, const int32_t* q_pos, int Tq, void* scores, int* err,
                      cudaStream_t st, const StepOpts& so) {
  using C = Cfg<QT>;
  CUtensorMap map_k, map_q;
  cudaError_t e = make_tmap_bf16_2d(&map_k, cki, kDim, uint64_t(p.B) * n_cap, kDim * 2, 64, kTileM);
  if (e != cudaSuccess) return e;
  e = make_tmap_bf16_2d(&map_q, q_idx, kDim, uint64_t(p.B) * Tq * kHeads, kDim * 2, 64, C::N);
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(index_scores_tc<QT>), C::kSmem);
  if (e != cudaSuccess) return e;
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    e = cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  IdxArgs a{w_idx, q_pos, static_cast<float*>(scores), p.B, Tq, n_cap, p.n_win, p.m, p.elig, err,
            so.pos_off, so.wait_last};
  return launch_pdl(index_scores_tc<QT>, dim3(g_num_sms), dim3(C::kThreadsQ), C::kSmem, st, 1, map_k,
                    map_q, a);
}

int num_sms_idx() {
  if (g_num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      g_num_sms = 148;
  }
  return g_num_sms;
}

template <int QT>
cudaError_t launch_qt4(const ha_params& p, const void* q_idx, const float* w_idx, const void* cki,
                       int n_cap, const int32_t* q_pos, int Tq, void* scores, int* err,
                       cudaStream_t st, const StepOpts& so) {
  using C = Cfg4<QT>;
  CUtensorMap map_q;
  cudaError_t e = make_tmap_bf16_2d(&map_q, q_idx, kDim, uint64_t(p.B) * Tq * kHeads, kDim * 2, 64, C::N);
  if (e != cudaSuccess) return e;
  e = ensure_smem(reinterpret_cast<const void*>(index_scores_fp4<QT>), C::kSmem);
  if (e != cudaSuccess) return e;
  IdxArgs a{w_idx, q_pos, static_cast<float*>(scores), p.B, Tq, n_cap, p.n_win, p.m, p.elig, err,
            so.pos_off, so.wait_last};
  return launch_pdl(index_scores_fp4<QT>, dim3(num_sms_idx()), dim3(kThreads4), C::kSmem, st, 1,
                    map_q, static_cast<const unsigned char*>(cki), a);
}

}  // namespace

bool index_scores_tc_supported(const ha_params& p, const void* q_idx, const void* cki) {
  return p.dtype == HA_BF16 && p.H_I == kHeads && p.d_I == kDim &&
         (reinterpret_cast<uintptr_t>(q_idx) & 15) == 0 && (reinterpret_cast<uintptr_t>(cki) & 15) == 0;
}

cudaError_t launch_index_scores_tc(const ha_params& p, const void* q_idx, const float* w_idx,
                                   const void* cki, int n_cap, const int32_t* q_pos, int Tq,
                                   void* scores, int* err, cudaStream_t st, const StepOpts& so) {
  if (p.fmt & HA_FMT_IDX4) {
    if (Tq >= 4) return launch_qt4<4>(p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores, err, st, so);
    return launch_qt4<1>(p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores, err, st, so);
  }
  if (Tq >= 4) return launch_qt<4>(p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores, err, st, so);
  return launch_qt<1>(p, q_idx, w_idx, cki, n_cap, q_pos, Tq, scores, err, st, so);
}

}  // namespace ha
