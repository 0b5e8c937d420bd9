// The FP8 KV format of the compressed caches ("DeepSeek-V4 深度研究剖析" §8: the KV
// cache keeps its RoPE dims in BF16 and the other dims in FP8).  A compressed K or V
// row of d = 512 is 608 bytes: dims 0..63 as bfloat16 (128 B), dims 64..511 as
// e4m3fn codes (448 B), one float32 scale per 64-dim group (28 B), 4 zero bytes;
// element value = code * scale.
//
// The attention's tensor cores take bfloat16 operands, so before an attention call
// kv8_expand widens exactly the rows that call reads into bfloat16 rows of the
// workspace: value = code * scale rounded to bfloat16 (nearest even), the RoPE
// dims copied.  Decode over a selection (CSA) widens the selected entries and
// packs them to the front of a per-row list in slot order, with an index list 0,
// 1, .. (-1 after the last), so that the attention reads them as entries 0 ..
// count-1; every other call widens every entry of the cache.  One warp per row,
// 16-byte loads and stores, no conversion of the 60 % of bytes it does not need.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

constexpr int kRows = 64;            // list slots (or entries) per CTA
constexpr int kThreadsX = 256;

// Eight e4m3fn codes (8 bytes) times scale, as 8 bfloat16 (16 bytes).
__device__ __forceinline__ uint4 widen8(uint2 codes, float scale) {
  uint32_t out[4];
  const uint32_t w[2] = {codes.x, codes.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t pair = uint16_t(w[i >> 1] >> (16 * (i & 1)));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));   // exact
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
    const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
    out[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// One lane's two 16-byte chunks of a widened row: chunk lane (RoPE dims copied when
// lane < 8, else 8 codes) and chunk lane + 32 (8 codes); loads and stores apart, so
// that a warp can have the loads of several rows in flight.
struct LaneChunks {
  uint4 rope;        // lane < 8
  uint2 c0, c1;      // codes of chunks lane (lane >= 8) and lane + 32
  float s0, s1;      // their scales
};
__device__ __forceinline__ void load_chunks(const unsigned char* src, int lane, LaneChunks& x) {
  if (lane < 8) {
    x.rope = __ldg(reinterpret_cast<const uint4*>(src) + lane);
  } else {
    x.c0 = __ldg(reinterpret_cast<const uint2*>(src + 128 + 8 * (lane - 8)));
    x.s0 = __ldg(reinterpret_cast<const float*>(src + 576) + (lane - 8) / 8);
  }
  x.c1 = __ldg(reinterpret_cast<const uint2*>(src + 128 + 8 * (lane + 24)));
  x.s1 = __ldg(reinterpret_cast<const float*>(src + 576) + (lane + 24) / 8);
}
__device__ __forceinline__ void store_chunks(__nv_bfloat16* dst, int lane, const LaneChunks& x) {
  reinterpret_cast<uint4*>(dst)[lane] = lane < 8 ? x.rope : widen8(x.c0, x.s0);
  reinterpret_cast<uint4*>(dst)[lane + 32] = widen8(x.c1, x.s1);
}

struct ExpandArgs {
  const unsigned char* ck8;   // [B, n_cap, 608]
  const unsigned char* cv8;
  const int32_t* idx;         // [rows, k] or null (widen every entry)
  const int32_t* pos;         // decode: ctx_len [B]
  int n_cap, k, n_win, m, elig;
  __nv_bfloat16* ck;          // [B, n_out, 512]: n_out = k (selection) or n_cap
  __nv_bfloat16* cv;
  int32_t* idx_out;           // [B, k] (selection) or null
};

__global__ void __launch_bounds__(kThreadsX, 2) kv8_expand(const ExpandArgs a) {
  pdl_wait_then_release();
  __shared__ int s_cnt[kThreadsX / 32];
  __shared__ int s_w0;
  __shared__ int s_pos[kRows];
  __shared__ int s_ent[kRows];
  const int b = blockIdx.y;
  const int s0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_out = a.idx ? a.k : a.n_cap;
  if (a.idx) {
    // Valid entries of the selection: 0 <= j < min(n_elig(t), n_cap).  The output
    // position of a valid slot = valid slots before it in the row (those before s0
    // counted by the whole CTA, those of this CTA's 64 slots by ballots).
    const int t = a.pos[b] - 1;
    const int ne = t >= 0 ? n_eligible(t, a.n_win, a.m, a.elig, a.n_cap) : 0;
    const int32_t* row = a.idx + (long long)b * a.k;
    int before = 0;
    for (int s = threadIdx.x; s < s0; s += kThreadsX) {
      const int j = __ldg(row + s);
      before += (j >= 0 && j < ne) ? 1 : 0;
    }
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (lane == 0) s_cnt[warp] = before;
    int j = -1;
    bool ok = false;
    if (threadIdx.x < kRows) {
      const int s = s0 + threadIdx.x;
      j = s < a.k ? __ldg(row + s) : -1;
      ok = s < a.k && j >= 0 && j < ne;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    if (threadIdx.x < kRows) {
      s_ent[threadIdx.x] = ok ? j : -1;
      s_pos[threadIdx.x] = __popc(bal & ((1u << lane) - 1u));
    }
    if (threadIdx.x == 0) s_w0 = __popc(bal);
    __syncthreads();
    int base = 0;
    for (int w = 0; w < kThreadsX / 32; ++w) base += s_cnt[w];
    if (threadIdx.x < kRows) s_pos[threadIdx.x] += base + (threadIdx.x >= 32 ? s_w0 : 0);
    __syncthreads();
  }
  // this CTA's rows: (entry, output position) pairs; warp w widens rows w, w + 8,
  // .. of K, then of V, with every row's loads issued before the first store
  constexpr int kPerWarp = kRows / (kThreadsX / 32);
  long long src_row[kPerWarp], dst_row[kPerWarp];
  bool live[kPerWarp];
#pragma unroll
  for (int i = 0; i < kPerWarp; ++i) {
    const int r = warp + i * (kThreadsX / 32);
    const int s = s0 + r;
    int j = s, p = s;
    if (a.idx && s < n_out) {
      j = s_ent[r];
      p = s_pos[r];
    }
    live[i] = s < n_out && j >= 0;
    src_row[i] = (long long)b * a.n_cap + (live[i] ? j : 0);
    dst_row[i] = (long long)b * n_out + (live[i] ? p : 0);
  }
#pragma unroll 1
  for (int tsr = 0; tsr < 2; ++tsr) {
    const unsigned char* src = tsr == 0 ? a.ck8 : a.cv8;
    __nv_bfloat16* dst = tsr == 0 ? a.ck : a.cv;
    LaneChunks x[kPerWarp];
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i)
      if (live[i]) load_chunks(src + src_row[i] * 608, lane, x[i]);
#pragma unroll
    for (int i = 0; i < kPerWarp; ++i)
      if (live[i]) store_chunks(dst + dst_row[i] * 512, lane, x[i]);
  }
}

// The index list of the packed selection: idx_out[b, s] = s for s < count(b), else
// -1, count(b) = the valid entries of the row's selection.
__global__ void __launch_bounds__(kThreadsX) kv8_index_list(const ExpandArgs a) {
  pdl_wait_then_release();
  const int b = blockIdx.x;
  const int t = a.pos[b] - 1;
  const int ne = t >= 0 ? n_eligible(t, a.n_win, a.m, a.elig, a.n_cap) : 0;
  const int32_t* row = a.idx + (long long)b * a.k;
  int cnt = 0;
  for (int s = threadIdx.x; s < a.k; s += kThreadsX) {
    const int j = __ldg(row + s);
    cnt += (j >= 0 && j < ne) ? 1 : 0;
  }
  __shared__ int s_red[kThreadsX / 32];
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = cnt;
  __syncthreads();
  int total = 0;
  for (int w = 0; w < kThreadsX / 32; ++w) total += s_red[w];
  for (int s = threadIdx.x; s < a.k; s += kThreadsX) a.idx_out[(long long)b * a.k + s] = s < total ? s : -1;
}

}  // namespace

size_t kv8_expand_bytes(const ha_params& p, int n_cap, bool select) {
  const size_t rows = size_t(p.B) * (select ? p.k : n_cap);
  return rows * 2 * 512 * 2 + (select ? size_t(p.B) * p.k * 4 : 0) + 256;
}

cudaError_t launch_kv8_expand(const ha_params& p, const void* ck8, const void* cv8, int n_cap,
                              const int32_t* idx, const int32_t* ctx_len, void* ws,
                              KvExpanded* out, cudaStream_t st) {
  ExpandArgs a{};
  a.ck8 = static_cast<const unsigned char*>(ck8);
  a.cv8 = static_cast<const unsigned char*>(cv8);
  a.idx = idx;
  a.pos = ctx_len;
  a.n_cap = n_cap;
  a.k = p.k;
  a.n_win = p.n_win;
  a.m = p.m;
  a.elig = p.elig;
  const bool select = idx != nullptr;
  const int n_out = select ? p.k : n_cap;
  a.ck = static_cast<__nv_bfloat16*>(ws);
  a.cv = a.ck + size_t(p.B) * n_out * 512;
  a.idx_out = select ? reinterpret_cast<int32_t*>(a.cv + size_t(p.B) * n_out * 512) : nullptr;
  const dim3 grid(unsigned((n_out + kRows - 1) / kRows), unsigned(p.B));
  cudaError_t e = launch_pdl(kv8_expand, grid, dim3(kThreadsX), 0, st, 1u, a);
  if (e != cudaSuccess) return e;
  if (select) {
    e = launch_pdl(kv8_index_list, dim3(unsigned(p.B)), dim3(kThreadsX), 0, st, 1u, a);
    if (e != cudaSuccess) return e;
  }
  out->ck = a.ck;
  out->cv = a.cv;
  out->n_cap = n_out;
  out->idx = a.idx_out;
  return cudaSuccess;
}

}  // namespace ha
