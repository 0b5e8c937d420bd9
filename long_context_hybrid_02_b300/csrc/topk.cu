// Per-query top-k of the indexer scores ("DeepSeek-V4 深度研究剖析" §5.3: the top-k
// compressed entries are attended, k = 512 for V4-Flash and 1024 for V4-Pro).
//
// Exact radix select over order-preserving 32-bit keys of the float scores (NaN
// ranks as -inf).  One CTA of 1024 threads per row:
//   1. four passes over 8-bit digits, most significant first, build a histogram of
//      the keys that still match the selected prefix (warp-aggregated shared-memory
//      atomics through __match_any_sync) and pick the digit holding the k-th
//      largest key -> the threshold key T and how many keys equal to T are needed;
//   2. one pass in ascending index order keeps every key > T and the first
//      `need` keys == T (block-wide prefix sums of warp ballots), which realises
//      the tie rule "larger score, then smaller index" and writes the result in
//      ascending index order without a sort.
// Rows of up to kSmemKeys keys are held in shared memory; longer rows are re-read
// from global memory (L2) on every pass.
#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

constexpr int kThreads = 1024;
constexpr int kSmemKeys = 48 * 1024;

// Exclusive prefix sum of v over the CTA; returns the prefix, total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = warp_tot[lane];
    int s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_tot[lane] = s - t;                 // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = s;
  }
  __syncthreads();
  const int res = warp_tot[wid] + x - v;
  *total = warp_tot[32];
  __syncthreads();                          // warp_tot reusable after return
  return res;
}

__global__ void __launch_bounds__(kThreads) topk_rows(const float* __restrict__ scores, int n_cap,
                                                      const int32_t* __restrict__ q_pos, int k,
                                                      int n_win, int m, int elig,
                                                      int32_t* __restrict__ idx) {
  extern __shared__ uint32_t skeys[];
  __shared__ int hist[256];
  __shared__ int warp_tot[33];
  __shared__ int sel_digit, sel_above;
  if (threadIdx.x == 0) { sel_digit = 0; sel_above = 0; }
  const int row = blockIdx.x;
  const int t = q_pos[row];
  const int n = n_eligible(t, n_win, m, elig, n_cap);
  int32_t* out = idx + (long long)row * k;
  if (n <= k) {
    for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* s = scores + (long long)row * n_cap;
  const bool in_smem = n <= kSmemKeys;
  if (in_smem) {
    for (int i = threadIdx.x; i < n; i += kThreads) skeys[i] = score_key(s[i]);
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint32_t { return in_smem ? skeys[i] : score_key(__ldg(s + i)); };

  uint32_t prefix = 0, pmask = 0;
  int remaining = k;                        // how many of the selected still to place
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < n; base += kThreads) {
      const int i = base + threadIdx.x;
      const bool valid = i < n;
      const uint32_t key = valid ? key_at(i) : 0u;
      const bool match = valid && ((key & pmask) == prefix);
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const uint32_t digit = (key >> shift) & 0xffu;
        const unsigned peers = __match_any_sync(act, digit);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns bins 255-8l .. 248-8l (descending); find the bin where the
      // running count from the top reaches `remaining`
      const int lane = threadIdx.x;
      int c[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { c[q] = hist[255 - 8 * lane - q]; tot += c[q]; }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      if (excl < remaining && remaining <= incl) {
        int run = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run < remaining && remaining <= run + c[q]) { sel_digit = 255 - 8 * lane - q; sel_above = run; }
          run += c[q];
        }
      }
    }
    __syncthreads();
    prefix |= uint32_t(sel_digit) << shift;
    pmask |= 0xffu << shift;
    remaining -= sel_above;
    __syncthreads();
  }
  // prefix is now the k-th largest key; `remaining` keys equal to it are taken.
  const uint32_t thr = prefix;
  const int need_eq = remaining;
  int eq_before = 0, out_before = 0;
  for (int base = 0; base < n; base += kThreads) {
    const int i = base + threadIdx.x;
    const uint32_t key = i < n ? key_at(i) : 0u;
    const int is_eq = (i < n && key == thr) ? 1 : 0;
    int eq_tot;
    const int eq_rank = eq_before + block_exclusive_scan(is_eq, warp_tot, &eq_tot);
    const int take = (i < n && (key > thr || (is_eq && eq_rank < need_eq))) ? 1 : 0;
    int take_tot;
    const int pos = out_before + block_exclusive_scan(take, warp_tot, &take_tot);
    if (take && pos < k) out[pos] = i;
    eq_before += eq_tot;
    out_before += take_tot;
  }
}

}  // namespace

size_t topk_workspace_bytes(const ha_params&, int, int) { return 0; }

cudaError_t launch_topk(const ha_params& p, const float* scores, int n_cap, const int32_t* q_pos,
                        int Tq, int32_t* idx, void*, size_t, cudaStream_t st) {
  const size_t smem = size_t(n_cap < kSmemKeys ? n_cap : kSmemKeys) * sizeof(uint32_t);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(topk_rows), smem);
  if (e != cudaSuccess) return e;
  topk_rows<<<p.B * Tq, kThreads, smem, st>>>(scores, n_cap, q_pos, p.k, p.n_win, p.m, p.elig, idx);
  return launched(cudaGetLastError());
}

}  // namespace ha
