// Per-query top-k of the indexer scores ("DeepSeek-V4 深度研究剖析" §5.3: the top-k
// compressed entries are attended, k = 512 for V4-Flash and 1024 for V4-Pro).
//
// Exact radix select over order-preserving 32-bit keys of the float scores (NaN
// ranks as -inf, -0 as +0), digits of 11, 11 and 10 bits from the top; ties go to
// the smaller index; the output is in ascending index order.
//
// A row of at most kRowMaxKeys entries (decode up to ~160K tokens, every prefill
// row of a 128K context) is handled by one 1024-thread CTA (topk_row): the keys
// go to shared memory once; a strided sample of 1,024 keys gives a threshold; the
// keys at or above it are compacted in index order and the digit passes run on
// those candidates only, stopping once every key of the selected bin is needed;
// when the sample misjudged the row the passes run over every key and the write
// goes through bitmaps of the keys above / equal to the threshold prefix.
//
// A longer row (decode at 1M tokens: 262,112 entries) is cut into segments of at
// most kRowMaxKeys keys (topk_seg, one CTA each, then topk_seg_merge, one CTA per
// row; see there).  Rows longer than kMaxSegRowKeys are not supported.
#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

constexpr int kBins = 2048;

// Inclusive scan of v over the CTA (NT threads); returns the inclusive prefix and
// the total in *total.  `scratch` holds NT / 32 + 1 ints.
template <int NT, typename T>
__device__ __forceinline__ T block_inclusive_scan(T v, T* scratch, T* total) {
  constexpr int kWarps = NT / 32;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[wid] = x;
  __syncthreads();
  if (wid == 0) {
    const T t = lane < kWarps ? scratch[lane] : T(0);
    T s = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < kWarps) scratch[lane] = s - t;   // exclusive prefix of warp totals
    if (lane == kWarps - 1) scratch[kWarps] = s;
  }
  __syncthreads();
  const T res = scratch[wid] + x;
  *total = scratch[kWarps];
  __syncthreads();
  return res;
}

// A score as float: float32 scores, or bfloat16 scores (the FP4 indexer's), widened
// exactly, so the same order-preserving keys serve both.
__device__ __forceinline__ float score_at(const float* s, long long i) { return __ldg(s + i); }
__device__ __forceinline__ float score_at(const __nv_bfloat16* s, long long i) {
  return __uint_as_float(uint32_t(__ldg(reinterpret_cast<const unsigned short*>(s) + i)) << 16);
}

// ------------------------------------------------------------------ one CTA per row
constexpr int kRowThreads = 1024;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowMaxKeys = 40 * 1024;
constexpr int kCandCap = 4096;            // candidates of the sampled threshold

struct RowShared {
  int hist[kBins];
  int scratch[kRowWarps + 1];
  int sel_digit, sel_above, sel_count;
};

// Keys are stored with one padding word per 32 so that both row-order sweeps and
// per-thread contiguous ranges read shared memory without bank conflicts.
__host__ __device__ __forceinline__ int pad32(int i) { return i + (i >> 5); }

// Dynamic shared memory of topk_row for rows of up to n_cap entries:
// keys[33 * words] | max(candidates (key, index) x kCandCap, bitmaps 2 x words).
__host__ __device__ inline size_t row_smem_bytes(int n_cap) {
  const size_t words = (size_t(n_cap) + 31) / 32;
  const size_t region = 2 * words > size_t(2) * kCandCap ? 2 * words : size_t(2) * kCandCap;
  return (words * 33 + region) * sizeof(uint32_t);
}

// sh.hist holds the histogram of the current digit over the keys still in play;
// finds the digit holding the `remaining`-th largest of them (thread t owns bins
// 2047-2t and 2046-2t, scanned from the top).  Ends with a barrier.
__device__ __forceinline__ void row_select_digit(RowShared& sh, int remaining) {
  const int b0 = kBins - 1 - 2 * int(threadIdx.x);
  const int c0 = sh.hist[b0], c1 = sh.hist[b0 - 1];
  int total;
  const int incl = block_inclusive_scan<kRowThreads, int>(c0 + c1, sh.scratch, &total);
  const int excl = incl - c0 - c1;
  if (excl < remaining && remaining <= incl) {
    const bool first = remaining <= excl + c0;
    sh.sel_digit = first ? b0 : b0 - 1;
    sh.sel_above = first ? excl : excl + c0;
    sh.sel_count = first ? c0 : c1;
  }
  __syncthreads();
}

// Adds the digit of `key` to sh.hist when `match`; every lane of the warp calls it.
__device__ __forceinline__ void row_hist_add(RowShared& sh, bool match, uint32_t digit) {
  const unsigned act = __ballot_sync(0xffffffffu, match);
  if (match) {
    const unsigned peers = __match_any_sync(act, digit);
    if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], __popc(peers));
  }
}

// Radix select of the `k`-th largest of `count` keys, key_at(i) for i < count:
// three digits (11, 11, 10 bits), stopping once every key of the selected bin is
// needed.  Returns the selected prefix and its mask; `need_eq` keys whose masked
// value equals the prefix are taken (the smallest indices), every key above it.
template <typename KeyAt>
__device__ __forceinline__ void row_radix(RowShared& sh, int count, int k, KeyAt key_at,
                                          uint32_t& prefix, uint32_t& pmask, int& need_eq) {
  prefix = 0;
  pmask = 0;
  int remaining = k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    for (int i = threadIdx.x; i < kBins; i += kRowThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < count; base += kRowThreads) {   // warp-uniform trip count
      const int i = base + int(threadIdx.x);
      const uint32_t key = i < count ? key_at(i) : 0u;
      row_hist_add(sh, i < count && (key & pmask) == prefix, (key >> shift) & dmask);
    }
    __syncthreads();
    row_select_digit(sh, remaining);
    prefix |= uint32_t(sh.sel_digit) << shift;
    pmask |= dmask << shift;
    remaining -= sh.sel_above;
    const bool all_of_bin = sh.sel_count == remaining;
    __syncthreads();
    if (all_of_bin) break;                        // uniform
  }
  need_eq = remaining;
}

template <typename S>
__global__ void __launch_bounds__(kRowThreads) topk_row(const S* __restrict__ scores,
                                                       int n_cap, const int32_t* __restrict__ q_pos,
                                                       int pos_off, int k, int n_win, int m,
                                                       int elig, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t skeys[];
  __shared__ RowShared sh;
  pdl_wait_then_release();
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = n_eligible(q_pos[row] + pos_off, n_win, m, elig, n_cap);
  int32_t* out = idx + (long long)row * k;
  if (n <= k) {                                   // every eligible entry, then -1
    for (int i = tid; i < k; i += kRowThreads) out[i] = i < n ? i : -1;
    return;
  }
  const int words = (n + 31) / 32;
  uint32_t* keys = skeys;                         // key i at pad32(i)
  uint32_t* region = skeys + words * 33;
  const S* s = scores + (long long)row * n_cap;
  // keys in, sixteen loads in flight per thread
  for (int base = 0; base < n; base += 16 * kRowThreads) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * kRowThreads + tid;
      v[u] = i < n ? score_at(s, i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * kRowThreads + tid;
      if (i < n) keys[pad32(i)] = score_key(v[u]);
    }
  }
  __syncthreads();

  // ---- threshold g from a strided sample of 1024 keys: the 22-bit prefix of the
  // sample's t-th largest key, t about twice the sample's expected share of the
  // top k plus 16, so that the keys >= g almost surely include the top k and
  // number a small multiple of k.
  {
    const uint32_t skey = keys[pad32(int((long long)tid * n / kRowThreads))];
    int srem = min(kRowThreads, 2 * int(((long long)k * kRowThreads + n - 1) / n) + 16);
    uint32_t sprefix = 0, smask = 0;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = pass == 0 ? 21 : 10;
      for (int i = tid; i < kBins; i += kRowThreads) sh.hist[i] = 0;
      __syncthreads();
      row_hist_add(sh, (skey & smask) == sprefix, (skey >> shift) & 0x7ffu);
      __syncthreads();
      row_select_digit(sh, srem);
      sprefix |= uint32_t(sh.sel_digit) << shift;
      smask |= 0x7ffu << shift;
      srem -= sh.sel_above;
      __syncthreads();
    }
    const uint32_t g = sprefix;                   // low 10 bits zero: key >= g <=> prefix >= g
    // candidates = keys >= g; thread t owns the contiguous range [t*kpt, (t+1)*kpt)
    const int kpt = (n + kRowThreads - 1) / kRowThreads;
    const int lo = min(n, tid * kpt), hi = min(n, lo + kpt);
    int c_own = 0;
    for (int i = lo; i < hi; ++i) c_own += keys[pad32(i)] >= g ? 1 : 0;
    int c_total;
    const int c_incl = block_inclusive_scan<kRowThreads, int>(c_own, sh.scratch, &c_total);
    if (c_total >= k && c_total <= kCandCap) {    // uniform
      uint32_t* ck = region;                      // candidate keys, in index order
      int* ci = reinterpret_cast<int*>(region + kCandCap);
      int c = c_incl - c_own;
      for (int i = lo; i < hi; ++i) {
        const uint32_t key = keys[pad32(i)];
        if (key >= g) { ck[c] = key; ci[c] = i; ++c; }
      }
      __syncthreads();
      uint32_t prefix, pmask;
      int need_eq;
      row_radix(sh, c_total, k, [&](int i) { return ck[i]; }, prefix, pmask, need_eq);
      // ordered write: thread t owns candidates [t*cpt, (t+1)*cpt)
      const int cpt = (c_total + kRowThreads - 1) / kRowThreads;
      const int clo = min(c_total, tid * cpt), chi = min(c_total, clo + cpt);
      unsigned cnt_gt = 0, cnt_eq = 0;
      for (int i = clo; i < chi; ++i) {
        const uint32_t km = ck[i] & pmask;
        cnt_gt += km > prefix ? 1u : 0u;
        cnt_eq += km == prefix ? 1u : 0u;
      }
      unsigned total;
      const unsigned packed = block_inclusive_scan<kRowThreads, unsigned>(
          cnt_gt | (cnt_eq << 16), reinterpret_cast<unsigned*>(sh.scratch), &total);
      int gt_before = int(packed & 0xffffu) - int(cnt_gt);
      int eq_before = int(packed >> 16) - int(cnt_eq);
      for (int i = clo; i < chi; ++i) {
        const uint32_t km = ck[i] & pmask;
        if (km > prefix) {
          out[gt_before + min(eq_before, need_eq)] = ci[i];
          ++gt_before;
        } else if (km == prefix) {
          if (eq_before < need_eq) out[gt_before + eq_before] = ci[i];
          ++eq_before;
        }
      }
      return;
    }
  }

  // ---- fallback (the sample misjudged the row): digit passes over every key, then
  // an ordered write from bitmaps of the keys above / equal to the threshold prefix
  uint32_t prefix, pmask;
  int need_eq;
  row_radix(sh, n, k, [&](int i) { return keys[pad32(i)]; }, prefix, pmask, need_eq);
  uint32_t* selw = region;
  uint32_t* tiew = region + words;
  for (int w = wid; w < words; w += kRowWarps) {
    const int i = w * 32 + lane;
    const bool valid = i < n;
    const uint32_t km = (valid ? keys[pad32(i)] : 0u) & pmask;
    const unsigned gt = __ballot_sync(0xffffffffu, valid && km > prefix);
    const unsigned eq = __ballot_sync(0xffffffffu, valid && km == prefix);
    if (lane == 0) { selw[w] = gt; tiew[w] = eq; }
  }
  __syncthreads();
  // thread t owns words [t*per, (t+1)*per); one scan of the packed counts
  // (selected | tied << 16: both totals are at most n < 65536)
  const int per = (words + kRowThreads - 1) / kRowThreads;
  const int w_lo = min(words, tid * per), w_hi = min(words, w_lo + per);
  unsigned cnt_gt = 0, cnt_eq = 0;
  for (int w = w_lo; w < w_hi; ++w) { cnt_gt += __popc(selw[w]); cnt_eq += __popc(tiew[w]); }
  unsigned total;
  const unsigned packed = block_inclusive_scan<kRowThreads, unsigned>(
      cnt_gt | (cnt_eq << 16), reinterpret_cast<unsigned*>(sh.scratch), &total);
  int gt_before = int(packed & 0xffffu) - int(cnt_gt);
  int eq_before = int(packed >> 16) - int(cnt_eq);
  for (int w = w_lo; w < w_hi; ++w) {
    const uint32_t gt = selw[w], eq = tiew[w];
    const int taken_before = min(eq_before, need_eq);
    const int take = min(need_eq - taken_before, __popc(eq));
    uint32_t rest = eq, kept = 0;                 // the `take` lowest set bits of eq
    for (int j = 0; j < take; ++j) { const uint32_t lsb = rest & (0u - rest); kept |= lsb; rest ^= lsb; }
    int pos = gt_before + taken_before;
    for (uint32_t bits = gt | kept; bits; bits &= bits - 1) out[pos++] = w * 32 + __ffs(bits) - 1;
    gt_before += __popc(gt);
    eq_before += __popc(eq);
  }
}

// ------------------------------------------------------------------ long rows in segments
// A row longer than one CTA's shared memory holds (decode at 1M tokens: 262,112
// entries) is cut into segments of at most kRowMaxKeys keys.  topk_seg (one CTA
// per segment) keeps the keys of its segment at or above a local threshold g_s
// taken from a strided sample, in index order, in the workspace; topk_seg_merge
// (one CTA per row) selects the k largest of the row's candidates, which the
// concatenation of the segments' lists gives in index order.  The result is the
// row's exact top k whenever the selected threshold prefix is >= every g_s (then
// no key left out by a segment can be selected); otherwise, or when a list
// overflows, the row is selected again from all of its scores.
constexpr int kSegCap = 2048;            // candidates one segment keeps
constexpr int kMergeCap = 12288;         // candidates of a row the merge holds

struct SegMeta {
  int count;                             // > kSegCap: the segment's list overflowed
  uint32_t g;                            // the segment's threshold (0 for an empty segment)
};

template <typename S>
__global__ void __launch_bounds__(kRowThreads) topk_seg(const S* __restrict__ scores,
                                                       int n_cap, const int32_t* __restrict__ q_pos,
                                                       int pos_off, int k, int n_win, int m,
                                                       int elig, int C,
                                                       int seg_len, SegMeta* __restrict__ meta,
                                                       uint2* __restrict__ cand) {
  extern __shared__ uint32_t skeys[];
  __shared__ RowShared sh;
  pdl_wait_then_release();
  const int row = blockIdx.x / C, c = blockIdx.x % C;
  const int tid = threadIdx.x;
  const int n = n_eligible(q_pos[row] + pos_off, n_win, m, elig, n_cap);
  const int lo = min(n, c * seg_len), hi = min(n, lo + seg_len), len = hi - lo;
  if (n <= k || len == 0) {                       // nothing to keep
    if (tid == 0) meta[blockIdx.x] = SegMeta{0, 0u};
    return;
  }
  uint32_t* keys = skeys;                         // key i of the segment at pad32(i)
  const S* s = scores + (long long)row * n_cap + lo;
  for (int base = 0; base < len; base += 16 * kRowThreads) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * kRowThreads + tid;
      v[u] = i < len ? score_at(s, i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * kRowThreads + tid;
      if (i < len) keys[pad32(i)] = score_key(v[u]);
    }
  }
  __syncthreads();
  // local threshold: the 22-bit prefix of the sample's t-th largest key, t about
  // twice the sample's share of the segment's expected part of the top k, plus 16
  const long long share = ((long long)k * len + n - 1) / n;
  int srem = int(min(1024LL, 2 * ((share * kRowThreads + len - 1) / len) + 16));
  const uint32_t skey = keys[pad32(int((long long)tid * len / kRowThreads))];
  uint32_t g = 0, smask = 0;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 21 : 10;
    for (int i = tid; i < kBins; i += kRowThreads) sh.hist[i] = 0;
    __syncthreads();
    row_hist_add(sh, (skey & smask) == g, (skey >> shift) & 0x7ffu);
    __syncthreads();
    row_select_digit(sh, srem);
    g |= uint32_t(sh.sel_digit) << shift;
    smask |= 0x7ffu << shift;
    srem -= sh.sel_above;
    __syncthreads();
  }
  // candidates (keys >= g) in index order: thread t owns [t*kpt, (t+1)*kpt)
  const int kpt = (len + kRowThreads - 1) / kRowThreads;
  const int a = min(len, tid * kpt), b = min(len, a + kpt);
  int own = 0;
  for (int i = a; i < b; ++i) own += keys[pad32(i)] >= g ? 1 : 0;
  int total;
  const int incl = block_inclusive_scan<kRowThreads, int>(own, sh.scratch, &total);
  if (total <= kSegCap) {
    uint2* out = cand + (long long)blockIdx.x * kSegCap;
    int pos = incl - own;
    for (int i = a; i < b; ++i) {
      const uint32_t key = keys[pad32(i)];
      if (key >= g) out[pos++] = make_uint2(key, uint32_t(lo + i));
    }
  }
  if (tid == 0) meta[blockIdx.x] = SegMeta{total, g};
}

template <typename S>
__global__ void __launch_bounds__(kRowThreads) topk_seg_merge(
    const S* __restrict__ scores, int n_cap, const int32_t* __restrict__ q_pos, int pos_off,
    int k, int n_win, int m, int elig, int C, const SegMeta* __restrict__ meta,
    const uint2* __restrict__ cand, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t smem[];
  __shared__ RowShared sh;
  __shared__ int s_flag;
  __shared__ uint32_t s_gmax;
  pdl_wait_then_release();
  const int row = blockIdx.x, tid = threadIdx.x;
  const int n = n_eligible(q_pos[row] + pos_off, n_win, m, elig, n_cap);
  int32_t* out = idx + (long long)row * k;
  if (n <= k) {
    for (int i = tid; i < k; i += kRowThreads) out[i] = i < n ? i : -1;
    return;
  }
  uint32_t* ck = smem;                            // candidate keys, in index order
  int* ci = reinterpret_cast<int*>(smem + kMergeCap);
  int* seg_off = ci + kMergeCap;                  // [C + 1]
  if (tid == 0) { s_flag = 1; s_gmax = 0u; }
  __syncthreads();
  // segment counts -> offsets (C <= kRowThreads)
  int cnt = 0;
  if (tid < C) {
    const SegMeta mt = meta[(long long)row * C + tid];
    cnt = mt.count;
    if (cnt > kSegCap) s_flag = 0;
    atomicMax(&s_gmax, mt.g);
  }
  int total;
  const int incl = block_inclusive_scan<kRowThreads, int>(min(cnt, kSegCap + 1), sh.scratch, &total);
  if (tid < C) seg_off[tid] = incl - min(cnt, kSegCap + 1);
  if (tid == 0) seg_off[C] = total;
  __syncthreads();
  const bool lists_ok = s_flag != 0 && total >= k && total <= kMergeCap;   // uniform
  if (lists_ok) {
    // every candidate slot finds its segment (binary search over the offsets), so
    // that all loads of the row's lists are in flight at once
    for (int base = 0; base < total; base += 4 * kRowThreads) {
      uint2 v[4];
      int at[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pos = base + u * kRowThreads + tid;
        at[u] = pos;
        if (pos < total) {
          int lo_s = 0, hi_s = C - 1;                 // last segment with seg_off <= pos
          while (lo_s < hi_s) {
            const int mid = (lo_s + hi_s + 1) >> 1;
            if (seg_off[mid] <= pos) lo_s = mid; else hi_s = mid - 1;
          }
          v[u] = cand[((long long)row * C + lo_s) * kSegCap + (pos - seg_off[lo_s])];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (at[u] < total) {
          ck[at[u]] = v[u].x;
          ci[at[u]] = int(v[u].y);
        }
      }
    }
    __syncthreads();
    uint32_t prefix, pmask;
    int need_eq;
    row_radix(sh, total, k, [&](int i) { return ck[i]; }, prefix, pmask, need_eq);
    if (prefix >= s_gmax) {                       // uniform: every selectable key is a candidate
      const int cpt = (total + kRowThreads - 1) / kRowThreads;
      const int clo = min(total, tid * cpt), chi = min(total, clo + cpt);
      unsigned cnt_gt = 0, cnt_eq = 0;
      for (int i = clo; i < chi; ++i) {
        const uint32_t km = ck[i] & pmask;
        cnt_gt += km > prefix ? 1u : 0u;
        cnt_eq += km == prefix ? 1u : 0u;
      }
      unsigned tot;
      const unsigned packed = block_inclusive_scan<kRowThreads, unsigned>(
          cnt_gt | (cnt_eq << 16), reinterpret_cast<unsigned*>(sh.scratch), &tot);
      int gt_before = int(packed & 0xffffu) - int(cnt_gt);
      int eq_before = int(packed >> 16) - int(cnt_eq);
      for (int i = clo; i < chi; ++i) {
        const uint32_t km = ck[i] & pmask;
        if (km > prefix) {
          out[gt_before + min(eq_before, need_eq)] = ci[i];
          ++gt_before;
        } else if (km == prefix) {
          if (eq_before < need_eq) out[gt_before + eq_before] = ci[i];
          ++eq_before;
        }
      }
      return;
    }
  }
  // fallback: digit passes over every score of the row (global memory), then an
  // ordered write over per-thread contiguous ranges
  const S* s = scores + (long long)row * n_cap;
  uint32_t prefix, pmask;
  int need_eq;
  row_radix(sh, n, k, [&](int i) { return score_key(score_at(s, i)); }, prefix, pmask, need_eq);
  const int kpt = (n + kRowThreads - 1) / kRowThreads;
  const int a = min(n, tid * kpt), b = min(n, a + kpt);
  int c_gt = 0, c_eq = 0;
  for (int i = a; i < b; ++i) {
    const uint32_t km = score_key(score_at(s, i)) & pmask;
    c_gt += km > prefix ? 1 : 0;
    c_eq += km == prefix ? 1 : 0;
  }
  int t_gt, t_eq;
  int gt_before = block_inclusive_scan<kRowThreads, int>(c_gt, sh.scratch, &t_gt) - c_gt;
  int eq_before = block_inclusive_scan<kRowThreads, int>(c_eq, sh.scratch, &t_eq) - c_eq;
  for (int i = a; i < b; ++i) {
    const uint32_t km = score_key(score_at(s, i)) & pmask;
    if (km > prefix) {
      out[gt_before + min(eq_before, need_eq)] = i;
      ++gt_before;
    } else if (km == prefix) {
      if (eq_before < need_eq) out[gt_before + eq_before] = i;
      ++eq_before;
    }
  }
}

// Segments per row for rows longer than kRowMaxKeys: enough CTAs to cover the GPU,
// each segment at most kRowMaxKeys keys and a multiple of 32.
struct SegPlan { int C, seg_len; };
SegPlan seg_plan(long long rows, int n_cap, int sms) {
  int C = (n_cap + kRowMaxKeys - 1) / kRowMaxKeys;
  const long long want = sms / (rows > 0 ? rows : 1);
  if (want > C) C = int(want < kRowThreads ? want : kRowThreads);
  int seg = (n_cap + C - 1) / C;
  seg = (seg + 31) / 32 * 32;
  if (seg > kRowMaxKeys) seg = kRowMaxKeys;
  C = (n_cap + seg - 1) / seg;
  return SegPlan{C, seg};
}
constexpr int kMaxSegRowKeys = kRowMaxKeys * kRowThreads;   // longest row supported

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

int topk_max_row_entries() { return kMaxSegRowKeys; }

size_t topk_workspace_bytes(const ha_params& p, int Tq, int n_cap) {
  if (n_cap <= kRowMaxKeys || n_cap > kMaxSegRowKeys) return 0;
  const long long rows = (long long)p.B * Tq;
  const SegPlan sp = seg_plan(rows, n_cap, num_sms());
  return size_t(rows) * sp.C * (sizeof(SegMeta) + size_t(kSegCap) * sizeof(uint2));
}

namespace {

template <typename S>
cudaError_t launch_topk_t(const ha_params& p, const S* scores, int n_cap, const int32_t* q_pos,
                          int Tq, int32_t* idx, void* ws, size_t ws_bytes, cudaStream_t st,
                          const StepOpts& so) {
  const long long rows = (long long)p.B * Tq;
  if (rows == 0) return cudaSuccess;
  if (n_cap <= kRowMaxKeys) {                     // the row fits one CTA's shared memory
    const size_t smem = row_smem_bytes(n_cap);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(topk_row<S>), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_row<S>, dim3(unsigned(rows)), dim3(kRowThreads), smem, st, 1u, scores,
                      n_cap, q_pos, so.pos_off, p.k, p.n_win, p.m, p.elig, idx);
  }
  if (n_cap <= kMaxSegRowKeys) {                  // segments, then one merge per row
    const SegPlan sp = seg_plan(rows, n_cap, num_sms());
    const size_t need = size_t(rows) * sp.C * (sizeof(SegMeta) + size_t(kSegCap) * sizeof(uint2));
    if (ws == nullptr || ws_bytes < need) return cudaErrorInvalidValue;
    uint2* cand = static_cast<uint2*>(ws);
    SegMeta* meta = reinterpret_cast<SegMeta*>(cand + size_t(rows) * sp.C * kSegCap);
    const size_t smem1 = size_t(sp.seg_len / 32) * 33 * sizeof(uint32_t);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(topk_seg<S>), smem1);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_seg<S>, dim3(unsigned(rows * sp.C)), dim3(kRowThreads), smem1, st, 1u,
                   scores, n_cap, q_pos, so.pos_off, p.k, p.n_win, p.m, p.elig, sp.C, sp.seg_len,
                   meta, cand);
    if (e != cudaSuccess) return e;
    const size_t smem2 = (size_t(2) * kMergeCap + sp.C + 1) * sizeof(uint32_t);
    e = ensure_smem(reinterpret_cast<const void*>(topk_seg_merge<S>), smem2);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_seg_merge<S>, dim3(unsigned(rows)), dim3(kRowThreads), smem2, st, 1u,
                      scores, n_cap, q_pos, so.pos_off, p.k, p.n_win, p.m, p.elig, sp.C,
                      static_cast<const SegMeta*>(meta), static_cast<const uint2*>(cand), idx);
  }
  return cudaErrorNotSupported;                  // rows longer than kMaxSegRowKeys
}

}  // namespace

cudaError_t launch_topk(const ha_params& p, const void* scores, int n_cap, const int32_t* q_pos,
                        int Tq, int32_t* idx, void* ws, size_t ws_bytes, cudaStream_t st,
                        const StepOpts& so) {
  if (p.fmt & HA_FMT_IDX4)                        // bfloat16 scores of the FP4 indexer
    return launch_topk_t(p, static_cast<const __nv_bfloat16*>(scores), n_cap, q_pos, Tq, idx, ws,
                         ws_bytes, st, so);
  return launch_topk_t(p, static_cast<const float*>(scores), n_cap, q_pos, Tq, idx, ws, ws_bytes,
                       st, so);
}

}  // namespace ha
