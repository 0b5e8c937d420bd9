// Per-query top-k of the indexer scores ("DeepSeek-V4 深度研究剖析" §5.3: the top-k
// compressed entries are attended, k = 512 for V4-Flash and 1024 for V4-Pro).
//
// Exact radix select over order-preserving 32-bit keys of the float scores (NaN
// ranks as -inf).  A row is handled by a thread-block cluster of C CTAs (C = 1
// when there are enough rows to fill the GPU, up to 16 for a few long rows); CTA
// r of the cluster holds the keys of segment r of the row in shared memory.
//   1. three passes over 11-, 11- and 10-bit digits, most significant first: every
//      CTA histograms the keys of its segment that still match the selected prefix
//      (warp-aggregated shared-memory atomics), the C histograms are summed over
//      distributed shared memory, and every CTA picks the same digit holding the
//      k-th largest key -> the threshold key T and how many keys equal to T are
//      needed (`need_eq`);
//   2. one ordered pass keeps every key > T and the first need_eq keys == T in
//      index order, which realises the tie rule "larger score, then smaller index"
//      and writes the result in ascending index order without a sort: each warp
//      owns a contiguous run of its CTA's segment, counts, and after a block scan
//      and a cluster-wide exchange of the per-CTA counts writes its selections at
//      their final positions.
// Segments longer than the shared-memory budget are re-read from global memory
// (L2) on every pass.
//
// A row of at most kRowMaxKeys entries (decode at up to ~160K tokens, every
// prefill row of a 128K context) is handled by one 1024-thread CTA instead, with
// no cluster: the row's keys are loaded into shared memory once, the first-digit
// histogram is taken from shared memory, the digit passes stop as soon as every
// key of the selected bin is needed, and the ordered write works on 32-key
// bitmaps (`selected` = keys above the threshold prefix, `tied` = keys equal to
// it) whose popcounts are scanned once over the CTA.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace ha {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kMaxCluster = 16;
constexpr int kSmemKeys = 40 * 1024;      // keys held in shared memory per CTA

struct TopkShared {
  int hist[kBins];          // this CTA's histogram of the current pass
  int hsum[2][kBins];       // cluster-wide histogram, by pass parity
  int warp_a[kWarps + 1];   // scan scratch
  int warp_b[kWarps + 1];
  int sel_digit, sel_above;
  int cnt_gt, cnt_eq;       // this CTA's counts of keys > T and == T
};

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

__global__ void __launch_bounds__(kRowThreads) topk_row(const float* __restrict__ scores,
                                                       int n_cap, const int32_t* __restrict__ q_pos,
                                                       int k, int n_win, int m, int elig,
                                                       int32_t* __restrict__ idx) {
  extern __shared__ uint32_t skeys[];
  __shared__ RowShared sh;
  pdl_wait_then_release();
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = n_eligible(q_pos[row], n_win, m, elig, n_cap);
  int32_t* out = idx + (long long)row * k;
  if (n <= k) {                                   // every eligible entry, then -1
    for (int i = tid; i < k; i += kRowThreads) out[i] = i < n ? i : -1;
    return;
  }
  const int words = (n + 31) / 32;
  uint32_t* keys = skeys;                         // key i at pad32(i)
  uint32_t* region = skeys + words * 33;
  const float* s = scores + (long long)row * n_cap;
  // keys in, sixteen loads in flight per thread
  for (int base = 0; base < n; base += 16 * kRowThreads) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = base + u * kRowThreads + tid;
      v[u] = i < n ? __ldg(s + i) : 0.f;
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

__global__ void __launch_bounds__(kThreads) topk_cluster(const float* __restrict__ scores,
                                                         int n_cap, const int32_t* __restrict__ q_pos,
                                                         int k, int n_win, int m, int elig,
                                                         int seg_len, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t skeys[];
  __shared__ TopkShared sh;
  pdl_wait_then_release();
  cg::cluster_group cluster = cg::this_cluster();
  const int C = int(cluster.num_blocks());
  const int rank = int(cluster.block_rank());
  const int row = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = n_eligible(q_pos[row], n_win, m, elig, n_cap);
  int32_t* out = idx + (long long)row * k;
  if (n <= k) {                                   // uniform over the cluster
    if (rank == 0)
      for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* s = scores + (long long)row * n_cap;
  const int lo = min(n, rank * seg_len), hi = min(n, lo + seg_len);
  const int len = hi - lo;
  const bool in_smem = len <= kSmemKeys;
  if (in_smem)
    for (int i = tid; i < len; i += kThreads) skeys[i] = score_key(s[lo + i]);
  auto key_at = [&](int i) -> uint32_t { return in_smem ? skeys[i] : score_key(__ldg(s + lo + i)); };

  uint32_t prefix = 0, pmask = 0;
  int remaining = k;                              // selected keys still to place
  for (int i = tid; i < kBins; i += kThreads) sh.hsum[0][i] = 0;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
    int* hsum = sh.hsum[pass & 1];
    // the other buffer was last read by this CTA's previous scan; peers add into it
    // only after the next cluster barrier
    for (int i = tid; i < kBins; i += kThreads) { sh.hist[i] = 0; sh.hsum[(pass + 1) & 1][i] = 0; }
    __syncthreads();
    for (int base = 0; base < len; base += kThreads) {
      const int i = base + tid;
      const bool valid = i < len;
      const uint32_t key = valid ? key_at(i) : 0u;
      const bool match = valid && ((key & pmask) == prefix);
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const uint32_t digit = (key >> shift) & dmask;
        const unsigned peers = __match_any_sync(act, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[digit], __popc(peers));
      }
    }
    if (pass == 0) cluster.sync();                // every peer's hsum[0] is zeroed
    else __syncthreads();
    // add this CTA's non-zero bins into every peer's (and its own) sum
    for (int b = tid; b < kBins; b += kThreads) {
      const int v = sh.hist[b];
      if (v != 0)
        for (int c = 0; c < C; ++c) atomicAdd(cluster.map_shared_rank(hsum, c) + b, v);
    }
    cluster.sync();                               // every CTA holds the full histogram
    // thread t owns bins 2047-4t .. 2044-4t (descending); find the bin where the
    // running count from the top reaches `remaining`
    int c4[4], own = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) { c4[q] = hsum[kBins - 1 - 4 * tid - q]; own += c4[q]; }
    int total;
    const int incl = block_inclusive_scan<kThreads, int>(own, sh.warp_a, &total);
    const int excl = incl - own;
    if (excl < remaining && remaining <= incl) {
      int run = excl;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (run < remaining && remaining <= run + c4[q]) {
          sh.sel_digit = kBins - 1 - 4 * tid - q;
          sh.sel_above = run;
        }
        run += c4[q];
      }
    }
    __syncthreads();
    prefix |= uint32_t(sh.sel_digit) << shift;
    pmask |= dmask << shift;
    remaining -= sh.sel_above;
    __syncthreads();
  }
  // prefix is the k-th largest key; `remaining` keys equal to it are taken.
  const uint32_t thr = prefix;
  const int need_eq = remaining;

  // ordered pass: warp w owns the contiguous run [w*per_warp, (w+1)*per_warp) of the segment
  const int per_warp = ((len + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int w_lo = min(len, wid * per_warp), w_hi = min(len, w_lo + per_warp);
  int gt = 0, eq = 0;
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w_hi ? key_at(i) : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, i < w_hi && key > thr));
    eq += __popc(__ballot_sync(0xffffffffu, i < w_hi && key == thr));
  }
  int gt_tot, eq_tot;
  const int gt_incl = block_inclusive_scan<kThreads, int>(lane == 0 ? gt : 0, sh.warp_a, &gt_tot);
  const int eq_incl = block_inclusive_scan<kThreads, int>(lane == 0 ? eq : 0, sh.warp_b, &eq_tot);
  int gt_before = __shfl_sync(0xffffffffu, gt_incl, 0) - gt;   // within this CTA
  int eq_before = __shfl_sync(0xffffffffu, eq_incl, 0) - eq;
  if (tid == 0) { sh.cnt_gt = gt_tot; sh.cnt_eq = eq_tot; }
  cluster.sync();
  for (int c = 0; c < rank; ++c) {
    const TopkShared* o = cluster.map_shared_rank(&sh, c);
    gt_before += o->cnt_gt;
    eq_before += o->cnt_eq;
  }
  for (int base = w_lo; base < w_hi; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w_hi ? key_at(i) : 0u;
    const bool is_gt = i < w_hi && key > thr;
    const bool is_eq = i < w_hi && key == thr;
    const unsigned bgt = __ballot_sync(0xffffffffu, is_gt);
    const unsigned beq = __ballot_sync(0xffffffffu, is_eq);
    const unsigned below = (1u << lane) - 1u;
    const int my_gt = gt_before + __popc(bgt & below);
    const int my_eq = eq_before + __popc(beq & below);
    const int taken_eq = min(my_eq, need_eq);    // equal keys taken before this one
    if (is_gt) out[my_gt + taken_eq] = lo + i;
    else if (is_eq && my_eq < need_eq) out[my_gt + my_eq] = lo + i;
    gt_before += __popc(bgt);
    eq_before += __popc(beq);
  }
  cluster.sync();                                 // keep shared memory alive for remote readers
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

// Largest cluster the current device can schedule for this kernel with a full
// shared-memory segment: 16 needs the non-portable cluster size, else 8.
int max_cluster() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  if (cached[dev] != 0) return cached[dev];
  int best = 8;
  const size_t smem = size_t(kSmemKeys) * sizeof(uint32_t);
  if (ensure_smem(reinterpret_cast<const void*>(topk_cluster), smem) == cudaSuccess &&
      cudaFuncSetAttribute(reinterpret_cast<const void*>(topk_cluster),
                           cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kMaxCluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMaxCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, topk_cluster, &cfg) == cudaSuccess && n > 0)
      best = kMaxCluster;
  }
  (void)cudaGetLastError();
  cached[dev] = best;
  return best;
}

}  // namespace

size_t topk_workspace_bytes(const ha_params&, int, int) { return 0; }

cudaError_t launch_topk(const ha_params& p, const float* scores, int n_cap, const int32_t* q_pos,
                        int Tq, int32_t* idx, void*, size_t, cudaStream_t st) {
  const long long rows = (long long)p.B * Tq;
  if (rows == 0) return cudaSuccess;
  if (n_cap <= kRowMaxKeys) {                     // the row fits one CTA's shared memory
    const size_t smem = row_smem_bytes(n_cap);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(topk_row), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_row, dim3(unsigned(rows)), dim3(kRowThreads), smem, st, 1u, scores,
                      n_cap, q_pos, p.k, p.n_win, p.m, p.elig, idx);
  }
  // CTAs per row: enough to cover the GPU when rows are few, and enough for every
  // segment to fit the shared-memory budget when possible.
  const int c_max = max_cluster();
  int C = 1;
  while (C < c_max && rows * C < num_sms()) C *= 2;
  while (C < c_max && (n_cap + C - 1) / C > kSmemKeys) C *= 2;
  const int seg_len = (n_cap + C - 1) / C;
  const size_t smem = size_t(seg_len < kSmemKeys ? seg_len : kSmemKeys) * sizeof(uint32_t);
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(topk_cluster), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(topk_cluster, dim3(unsigned(rows * C)), dim3(kThreads), smem, st, unsigned(C),
                    scores, n_cap, q_pos, p.k, p.n_win, p.m, p.elig, seg_len, idx);
}

}  // namespace ha
