// Joint attention of the query heads over the selected (CSA) or all eligible (HCA)
// compressed entries plus the uncompressed sliding window, on CUDA cores, for any
// storage type and shape ("DeepSeek-V4 深度研究剖析" §5.2 SWA, §5.3 CSA, §5.4 HCA;
// "EP 95 解读 DeepSeek-V4 论文": window and compressed entries are concatenated
// before one multi-query attention, so they share one softmax).
//
// Key list of a query at position t (fixed order):
//   slots [0, n_c)            compressed entries: idx[i] (CSA; skipped when outside
//                             [0, n_elig)) or i (HCA, n_c = n_elig),
//   slots [n_c, n_c + n_w)    window positions t-n_w+1 .. t, n_w = min(n_win, t+1).
// The list is cut into `n_splits` contiguous ranges (split-KV); each CTA handles
// one range for 8 heads (one warp per head) with an online softmax over tiles of
// kTile keys staged in shared memory, and writes either the final (o, lse) or a
// float32 partial that attn_merge combines in split order.  Everything is
// float32 with fixed orders, so results are bitwise repeatable.
#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

constexpr int kHeadsPerCta = 8;   // one warp per head
constexpr int kDecodeKeysPerSplit = 128;
constexpr int kThreads = 32 * kHeadsPerCta;

struct AttnArgs {
  const void* q;        // [rows, H, d]
  const void* ck;       // [B, n_cap, d]
  const void* cv;
  const int32_t* idx;   // [rows, k] or null (HCA)
  const void* k_tok;    // [B, tok_cap, d]
  const void* v_tok;
  const int32_t* pos;   // decode: ctx_len [B]; prefill: q_pos [rows]
  int decode;           // 1: t = pos[b] - 1, rows = B
  int Tq, H, d, n_cap, tok_cap, n_win, m, k, elig;
  float scale;
  int n_splits, keys_per_split, tile;
  void* o;              // [rows, H, d]       (n_splits == 1)
  float* lse;           // [rows, H] or null  (n_splits == 1)
  float* o_part;        // [rows, S, H, d]    (n_splits > 1)
  float* lse_part;      // [rows, S, H]
};

template <typename T, int DPL>
__global__ void __launch_bounds__(kThreads) attn_simt(AttnArgs a) {
  pdl_wait_then_release();
  constexpr int V = Elem<T>::kVec;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int row = blockIdx.x;
  const int split = blockIdx.y;
  const int h0 = blockIdx.z * kHeadsPerCta;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = row / a.Tq;
  const int t = a.decode ? a.pos[b] - 1 : a.pos[row];
  const int ld = a.d + V;                           // padded row stride (elements)
  T* sk = reinterpret_cast<T*>(smem_raw);
  T* sv = sk + a.tile * ld;
  float* sq = reinterpret_cast<float*>(sv + a.tile * ld);   // [8][d]
  int* sok = reinterpret_cast<int*>(sq + kHeadsPerCta * a.d);

  const int ne = t >= 0 ? n_eligible(t, a.n_win, a.m, a.elig, a.n_cap) : 0;
  const int n_c = a.idx ? a.k : ne;
  const int n_w = (t >= 0 && a.k_tok != nullptr) ? min(a.n_win, t + 1) : 0;   // null: no window
  const int n_keys = n_c + n_w;
  const int s_lo = split * a.keys_per_split;
  const int s_hi = min(n_keys, s_lo + a.keys_per_split);

  // stage q of this CTA's heads as float32
  const T* qrow = static_cast<const T*>(a.q) + (long long)row * a.H * a.d;
  for (int i = threadIdx.x; i < kHeadsPerCta * a.d; i += kThreads) {
    const int hh = h0 + i / a.d;
    sq[i] = hh < a.H ? to_f32(qrow[(long long)hh * a.d + i % a.d]) : 0.f;
  }

  const int h = h0 + warp;
  float o[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) o[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  const T* ck = static_cast<const T*>(a.ck) + (long long)b * a.n_cap * a.d;
  const T* cv = static_cast<const T*>(a.cv) + (long long)b * a.n_cap * a.d;
  const T* kt = static_cast<const T*>(a.k_tok) + (long long)b * a.tok_cap * a.d;
  const T* vt = static_cast<const T*>(a.v_tok) + (long long)b * a.tok_cap * a.d;
  const int chunks = a.d / V;

  for (int base = s_lo; base < s_hi; base += a.tile) {
    __syncthreads();                                // previous tile fully consumed
    // resolve the tile's slots to rows
    for (int r = threadIdx.x; r < a.tile; r += kThreads) {
      const int slot = base + r;
      int ok = 0;
      if (slot < s_hi) {
        if (slot < n_c) {
          const int j = a.idx ? a.idx[(long long)row * a.k + slot] : slot;
          ok = (j >= 0 && j < ne) ? 1 + j : 0;      // 1 + entry
        } else {
          const int u = t - n_w + 1 + (slot - n_c);
          ok = -(1 + (u % a.tok_cap));              // -(1 + token slot)
        }
      }
      sok[r] = ok;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.tile * chunks; i += kThreads) {
      const int r = i / chunks, c = (i % chunks) * V;
      const int ok = sok[r];
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (ok > 0) {
        kv = ld16(ck + (long long)(ok - 1) * a.d + c);
        vv = ld16(cv + (long long)(ok - 1) * a.d + c);
      } else if (ok < 0) {
        kv = ld16(kt + (long long)(-ok - 1) * a.d + c);
        vv = ld16(vt + (long long)(-ok - 1) * a.d + c);
      }
      *reinterpret_cast<uint4*>(sk + r * ld + c) = kv;
      *reinterpret_cast<uint4*>(sv + r * ld + c) = vv;
    }
    __syncthreads();
    if (h >= a.H) continue;
    const float* qh = sq + warp * a.d;
    const int nt = min(a.tile, s_hi - base);
    for (int sub = 0; sub < nt; sub += 32) {
      const int r = sub + lane;
      float s = -INFINITY;
      if (r < nt && sok[r] != 0) {
        float dot = 0.f;
        const T* kr = sk + r * ld;
        for (int c = 0; c < a.d; c += V) {
          float f[V];
          unpack(*reinterpret_cast<const uint4*>(kr + c), f);
#pragma unroll
          for (int e = 0; e < V; ++e) dot = fmaf(qh[c + e], f[e], dot);
        }
        s = a.scale * dot;
      }
      const float m_new = fmaxf(m_run, warp_max(s));
      if (m_new == -INFINITY) continue;             // nothing valid yet (warp-uniform)
      const float alpha = expf(m_run - m_new);      // exp(-inf) = 0 on the first tile
      const float pr = expf(s - m_new);
      l_run = l_run * alpha + warp_sum(pr);
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[i] *= alpha;
      const int lim = min(32, nt - sub);
      for (int kk = 0; kk < lim; ++kk) {
        const float pk = __shfl_sync(0xffffffffu, pr, kk);
        const T* vr = sv + (sub + kk) * ld;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          const int c = lane + 32 * i;
          if (c < a.d) o[i] = fmaf(pk, to_f32(vr[c]), o[i]);
        }
      }
      m_run = m_new;
    }
  }
  if (h >= a.H) return;
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  const float lse = l_run > 0.f ? m_run + logf(l_run) : -INFINITY;
  if (a.n_splits == 1) {
    T* orow = static_cast<T*>(a.o) + ((long long)row * a.H + h) * a.d;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int c = lane + 32 * i;
      if (c < a.d) orow[c] = from_f32<T>(o[i] * inv);
    }
    if (a.lse && lane == 0) a.lse[(long long)row * a.H + h] = lse;
  } else {
    float* prow = a.o_part + (((long long)row * a.n_splits + split) * a.H + h) * a.d;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int c = lane + 32 * i;
      if (c < a.d) prow[c] = o[i] * inv;
    }
    if (lane == 0) a.lse_part[((long long)row * a.n_splits + split) * a.H + h] = lse;
  }
}

// o = sum_s exp(lse_s - LSE) o_s, LSE = log sum_s exp(lse_s), splits in order.
// One warp per (row, head, slice of dims), kMergeHeads warps per CTA; lane l owns
// QPL 4-dim groups l, l + 32, .. of its slice (128 * QPL dims).  The splits are
// taken 16 / QPL at a time with all sixteen loads of a lane in flight, the first
// group requested before the weights: with few splits (S <= 4, QPL = 4) the
// partials and the lse values arrive in one round trip; with many (QPL = 1) the
// dims are spread over more warps and 16 splits arrive per round trip.
__device__ __forceinline__ void store4(float* o, const float4& v) {
  *reinterpret_cast<float4*>(o) = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* o, const float4& v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(o) = pk;
}

constexpr int kMergeHeads = 8;

// v[j][u] = split s0 + j, dims c0 + 4 * (lane + 32 u) .. + 3 (zeros past S or d)
template <int QPL>
__device__ __forceinline__ void merge_load(float4 (&v)[16 / QPL][QPL], const float* base,
                                           long long ss, int S, int d, int s0, int c0, int lane) {
#pragma unroll
  for (int j = 0; j < 16 / QPL; ++j)
#pragma unroll
    for (int u = 0; u < QPL; ++u) {
      const int c = c0 + 4 * (lane + 32 * u);
      v[j][u] = (s0 + j < S && c < d)
                    ? __ldcg(reinterpret_cast<const float4*>(base + (s0 + j) * ss + c))
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

template <typename T, int QPL>
__global__ void __launch_bounds__(32 * kMergeHeads) attn_merge(const float* __restrict__ o_part,
                                                  const float* __restrict__ lse_part, int S,
                                                  int H, int d, T* __restrict__ o,
                                                  float* __restrict__ lse) {
  constexpr int SPC = 16 / QPL;                   // splits per round trip
  extern __shared__ float wts[];                  // [kMergeHeads][S]
  pdl_wait_then_release();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_sl = (d + 128 * QPL - 1) / (128 * QPL);
  const int gw = blockIdx.y * kMergeHeads + warp;
  const int row = blockIdx.x, h = gw / n_sl, c0 = (gw % n_sl) * (128 * QPL);
  if (h >= H) return;
  float* wv = wts + warp * S;
  const float* lp = lse_part + (long long)row * S * H + h;
  const float* base = o_part + ((long long)row * S * H + h) * d;
  const long long ss = (long long)H * d;
  float4 v[SPC][QPL];
  merge_load<QPL>(v, base, ss, S, d, 0, c0, lane);
  float mx = -INFINITY;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, __ldcg(lp + (long long)s * H));
  mx = warp_max(mx);
  float tot = 0.f;
  for (int s = lane; s < S; s += 32) {
    const float w = mx == -INFINITY ? 0.f : expf(__ldcg(lp + (long long)s * H) - mx);
    wv[s] = w;
    tot += w;
  }
  tot = warp_sum(tot);
  __syncwarp();
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  if (lane == 0 && lse && c0 == 0) lse[(long long)row * H + h] = tot > 0.f ? mx + logf(tot) : -INFINITY;
  float4 acc[QPL];
#pragma unroll
  for (int u = 0; u < QPL; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += SPC) {
    if (s0 != 0) merge_load<QPL>(v, base, ss, S, d, s0, c0, lane);
#pragma unroll
    for (int j = 0; j < SPC; ++j) {
      if (s0 + j >= S) break;
      const float w = wv[s0 + j];
#pragma unroll
      for (int u = 0; u < QPL; ++u) {
        acc[u].x = fmaf(w, v[j][u].x, acc[u].x);
        acc[u].y = fmaf(w, v[j][u].y, acc[u].y);
        acc[u].z = fmaf(w, v[j][u].z, acc[u].z);
        acc[u].w = fmaf(w, v[j][u].w, acc[u].w);
      }
    }
  }
  T* orow = o + ((long long)row * H + h) * d;
#pragma unroll
  for (int u = 0; u < QPL; ++u) {
    const int c = c0 + 4 * (lane + 32 * u);
    if (c < d)
      store4(orow + c, make_float4(acc[u].x * inv, acc[u].y * inv, acc[u].z * inv, acc[u].w * inv));
  }
}

int dpl_for(int d) {
  const int need = (d + 31) / 32;
  int dpl = 2;
  while (dpl < need) dpl *= 2;
  return dpl;
}

template <typename T, int DPL>
cudaError_t launch_dpl(const AttnArgs& a, int rows, size_t smem, cudaStream_t st) {
  auto kern = attn_simt<T, DPL>;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(kern), smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(rows, a.n_splits, (a.H + kHeadsPerCta - 1) / kHeadsPerCta);
  return launch_pdl(kern, grid, dim3(kThreads), smem, st, 1, a);
}

template <typename T>
cudaError_t launch_t(const AttnArgs& a, int rows, cudaStream_t st) {
  const int V = Elem<T>::kVec;
  const size_t smem = size_t(2) * a.tile * (a.d + V) * sizeof(T) +
                      size_t(kHeadsPerCta) * a.d * sizeof(float) + size_t(a.tile) * sizeof(int);
  cudaError_t e;
  switch (dpl_for(a.d)) {
    case 2: e = launch_dpl<T, 2>(a, rows, smem, st); break;
    case 4: e = launch_dpl<T, 4>(a, rows, smem, st); break;
    case 8: e = launch_dpl<T, 8>(a, rows, smem, st); break;
    case 16: e = launch_dpl<T, 16>(a, rows, smem, st); break;
    default: e = launch_dpl<T, 32>(a, rows, smem, st); break;
  }
  return e;
}

}  // namespace

template <typename T, int QPL>
cudaError_t launch_merge_t(int rows, int S, int H, int d, const float* o_part, const float* lse_part,
                           void* o, float* lse, cudaStream_t st) {
  const int n_sl = (d + 128 * QPL - 1) / (128 * QPL);
  const dim3 grid(rows, (H * n_sl + kMergeHeads - 1) / kMergeHeads);
  const size_t smem = size_t(kMergeHeads) * S * sizeof(float);   // up to 128 KiB (S <= 4096)
  if (smem > 48 * 1024) {
    const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(attn_merge<T, QPL>), smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(attn_merge<T, QPL>, grid, dim3(32 * kMergeHeads), smem, st, 1, o_part,
                    lse_part, S, H, d, static_cast<T*>(o), lse);
}

cudaError_t launch_attn_merge(const ha_params& p, int rows, int S, const float* o_part,
                              const float* lse_part, void* o, float* lse, cudaStream_t st) {
  if (p.dtype == HA_BF16)
    return S <= 4 ? launch_merge_t<__nv_bfloat16, 4>(rows, S, p.H, p.d, o_part, lse_part, o, lse, st)
                  : launch_merge_t<__nv_bfloat16, 1>(rows, S, p.H, p.d, o_part, lse_part, o, lse, st);
  return S <= 4 ? launch_merge_t<float, 4>(rows, S, p.H, p.d, o_part, lse_part, o, lse, st)
                : launch_merge_t<float, 1>(rows, S, p.H, p.d, o_part, lse_part, o, lse, st);
}

AttnPlan plan_attention_simt(const ha_params& p, int rows, int max_keys, bool decode) {
  AttnPlan pl{};
  const int elt = p.dtype == HA_BF16 ? 2 : 4;
  const int V = 16 / elt;
  pl.tile = (size_t(2) * 64 * (p.d + V) * elt <= 150 * 1024) ? 64 : 32;
  const int head_groups = (p.H + kHeadsPerCta - 1) / kHeadsPerCta;
  // Decode cuts every key list into ranges of kDecodeKeysPerSplit keys; the plan
  // depends only on the longest possible list, never on the batch, so a sequence
  // gives the same bits at any batch position and batch size.
  (void)rows;
  (void)head_groups;
  int S = 1;
  int kps = max_keys;
  if (decode) {
    kps = kDecodeKeysPerSplit;
    S = (max_keys + kps - 1) / kps;
    if (S < 1) S = 1;
    if (S == 1) kps = max_keys;
  }
  pl.n_splits = S;
  kps = (kps + 31) / 32 * 32;
  pl.keys_per_split = kps > 0 ? kps : 32;
  pl.ws_bytes = S > 1 ? size_t(rows) * S * p.H * (p.d + 1) * sizeof(float) + 256 : 0;
  return pl;
}

cudaError_t launch_attention_simt(const ha_params& p, const AttnPlan& pl, int decode, int Tq,
                                  const void* q, const int32_t* pos, const void* ck,
                                  const void* cv, int n_cap, const int32_t* idx,
                                  const void* k_tok, const void* v_tok, int tok_cap, void* o,
                                  float* lse, void* ws, cudaStream_t st) {
  AttnArgs a{};
  a.q = q; a.ck = ck; a.cv = cv; a.idx = idx; a.k_tok = k_tok; a.v_tok = v_tok;
  a.pos = pos; a.decode = decode; a.Tq = Tq; a.H = p.H; a.d = p.d; a.n_cap = n_cap;
  a.tok_cap = tok_cap; a.n_win = p.n_win; a.m = p.m; a.k = p.k; a.elig = p.elig;
  a.scale = p.scale > 0.f ? p.scale : 1.f / sqrtf(float(p.d));
  a.n_splits = pl.n_splits; a.keys_per_split = pl.keys_per_split; a.tile = pl.tile;
  a.o = o; a.lse = lse;
  const int rows = p.B * Tq;
  if (pl.n_splits > 1) {
    a.o_part = static_cast<float*>(ws);
    a.lse_part = a.o_part + size_t(rows) * pl.n_splits * p.H * p.d;
  }
  const cudaError_t e =
      p.dtype == HA_BF16 ? launch_t<__nv_bfloat16>(a, rows, st) : launch_t<float>(a, rows, st);
  if (e != cudaSuccess || a.n_splits == 1) return e;
  return launch_attn_merge(p, rows, a.n_splits, a.o_part, a.lse_part, a.o, a.lse, st);
}

}  // namespace ha
