// Token compressor of CSA (m = 4) and HCA (m' = 128): every complete block of m
// tokens becomes one entry, the softmax-gated sum of the block's rows
// ("DeepSeek-V4 深度研究剖析" §5.3 CSA compression, §5.4 HCA; the per-block
// softmax-gated sum is the formula this library fixes).  K, V and, for CSA, the
// indexer keys are compressed with the same gates.
//
// HBM-bound streaming kernel: every thread owns one 16-byte chunk of one output
// row and walks the block's tokens with 128-bit read-only loads; consecutive
// threads read consecutive chunks of the same token row, so each warp issues
// fully coalesced 512-byte requests.  Accumulation is float32 in token order.
//   m <= 16 : one thread per (block, chunk) walks all m tokens.
//   m  > 16 : the block's tokens are split into G = min(8, ceil(m/8)) contiguous
//             groups; the G partial sums of a chunk are added in group order
//             through shared memory, so the result does not depend on scheduling.
#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

struct CompressArgs {
  const void* src[3];   // per-token K, V, indexer keys
  void* dst[3];         // compressed K, V, indexer keys
  int chunks[3];        // 16-byte chunks per row of each tensor
  int n_tensors;
  const float* gate;
  const int32_t* blk_begin;
  const int32_t* ctx_len;   // non-null: the block the newest token completes (n_blk = 1)
  int B, n_blk, m, tok_cap, n_cap;
};

// First block to compress for sequence b: blk_begin[b], or the block completed by
// the newest token (ctx_len[b] / m - 1 when ctx_len[b] is a positive multiple of m,
// else none).  Negative: none of the sequence's blocks is compressed.
__device__ __forceinline__ int first_block(const CompressArgs& a, int b) {
  if (!a.ctx_len) return a.blk_begin[b];
  const int c = a.ctx_len[b];
  return (c > 0 && c % a.m == 0) ? c / a.m - 1 : -1;
}

template <typename T>
__device__ __forceinline__ void locate(const CompressArgs& a, int c, int& tsr, int& chunk) {
  tsr = 0;
  chunk = c;
  while (tsr + 1 < a.n_tensors && chunk >= a.chunks[tsr]) { chunk -= a.chunks[tsr]; ++tsr; }
}

// Softmax weights of one block's gates, computed by one thread (m small).
template <typename T>
__global__ void __launch_bounds__(256) compress_small_m(CompressArgs a) {
  constexpr int V = Elem<T>::kVec;
  pdl_wait_then_release();
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  const long long n_items = (long long)a.B * a.n_blk * total_chunks;
  for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < n_items;
       it += (long long)gridDim.x * blockDim.x) {
    const int c = int(it % total_chunks);
    const long long task = it / total_chunks;
    const int b = int(task / a.n_blk);
    const int fb = first_block(a, b);
    const int j = fb < 0 ? -1 : fb + int(task % a.n_blk);
    if (j < 0 || j >= a.n_cap) continue;
    int tsr, chunk;
    locate<T>(a, c, tsr, chunk);
    const int row_elems = a.chunks[tsr] * V;
    // the block's rows and gates are loaded together (neither depends on the other)
    const T* src = static_cast<const T*>(a.src[tsr]);
    uint4 raw[16];
    float g[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < a.m) {
        const long long u = (long long)j * a.m + i;
        const long long slot = (long long)b * a.tok_cap + u % a.tok_cap;
        raw[i] = ld16(src + slot * row_elems + chunk * V);
        g[i] = a.gate[slot];
      }
    }
    float gmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < a.m) gmax = fmaxf(gmax, g[i]);
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < a.m) { g[i] = expf(g[i] - gmax); den += g[i]; }
    const float inv = 1.f / den;
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < a.m) {
        float f[V];
        unpack(raw[i], f);
        const float al = g[i] * inv;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(al, f[e], acc[e]);
      }
    }
    T* dst = static_cast<T*>(a.dst[tsr]) + ((long long)b * a.n_cap + j) * row_elems;
    st16(dst + chunk * V, pack(acc));
  }
}

// CTA = (block task, slice of kSlice chunks) x G token groups.
constexpr int kSlice = 64;
constexpr int kBatch = 8;        // loads in flight per thread
constexpr int kMaxGroups = 8;

__host__ __device__ inline int n_groups(int m) {
  const int g = (m + kBatch - 1) / kBatch;
  return g < kMaxGroups ? g : kMaxGroups;
}

template <typename T>
__global__ void __launch_bounds__(512) compress_large_m(CompressArgs a) {
  constexpr int V = Elem<T>::kVec;
  pdl_wait_then_release();
  extern __shared__ float sm[];                    // alpha[m] | partial[G][kSlice][V]
  const int G = n_groups(a.m);
  const int per_group = (a.m + G - 1) / G;
  float* alpha = sm;
  float* part = sm + ((a.m + 3) & ~3);
  const int task = blockIdx.x;
  const int b = task / a.n_blk;
  const int fb = first_block(a, b);
  const int j = fb < 0 ? -1 : fb + task % a.n_blk;
  if (j < 0 || j >= a.n_cap) return;                // uniform over the CTA
  const int lane_c = threadIdx.x % kSlice;          // chunk within the slice
  const int grp = threadIdx.x / kSlice;             // token group
  const long long base_u = (long long)j * a.m;

  // the first batch of this thread's rows is requested before the gate softmax
  const int c = blockIdx.y * kSlice + lane_c;       // chunk over all tensors
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  int tsr = 0, chunk = 0, row_elems = 0;
  const T* src = nullptr;
  const int i_beg = grp * per_group, i_end = min(a.m, (grp + 1) * per_group);
  uint4 raw[kBatch];
  if (c < total_chunks) {
    locate<T>(a, c, tsr, chunk);
    row_elems = a.chunks[tsr] * V;
    src = static_cast<const T*>(a.src[tsr]) + (long long)b * a.tok_cap * row_elems;
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (i_beg + i < i_end) raw[i] = ld16(src + ((base_u + i_beg + i) % a.tok_cap) * row_elems + chunk * V);
  }
  // gate softmax of this block (warp 0, fixed order)
  if (threadIdx.x < 32) {
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < a.m; i += 32)
      mx = fmaxf(mx, a.gate[(long long)b * a.tok_cap + (base_u + i) % a.tok_cap]);
    mx = warp_max(mx);
    float den = 0.f;
    for (int i = threadIdx.x; i < a.m; i += 32) {
      const float e = expf(a.gate[(long long)b * a.tok_cap + (base_u + i) % a.tok_cap] - mx);
      alpha[i] = e;
      den += e;
    }
    den = warp_sum(den);
    const float inv = 1.f / den;
    __syncwarp();
    for (int i = threadIdx.x; i < a.m; i += 32) alpha[i] *= inv;
  }
  __syncthreads();

  float acc[V];
#pragma unroll
  for (int e = 0; e < V; ++e) acc[e] = 0.f;
  if (c < total_chunks) {
    for (int i0 = i_beg; i0 < i_end; i0 += kBatch) {
      if (i0 != i_beg) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i)
          if (i0 + i < i_end) raw[i] = ld16(src + ((base_u + i0 + i) % a.tok_cap) * row_elems + chunk * V);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (i0 + i < i_end) {
          float f[V];
          unpack(raw[i], f);
          const float al = alpha[i0 + i];
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = fmaf(al, f[e], acc[e]);
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < V; ++e) part[(grp * kSlice + lane_c) * V + e] = acc[e];
  __syncthreads();
  if (grp == 0 && c < total_chunks) {
    for (int g2 = 1; g2 < G; ++g2) {
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] += part[(g2 * kSlice + lane_c) * V + e];
    }
    T* dst = static_cast<T*>(a.dst[tsr]) + ((long long)b * a.n_cap + j) * row_elems;
    st16(dst + chunk * V, pack(acc));
  }
}

template <typename T>
cudaError_t launch(const CompressArgs& a, cudaStream_t st) {
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  if (a.m <= 16) {
    const long long n_items = (long long)a.B * a.n_blk * total_chunks;
    const long long want = (n_items + 255) / 256;
    const int grid = int(want < 148LL * 32 ? want : 148LL * 32);
    return launch_pdl(compress_small_m<T>, dim3(grid), dim3(256), 0, st, 1, a);
  } else {
    const int G = n_groups(a.m);
    const dim3 grid(a.B * a.n_blk, (total_chunks + kSlice - 1) / kSlice);
    const size_t smem = (size_t(((a.m + 3) & ~3)) + size_t(G) * kSlice * Elem<T>::kVec) * sizeof(float);
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(compress_large_m<T>), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(compress_large_m<T>, grid, dim3(G * kSlice), smem, st, 1, a);
  }
}

}  // namespace

cudaError_t launch_compress(const ha_params& p, int n_tensors, const void* const* src,
                            void* const* dst, const int* dims, const float* gate,
                            const int32_t* blk_begin, int n_blk, int tok_cap, int n_cap,
                            cudaStream_t st, const StepOpts& so) {
  CompressArgs a{};
  a.ctx_len = so.ctx_len;
  const int V = p.dtype == HA_BF16 ? 8 : 4;
  for (int i = 0; i < 3; ++i) {
    a.src[i] = i < n_tensors ? src[i] : nullptr;
    a.dst[i] = i < n_tensors ? dst[i] : nullptr;
    a.chunks[i] = i < n_tensors ? dims[i] / V : 0;
  }
  a.n_tensors = n_tensors;
  a.gate = gate;
  a.blk_begin = blk_begin;
  a.B = p.B;
  a.n_blk = n_blk;
  a.m = p.m;
  a.tok_cap = tok_cap;
  a.n_cap = n_cap;
  return p.dtype == HA_BF16 ? launch<__nv_bfloat16>(a, st) : launch<float>(a, st);
}

}  // namespace ha
