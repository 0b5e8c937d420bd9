// Token compressor of CSA (m = 4) and HCA (m' = 128): every complete block of m
// tokens becomes one entry, the softmax-gated sum of the block's rows
// ("DeepSeek-V4 深度研究剖析" §5.3 CSA compression, §5.4 HCA; the per-block
// softmax-gated sum is the formula this library fixes).  K, V and, for CSA, the
// indexer keys are compressed with the same gates.
//
// HBM-bound streaming kernel: every thread owns 16-byte chunks of output rows and
// walks the block's tokens with 128-bit read-only loads; consecutive threads read
// consecutive chunks of the same token row, so each warp issues fully coalesced
// 512-byte requests.  Accumulation is float32 in token order.
//   m <= 16 : one thread per (block, chunk) walks all m tokens; each thread keeps
//             the loads of kItems such items in flight (m = 4 is compiled apart,
//             with fewer registers).
//   m  > 16 : the block's tokens are split into G = min(8, ceil(m/16)) contiguous
//             groups whose loads are all issued at once; the G partial sums of a
//             chunk are added in group order through shared memory, so the result
//             does not depend on scheduling.
// Ring slots: the block's first token slot is computed once per block; the next
// slots follow by one increment and at most one wrap (m <= tok_cap).
#include "common.cuh"
#include "fp4.cuh"
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
  int fp4_third;            // the third tensor (indexer keys) is written in the FP4 format
  int kv8;                  // K and V are written in the FP8 KV format (608-byte rows)
};

// Chunk `chunk` (8 dims, of 64 per row of d = 512) of a compressed K or V row in the
// FP8 KV format: dims 0..63 as bfloat16 at byte 16 chunk; dims 64..511 as e4m3fn
// codes at byte 128 + 8 (chunk - 8) with the float32 scale of their 64-dim group,
// scale = amax / 448 (float32 division), at byte 576 + 4 group.  The 8 chunks of a
// group sit on 8 consecutive lanes (lane % 8 == chunk % 8), all of which call this,
// live or not, so that the group's amax can be reduced among them.
__device__ __forceinline__ void write_kv8(unsigned char* row, int chunk, const float (&acc)[8],
                                          bool live) {
  const unsigned lane = threadIdx.x & 31;
  const unsigned grp = 0xffu << (lane & 24u);
  float amax = 0.f;
  if (live && chunk >= 8)
#pragma unroll
    for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(acc[e]));
  amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(grp, amax, 4));
  if (!live) return;
  if (chunk < 8) {
    st16(reinterpret_cast<__nv_bfloat16*>(row) + 8 * chunk, pack(acc));
    return;
  }
  const float scale = __fdiv_rn(amax, 448.f);
  uint32_t w[2] = {0u, 0u};
  if (scale > 0.f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t r;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
          : "=h"(r)
          : "f"(__fdiv_rn(acc[2 * i + 1], scale)), "f"(__fdiv_rn(acc[2 * i], scale)));
      w[i >> 1] |= uint32_t(r) << (16 * (i & 1));
    }
  }
  *reinterpret_cast<uint2*>(row + 128 + 8 * (chunk - 8)) = make_uint2(w[0], w[1]);
  if ((chunk & 7) == 0) *reinterpret_cast<float*>(row + 576 + 4 * ((chunk - 8) >> 3)) = scale;
}

// First block to compress for sequence b: blk_begin[b], or the block completed by
// the newest token (ctx_len[b] / m - 1 when ctx_len[b] is a positive multiple of m,
// else none).  Negative: none of the sequence's blocks is compressed.
__device__ __forceinline__ int first_block(const CompressArgs& a, int b) {
  if (!a.ctx_len) return a.blk_begin[b];
  const int c = a.ctx_len[b];
  return (c > 0 && c % a.m == 0) ? c / a.m - 1 : -1;
}

// Tensor of chunk c of the concatenated rows (K | V | indexer keys), by selects
// rather than indexing the argument arrays (which would copy them to local memory).
struct ChunkRef {
  const void* src;
  void* dst;
  int chunk, row_chunks, tensor;
};
__device__ __forceinline__ ChunkRef chunk_ref(const CompressArgs& a, int c) {
  ChunkRef r;
  if (c < a.chunks[0]) {
    r.src = a.src[0]; r.dst = a.dst[0]; r.chunk = c; r.row_chunks = a.chunks[0]; r.tensor = 0;
  } else if (c < a.chunks[0] + a.chunks[1]) {
    r.src = a.src[1]; r.dst = a.dst[1]; r.chunk = c - a.chunks[0]; r.row_chunks = a.chunks[1];
    r.tensor = 1;
  } else {
    r.src = a.src[2]; r.dst = a.dst[2]; r.chunk = c - a.chunks[0] - a.chunks[1];
    r.row_chunks = a.chunks[2];
    r.tensor = 2;
  }
  return r;
}

// Slot of the first token of block j in the per-token cache of capacity tok_cap.
__device__ __forceinline__ int block_slot(int j, int m, int tok_cap) {
  return int((unsigned long long)j * unsigned(m) % unsigned(tok_cap));
}

constexpr int kItems = 2;        // (block, chunk) items per thread in flight

// One item of compress_small_m: the loads of its m rows and gates.
template <typename T, int MM>
struct SmallItem {
  uint4 raw[MM];
  float g[MM];
  T* dst;
  unsigned char* row4;   // FP4 indexer-key row (fp4_third) or FP8 K / V row (kv8), else null
  int chunk, tensor;
  bool live, in_range;
};

template <typename T, int M>     // M > 0: block size fixed at compile time
__global__ void __launch_bounds__(256) compress_small_m(CompressArgs a) {
  constexpr int V = Elem<T>::kVec;
  constexpr int MM = M > 0 ? M : 16;
  const int m = M > 0 ? M : a.m;
  pdl_wait_then_release();
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  const long long n_items = (long long)a.B * a.n_blk * total_chunks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long base = blockIdx.x * (long long)blockDim.x + threadIdx.x; base < n_items;
       base += kItems * stride) {
    SmallItem<T, MM> itm[kItems];
    // every item's rows and gates are requested before any of them is used
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      const long long it = base + k * stride;
      itm[k].live = false;
      itm[k].row4 = nullptr;
      itm[k].in_range = it < n_items;
      if (it >= n_items) continue;
      const int c = int(it % total_chunks);
      {
        const ChunkRef r0 = chunk_ref(a, c);
        itm[k].tensor = r0.tensor;
        itm[k].chunk = r0.chunk;
      }
      const long long task = it / total_chunks;
      const int b = int(task / a.n_blk);
      const int fb = first_block(a, b);
      const int j = fb < 0 ? -1 : fb + int(task % a.n_blk);
      if (j < 0 || j >= a.n_cap) continue;
      const ChunkRef r = chunk_ref(a, c);
      const long long rowb = (long long)r.row_chunks * V;
      const T* src = static_cast<const T*>(r.src) + (long long)b * a.tok_cap * rowb + r.chunk * V;
      const float* gate = a.gate + (long long)b * a.tok_cap;
      int slot = block_slot(j, m, a.tok_cap);
#pragma unroll
      for (int i = 0; i < MM; ++i) {
        if (i < m) {
          itm[k].raw[i] = ld16(src + slot * rowb);
          itm[k].g[i] = gate[slot];
          if (++slot == a.tok_cap) slot = 0;
        }
      }
      itm[k].dst = static_cast<T*>(r.dst) + ((long long)b * a.n_cap + j) * rowb + r.chunk * V;
      if (a.fp4_third && r.tensor == 2)
        itm[k].row4 = static_cast<unsigned char*>(a.dst[2]) +
                      ((long long)b * a.n_cap + j) * fp4::kRowBytes;
      if (a.kv8 && r.tensor < 2)
        itm[k].row4 = static_cast<unsigned char*>(r.dst) + ((long long)b * a.n_cap + j) * 608;
      itm[k].live = true;
    }
#pragma unroll
    for (int k = 0; k < kItems; ++k) {
      float acc[V];
#pragma unroll
      for (int e = 0; e < V; ++e) acc[e] = 0.f;
      if (itm[k].live) {
      float gmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < MM; ++i)
        if (i < m) gmax = fmaxf(gmax, itm[k].g[i]);
      float den = 0.f;
#pragma unroll
      for (int i = 0; i < MM; ++i)
        if (i < m) { itm[k].g[i] = expf(itm[k].g[i] - gmax); den += itm[k].g[i]; }
      const float inv = 1.f / den;
#pragma unroll
      for (int i = 0; i < MM; ++i) {
        if (i < m) {
          float f[V];
          unpack(itm[k].raw[i], f);
          const float al = itm[k].g[i] * inv;
#pragma unroll
          for (int e = 0; e < V; ++e) acc[e] = fmaf(al, f[e], acc[e]);
        }
      }
      }
      if constexpr (V == 8) {
        if (a.kv8 && itm[k].in_range && itm[k].tensor < 2) {
          write_kv8(itm[k].row4, itm[k].chunk, acc, itm[k].live);
          continue;
        }
        if (a.fp4_third) {
          // FP4 indexer keys: a 16-element group is the chunk pair (2g, 2g + 1), held
          // by lanes (2l, 2l + 1) (items and chunks alternate parity alike, and both
          // lanes of a pair are live or not together); the pair's amax gives the scale
          const int lane = threadIdx.x & 31;
          const bool q4 = itm[k].live && itm[k].row4 != nullptr;
          float amax = 0.f;
          if (q4)
#pragma unroll
            for (int e = 0; e < V; ++e) amax = fmaxf(amax, fabsf(acc[e]));
          amax = fmaxf(amax, __shfl_xor_sync(3u << (lane & ~1), amax, 1));
          if (q4) {
            uint32_t sbyte;
            float sv;
            const uint32_t codes = fp4::quantize8(acc, amax, sbyte, sv);
            *reinterpret_cast<uint32_t*>(itm[k].row4 + 4 * itm[k].chunk) = codes;
            if ((itm[k].chunk & 1) == 0) itm[k].row4[64 + itm[k].chunk / 2] = uint8_t(sbyte);
            continue;
          }
        }
      }
      if (itm[k].live) st16(itm[k].dst, pack(acc));
    }
  }
}

// CTA = (block task, slice of kSlice chunks) x G token groups.
constexpr int kSlice = 32;
constexpr int kBatch = 16;       // loads in flight per thread (a whole token group)
constexpr int kMaxGroups = 8;

__host__ __device__ inline int n_groups(int m) {
  const int g = (m + kBatch - 1) / kBatch;
  return g < kMaxGroups ? g : kMaxGroups;
}

template <typename T>
__global__ void __launch_bounds__(kMaxGroups * kSlice) compress_large_m(CompressArgs a) {
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
  const int slot0 = block_slot(j, a.m, a.tok_cap);  // slot of the block's first token

  // this thread's rows: the first kBatch of its group are requested before the
  // gate softmax
  const int c = blockIdx.y * kSlice + lane_c;       // chunk over all tensors
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  const int i_beg = grp * per_group, i_end = min(a.m, (grp + 1) * per_group);
  const T* src = nullptr;
  long long rowb = 0;
  ChunkRef r{};
  uint4 raw[kBatch];
  auto load_batch = [&](int i0) {
    int slot = slot0 + i0;
    if (slot >= a.tok_cap) slot -= a.tok_cap;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (i0 + i < i_end) {
        raw[i] = ld16(src + slot * rowb);
        if (++slot == a.tok_cap) slot = 0;
      }
    }
  };
  if (c < total_chunks) {
    r = chunk_ref(a, c);
    rowb = (long long)r.row_chunks * V;
    src = static_cast<const T*>(r.src) + (long long)b * a.tok_cap * rowb + r.chunk * V;
    load_batch(i_beg);
  }
  // gate softmax of this block (warp 0, fixed order)
  if (threadIdx.x < 32) {
    const float* gate = a.gate + (long long)b * a.tok_cap;
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < a.m; i += 32) {
      int slot = slot0 + i;
      if (slot >= a.tok_cap) slot -= a.tok_cap;
      alpha[i] = gate[slot];
      mx = fmaxf(mx, alpha[i]);
    }
    mx = warp_max(mx);
    float den = 0.f;
    for (int i = threadIdx.x; i < a.m; i += 32) {
      const float e = expf(alpha[i] - mx);
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
      if (i0 != i_beg) load_batch(i0);
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
    if constexpr (V == 8) {
      if (a.kv8 && r.tensor < 2) {   // a slice of 32 chunks holds whole 8-chunk groups
        write_kv8(static_cast<unsigned char*>(r.dst) + ((long long)b * a.n_cap + j) * 608,
                  r.chunk, acc, true);
        return;
      }
    }
    T* dst = static_cast<T*>(r.dst) + ((long long)b * a.n_cap + j) * rowb;
    st16(dst + r.chunk * V, pack(acc));
  }
}

template <typename T>
cudaError_t launch(const CompressArgs& a, cudaStream_t st) {
  const int total_chunks = a.chunks[0] + a.chunks[1] + a.chunks[2];
  if (a.m <= 16) {
    const long long n_items = (long long)a.B * a.n_blk * total_chunks;
    const long long want = (n_items + 256 * kItems - 1) / (256 * kItems);
    const int grid = int(want < 148LL * 32 ? want : 148LL * 32);
    if (a.m == 4) return launch_pdl(compress_small_m<T, 4>, dim3(grid), dim3(256), 0, st, 1, a);
    return launch_pdl(compress_small_m<T, 0>, dim3(grid), dim3(256), 0, st, 1, a);
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
  a.fp4_third = (p.fmt & HA_FMT_IDX4) && n_tensors == 3 ? 1 : 0;
  a.kv8 = (p.fmt & HA_FMT_KV8) ? 1 : 0;
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
