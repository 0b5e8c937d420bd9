// Lightning Indexer scores on CUDA cores, any storage type and shape
// ("DeepSeek-V4 深度研究剖析" §5.3: the indexer scores every compressed CSA
// entry; score formula fixed by this library):
//   s[b,t,j] = sum_h w[b,t,h] * max(0, qI[b,t,h,:] . cI[b,j,:]),  j < n_elig(t).
// One thread per entry; the row's query heads and weights sit in shared memory
// as float32 and are read as broadcasts.  Heads are visited in order and each dot
// product accumulates in index order, all in float32.  This is the general path;
// bfloat16 layers with H_I = 64 and d_I = 128 use the tensor-core kernel.
#include "common.cuh"
#include "kernels.h"

namespace ha {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) index_scores_simt(const T* __restrict__ qI,
                                                         const float* __restrict__ w,
                                                         const T* __restrict__ cI, int n_cap,
                                                         const int32_t* __restrict__ q_pos,
                                                         int pos_off,
                                                         int Tq, int H_I, int d_I, int n_win,
                                                         int m, int elig,
                                                         float* __restrict__ scores) {
  constexpr int V = Elem<T>::kVec;
  pdl_wait_then_release();
  extern __shared__ float sq[];                    // q [H_I][d_I] | w [H_I]
  float* sw = sq + H_I * d_I;
  const int row = blockIdx.x;                      // b * Tq + t
  const int b = row / Tq;
  const int t = q_pos[row] + pos_off;
  const int ne = n_eligible(t, n_win, m, elig, n_cap);
  const int j0 = blockIdx.y * blockDim.x;
  if (j0 >= ne) return;                            // uniform
  const T* q = qI + (long long)row * H_I * d_I;
  for (int i = threadIdx.x; i < H_I * d_I; i += blockDim.x) sq[i] = to_f32(q[i]);
  for (int i = threadIdx.x; i < H_I; i += blockDim.x) sw[i] = w[(long long)row * H_I + i];
  __syncthreads();
  const int j = j0 + threadIdx.x;
  if (j >= ne) return;
  const T* key = cI + ((long long)b * n_cap + j) * d_I;
  float s = 0.f;
  for (int h = 0; h < H_I; ++h) {
    const float* qh = sq + h * d_I;
    float dot = 0.f;
    for (int c = 0; c < d_I; c += V) {
      float f[V];
      unpack(ld16(key + c), f);
#pragma unroll
      for (int e = 0; e < V; ++e) dot = fmaf(qh[c + e], f[e], dot);
    }
    s = fmaf(sw[h], fmaxf(dot, 0.f), s);
  }
  scores[(long long)row * n_cap + j] = s;
}

}  // namespace

cudaError_t launch_index_scores_simt(const ha_params& p, const void* q_idx, const float* w_idx,
                                     const void* cki, int n_cap, const int32_t* q_pos, int Tq,
                                     float* scores, cudaStream_t st, const StepOpts& so) {
  const dim3 grid(p.B * Tq, (n_cap + 255) / 256);
  const size_t smem = (size_t(p.H_I) * p.d_I + p.H_I) * sizeof(float);
  if (p.dtype == HA_BF16) {
    auto k = index_scores_simt<__nv_bfloat16>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(k), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, grid, dim3(256), smem, st, 1, static_cast<const __nv_bfloat16*>(q_idx),
                      w_idx, static_cast<const __nv_bfloat16*>(cki), n_cap, q_pos, so.pos_off, Tq, p.H_I,
                      p.d_I, p.n_win, p.m, p.elig, scores);
  } else {
    auto k = index_scores_simt<float>;
    cudaError_t e = ensure_smem(reinterpret_cast<const void*>(k), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, grid, dim3(256), smem, st, 1, static_cast<const float*>(q_idx), w_idx,
                      static_cast<const float*>(cki), n_cap, q_pos, so.pos_off, Tq, p.H_I, p.d_I,
                      p.n_win,
                      p.m, p.elig, scores);
  }
}

}  // namespace ha
