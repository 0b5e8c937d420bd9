// Shared device helpers of the CUDA library (storage types, 16-byte vector access,
// eligibility).  Nothing here is shared with the CPU oracle.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "hybrid_attn.h"

namespace ha {

// ---------------------------------------------------------------- host helpers
// Grant `func` at least `bytes` of dynamic shared memory on the current device,
// calling cudaFuncSetAttribute only the first time a larger size is needed.
cudaError_t ensure_smem(const void* func, size_t bytes);
// Count one successful kernel launch (ha_launch_count) and pass the status on.
cudaError_t launched(cudaError_t e);

// Launch `kernel` on `st` as a programmatic dependent of the stream's previous
// kernel: it may be scheduled while that kernel is still running, and must call
// pdl_wait() before it reads or writes any global memory.  cluster_x > 1 also
// groups the CTAs into thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return launched(cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...));
}

// Wait until the preceding kernel of the stream has completed and its memory is
// visible (a no-op when the kernel was not launched as a programmatic dependent);
// then let the next kernel of the stream be scheduled.  Every kernel calls this
// before its first global-memory access, so any kernel launched after it sees
// every earlier kernel complete.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// The two halves, for kernels of a fused step that read nothing the previous
// kernel writes: they let the next kernel be scheduled at once and wait for the
// previous one only before they exit, so that their completion still implies the
// completion of everything before them in the stream.
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- storage types
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kVec = 4;   // elements per 16-byte chunk
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kVec = 8;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Unpack one 16-byte chunk into kVec floats.
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ void unpack(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);            // low half = element 2i
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
// Pack kVec floats (already rounded by from_f32 semantics) into one chunk.
__device__ __forceinline__ uint4 pack(const float (&f)[4]) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}
__device__ __forceinline__ uint4 pack(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i]));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * i + 1]));
    w[i] = lo | (hi << 16);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__device__ __forceinline__ uint4 ld16(const T* p) {   // read-only path, 16-byte aligned
  return __ldg(reinterpret_cast<const uint4*>(p));
}
template <typename T>
__device__ __forceinline__ void st16(T* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// ---------------------------------------------------------------- eligibility
// Number of compressed entries visible to the query at position t, clamped to n_cap.
__device__ __forceinline__ int n_eligible(int t, int n_win, int m, int elig, int n_cap) {
  int n = (elig == HA_ELIG_OVERLAP) ? (t + 1) / m : max(0, t + 1 - n_win) / m;
  return min(max(n, 0), n_cap);
}

// Order-preserving key of a float score for top-k: larger score -> larger key,
// NaN ranks like -inf, -0 and +0 are the same score (a tie, broken by index).
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (s != s) u = 0xff800000u;  // NaN -> -inf
  if (s == 0.f) u = 0u;         // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace ha
