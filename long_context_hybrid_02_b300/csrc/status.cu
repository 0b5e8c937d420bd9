// Device error word of the tensor-core kernels: a kernel whose pipeline wait
// runs out of time records a code here (first one wins) and returns instead of
// hanging.  ha_device_error() reads it back.
#include <mutex>

#include "common.cuh"
#include "hybrid_attn.h"
#include "kernels.h"
#include "tc.cuh"

namespace {

__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int* g_error_addr[kMaxDevices] = {};
std::mutex g_error_mu;

}  // namespace

namespace ha {

int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_error_mu);
  if (g_error_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) return nullptr;
    g_error_addr[dev] = static_cast<int*>(addr);
  }
  return g_error_addr[dev];
}

}  // namespace ha

namespace {

// One CTA waits on a barrier that nothing arrives at, through the same bounded
// wait as the tensor-core kernels' pipelines: the wait gives up after its wall-time
// limit, records `code` in the error word (unless a code is already there) and the
// kernel returns.
__global__ void wait_timeout_selftest(int* err, int code) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ha::tc::mbar_init(&bar, 1);
    ha::tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)ha::tc::mbar_wait(&bar, 0u, err, code);
}

}  // namespace

extern "C" ha_status ha_selftest_wait_timeout(int32_t code, ha_stream_t stream) {
  ha::set_last_error("");
  if (code <= 0) {
    ha::set_last_error("code must be positive");
    return HA_ERR_INVALID_ARG;
  }
  int* err = ha::device_error_word();
  if (err == nullptr) {
    ha::set_last_error("device error word unavailable");
    return HA_ERR_CUDA;
  }
  wait_timeout_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, code);
  const cudaError_t e = ha::launched(cudaGetLastError());
  if (e != cudaSuccess) {
    ha::set_last_error(cudaGetErrorString(e));
    return HA_ERR_CUDA;
  }
  return HA_OK;
}

extern "C" ha_status ha_device_error(int32_t* code, int32_t clear) {
  if (code == nullptr) return HA_ERR_INVALID_ARG;
  *code = 0;
  int value = 0;
  if (cudaMemcpyFromSymbol(&value, g_device_error, sizeof(int)) != cudaSuccess) return HA_ERR_CUDA;
  *code = value;
  if (clear && value != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return HA_ERR_CUDA;
  }
  return HA_OK;
}
