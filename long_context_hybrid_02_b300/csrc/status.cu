// Device error word of the tensor-core kernels: a kernel whose pipeline wait
// runs out of time records a code here (first one wins) and returns instead of
// hanging.  ha_device_error() reads it back.
#include <mutex>

#include "hybrid_attn.h"
#include "kernels.h"

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
