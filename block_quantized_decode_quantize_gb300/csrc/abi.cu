// Status strings, the per-thread last CUDA error and the per-device property cache.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace memra {

namespace {
thread_local int32_t g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
std::mutex g_info_mu;
bool g_info_valid[kMaxDevices] = {};
DeviceInfo g_info[kMaxDevices];
}  // namespace

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MEMRA_PDL");
    return !(v && std::strcmp(v, "0") == 0);
  }();
  return on;
}

memra_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = (int32_t)e;
  return MEMRA_ERR_CUDA;
}

memra_status check_launch() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  return MEMRA_OK;
}

bool device_info(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return false;
  }
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_info_mu);
    if (g_info_valid[dev]) {
      *info = g_info[dev];
      return true;
    }
  }
  DeviceInfo d{};
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return false;
  }
  if (dev >= 0 && dev < kMaxDevices) {
    std::lock_guard<std::mutex> lock(g_info_mu);
    g_info[dev] = d;
    g_info_valid[dev] = true;
  }
  *info = d;
  return true;
}

}  // namespace memra

extern "C" const char* memra_status_string(memra_status status) {
  switch (status) {
    case MEMRA_OK: return "MEMRA_OK";
    case MEMRA_ERR_INVALID_ARG: return "MEMRA_ERR_INVALID_ARG: invalid argument";
    case MEMRA_ERR_ALIGNMENT: return "MEMRA_ERR_ALIGNMENT: misaligned pointer";
    case MEMRA_ERR_UNSUPPORTED: return "MEMRA_ERR_UNSUPPORTED: size beyond the library limits";
    case MEMRA_ERR_CUDA: return "MEMRA_ERR_CUDA: CUDA runtime error";
  }
  return "unknown memra_status";
}

extern "C" int32_t memra_last_cuda_error(void) { return memra::g_last_cuda_error; }

extern "C" const char* memra_version(void) { return "memra-gb300 0.1.0 (sm_103a)"; }
