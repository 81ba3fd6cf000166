// api.cu -- status strings, row sizes and the per-device capability check.
#include <atomic>

#include "common.cuh"

namespace nvfp4_mla {

namespace {
constexpr int kMaxDevices = 64;
// 0 = unknown, -1 = not sm_103, >0 = SM count of an sm_103 device.
std::atomic<int> g_sm_count[kMaxDevices];
}  // namespace

int32_t current_device_checked(int* device, int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return NVFP4_MLA_ERR_DEVICE;
  }
  *device = dev;
  int cached = dev < kMaxDevices ? g_sm_count[dev].load(std::memory_order_relaxed) : 0;
  if (cached == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return NVFP4_MLA_ERR_DEVICE;
    }
    cached = (major == 10 && minor == 3 && sms > 0) ? sms : -1;
    if (dev < kMaxDevices) g_sm_count[dev].store(cached, std::memory_order_relaxed);
  }
  if (cached < 0) return NVFP4_MLA_ERR_ARCH;
  *num_sms = cached;
  return NVFP4_MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int32_t launch_status() {
  return cudaGetLastError() == cudaSuccess ? NVFP4_MLA_OK : NVFP4_MLA_ERR_LAUNCH;
}

}  // namespace nvfp4_mla

extern "C" int32_t nvfp4_mla_row_bytes(int32_t row_format) {
  switch (row_format) {
    case NVFP4_MLA_ROW_NVFP4_352: return NVFP4_MLA_NVFP4_ROW_BYTES;
    case NVFP4_MLA_ROW_FP8_576: return NVFP4_MLA_FP8_ROW_BYTES;
    default: return 0;
  }
}

extern "C" const char* nvfp4_mla_status_string(int32_t status) {
  switch (status) {
    case NVFP4_MLA_OK: return "ok";
    case NVFP4_MLA_ERR_NULL: return "a required pointer is NULL";
    case NVFP4_MLA_ERR_SHAPE: return "a size or count is out of range";
    case NVFP4_MLA_ERR_ALIGN: return "a pointer or stride is not 16-byte aligned";
    case NVFP4_MLA_ERR_ARCH: return "the current CUDA device is not an sm_103 (GB300) part";
    case NVFP4_MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_MLA_ERR_LAUNCH: return "a CUDA call failed while enqueuing work";
    case NVFP4_MLA_ERR_FORMAT: return "unknown row format";
    case NVFP4_MLA_ERR_VALUE: return "a scalar argument is not finite or not positive";
    case NVFP4_MLA_ERR_DEVICE: return "no current CUDA device or device query failed";
    default: return "unknown status";
  }
}
