// libpkv: status strings, version, device queries shared by the entry points.
#include <mutex>

#include "pkv.h"
#include "pkv_host.h"

namespace pkv {

int device_sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev >= 64) dev = 63;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace pkv

extern "C" const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG: a pointer, size or stride is invalid";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: dtype, head_dim, group or block size not supported";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing or too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA launch or driver call failed";
    default: return "PKV: unknown status";
  }
}

extern "C" int pkv_abi_version(void) { return 1; }
