// Host-side pieces shared by the entry points: status text, version, RoPE
// frequency tables and launch status.
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace dts_host {

void make_rope_freqs(float theta, int d, dts::RopeFreqs *out) {
  for (int k = 0; k < 64; ++k) {
    double w = 0.0;
    if (k < d / 2) w = std::pow(static_cast<double>(theta), -2.0 * k / static_cast<double>(d));
    const float hi = static_cast<float>(w);
    const float lo = static_cast<float>(w - static_cast<double>(hi));
    out->w[k] = make_float2(hi, lo);
  }
}

int launch_status() {
  return cudaGetLastError() == cudaSuccess ? DTS_OK : DTS_ERR_CUDA;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace dts_host

extern "C" int dts_version(void) { return 100; }

extern "C" const char *dts_status_string(int status) {
  switch (status) {
    case DTS_OK: return "ok";
    case DTS_ERR_INVALID: return "invalid argument (null pointer, shape or alignment)";
    case DTS_ERR_UNSUPPORTED: return "unsupported size (N > 64, d not 64/128, ...)";
    case DTS_ERR_WORKSPACE: return "workspace missing or too small";
    case DTS_ERR_CUDA: return "CUDA launch or driver call failed";
    default: return "unknown status";
  }
}

extern "C" const char *dts_device_error_string(int code) {
  switch (code) {
    case DTS_DEV_OK: return "ok";
    case DTS_DEV_BAD_PARENT: return "bad parent index";
    case DTS_DEV_BAD_DEPTH: return "depth does not match parents";
    case DTS_DEV_BAD_LINK: return "bad child/sibling link";
    case DTS_DEV_BAD_SLOT: return "page, slot or prefix length out of range";
    case DTS_DEV_BAD_PATH: return "accept_len / accepted_path not a valid packed path";
    case DTS_DEV_BAD_BUFFER: return "KV buffer entry misaligned or partly overlapping";
    case DTS_DEV_TIMEOUT: return "a bounded wait inside a kernel gave up";
    default: return "unknown device error";
  }
}
