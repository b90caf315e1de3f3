// Library-wide entry points (error string, version) and the host helpers
// declared in common.cuh.
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace dsa {

namespace {
thread_local char g_last_error[512] = "";
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
int g_device_ok[kMaxDevices] = {0};  // 0 unknown, 1 ok, -1 unsupported
}  // namespace

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

dsa_status_t check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  if (g_device_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = sms > 0 ? sms : 148;
    g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    if (g_device_ok[dev] < 0) g_sm_count[dev] = 0;
  }
  if (g_device_ok[dev] < 0) return fail(DSA_ERR_UNSUPPORTED, "libdsa is built for sm_103a (GB300) only");
  return DSA_OK;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (g_sm_count[dev] <= 0) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = sms > 0 ? sms : 148;
  }
  return g_sm_count[dev];
}

dsa_status_t check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
  return DSA_OK;
}

}  // namespace dsa

extern "C" const char* dsa_last_error(void) { return dsa::g_last_error; }

extern "C" const char* dsa_version(void) { return "dsa-gb300 0.1 (sm_103a)"; }
