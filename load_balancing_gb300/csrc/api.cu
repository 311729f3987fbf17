// Status strings, device checks and the device error word.
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace {

// One word per device that loads the library; kernels set it with atomicCAS
// instead of trapping, dbsp_device_status() reads and clears it.
__device__ int g_error_word;

constexpr int kMaxDevices = 64;
thread_local char t_last_error[256] = "";

std::mutex g_mu;
int g_device_state[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
int* g_error_ptr[kMaxDevices];
int g_sms[kMaxDevices];

}  // namespace

namespace dbsp {

int cuda_fail(cudaError_t err, const char* where) {
  std::snprintf(t_last_error, sizeof(t_last_error), "%s: %s", where, cudaGetErrorString(err));
  cudaGetLastError();  // clear a sticky-free error so the next call starts clean
  return DBSP_ERR_CUDA;
}

int check_device(int* device) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return DBSP_ERR_UNSUPPORTED;
  *device = dev;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_device_state[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_sms[dev] = sms;
    if (major == 10 && minor == 3) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_error_word);
      if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
      g_error_ptr[dev] = static_cast<int*>(p);
      g_device_state[dev] = 1;
    } else {
      std::snprintf(t_last_error, sizeof(t_last_error),
                    "device %d has compute capability %d.%d; libdbsp is built for sm_103a only",
                    dev, major, minor);
      g_device_state[dev] = 2;
    }
  }
  return g_device_state[dev] == 1 ? DBSP_OK : DBSP_ERR_UNSUPPORTED;
}

int* error_word(int device) { return g_error_ptr[device]; }
int sm_count(int device) { return g_sms[device]; }

}  // namespace dbsp

extern "C" const char* dbsp_status_string(int status) {
  switch (status) {
    case DBSP_OK: return "ok";
    case DBSP_ERR_INVALID_ARG: return "invalid argument";
    case DBSP_ERR_UNSUPPORTED: return "unsupported shape or device";
    case DBSP_ERR_CUDA: return "CUDA error";
    case DBSP_ERR_TIMEOUT: return "device pipeline wait timed out";
    default: return "unknown status";
  }
}

extern "C" const char* dbsp_last_error_string(void) { return t_last_error; }

extern "C" int dbsp_device_status(void* stream) {
  int dev = 0;
  int st = dbsp::check_device(&dev);
  if (st != DBSP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "cudaStreamSynchronize");
  int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(int));
  if (e != cudaSuccess) return dbsp::cuda_fail(e, "read error word");
  if (word != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
    if (e != cudaSuccess) return dbsp::cuda_fail(e, "clear error word");
  }
  return word;
}
