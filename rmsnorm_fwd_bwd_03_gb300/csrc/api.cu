// Library-wide entry points of libgbln: status strings, version, and the
// per-device SM-count cache used to size persistent grids.

#include <atomic>

#include "common.cuh"

namespace gbln {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];  // 0 = not yet queried
std::atomic<unsigned int*> g_err_ptr[kMaxDevices];
// Per-device error word: kernels that wait on asynchronous copies OR in a bit
// here when a wait exceeds its bound (they then stop instead of hanging).
__device__ unsigned int g_device_error;
}  // namespace

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  unsigned int* p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess || !addr) {
    cudaGetLastError();
    return nullptr;
  }
  p = static_cast<unsigned int*>(addr);
  g_err_ptr[dev].store(p, std::memory_order_release);
  return p;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (dev < 0 || dev >= kMaxDevices) return -1;
  int v = g_sms[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return -1;
  }
  g_sms[dev].store(v, std::memory_order_relaxed);
  return v;
}

}  // namespace gbln

extern "C" const char* gbln_status_string(int status) {
  switch (status) {
    case GBLN_OK: return "GBLN_OK";
    case GBLN_ERR_INVALID_ARG: return "GBLN_ERR_INVALID_ARG: invalid argument";
    case GBLN_ERR_UNSUPPORTED: return "GBLN_ERR_UNSUPPORTED: unsupported dtype combination";
    case GBLN_ERR_WORKSPACE: return "GBLN_ERR_WORKSPACE: dW partial workspace too small";
    case GBLN_ERR_CUDA: return "GBLN_ERR_CUDA: CUDA launch or runtime call failed";
    default: return "unknown gbln status";
  }
}

extern "C" int gbln_version(void) { return 10100; }

extern "C" gbln_status gbln_device_error(uint32_t* code, int clear) {
  if (!code) return GBLN_ERR_INVALID_ARG;
  unsigned int* p = gbln::device_error_word();
  if (!p) return GBLN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return GBLN_ERR_CUDA;
  }
  *code = v;
  if (clear && v) {
    const unsigned int zero = 0;
    if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return GBLN_ERR_CUDA;
    }
  }
  return GBLN_OK;
}

namespace gbln {
namespace {
// One thread waits, with the same bounded poll loop the TMA pipelines use, on an
// mbarrier that nothing will ever complete; when the bound runs out it reports
// a wait timeout exactly as a pipeline would and returns.
__global__ void wait_timeout_kernel(uint32_t polls, unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  mbar_init_fence();
  if (!mbar_wait(&bar, 0u, polls)) atomicOr(err, kErrWaitTimeout);
}
}  // namespace
}  // namespace gbln

extern "C" gbln_status gbln_selftest_wait_timeout(uint32_t polls, gbln_stream_t stream) {
  if (polls == 0 || polls > gbln::kWaitPolls) return GBLN_ERR_INVALID_ARG;
  unsigned int* err = gbln::device_error_word();
  if (!err) return GBLN_ERR_CUDA;
  gbln::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(polls, err);
  return cudaGetLastError() == cudaSuccess ? GBLN_OK : GBLN_ERR_CUDA;
}
