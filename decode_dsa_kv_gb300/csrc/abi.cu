// Host-side parts of the C ABI that launch nothing: status text, host-memory
// registration for zero-copy reads, the error-word read-back, and the wait
// limit of the attention kernels.
#include "common.cuh"

namespace dsakv {
namespace {
std::atomic<uint64_t> g_wait_limit_ns{0};
}  // namespace

uint64_t wait_limit_ns(uint64_t default_ns) {
  const uint64_t v = g_wait_limit_ns.load(std::memory_order_relaxed);
  return v ? v : default_ns;
}
}  // namespace dsakv

extern "C" void ts_set_wait_limit_ns(uint64_t ns) {
  dsakv::g_wait_limit_ns.store(ns, std::memory_order_relaxed);
}

extern "C" const char* ts_status_string(ts_status s) {
  switch (s) {
    case TS_OK: return "ok";
    case TS_ERR_INVALID_ARG: return "invalid argument";
    case TS_ERR_UNSUPPORTED: return "unsupported size or shape";
    case TS_ERR_WORKSPACE: return "workspace too small or misaligned";
    case TS_ERR_CUDA: return "CUDA error";
    case TS_ERR_DEVICE_CHECK: return "device-side check failed (see the error word)";
  }
  return "unknown status";
}

extern "C" ts_status ts_host_register(void* host, size_t bytes, void** dev) {
  if (!host || !dev || bytes == 0) return TS_ERR_INVALID_ARG;
  if (cudaHostRegister(host, bytes, cudaHostRegisterMapped | cudaHostRegisterPortable) !=
      cudaSuccess) {
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  if (cudaHostGetDevicePointer(dev, host, 0) != cudaSuccess) {
    cudaGetLastError();
    cudaHostUnregister(host);
    return TS_ERR_CUDA;
  }
  return TS_OK;
}

extern "C" ts_status ts_host_unregister(void* host) {
  if (!host) return TS_ERR_INVALID_ARG;
  if (cudaHostUnregister(host) != cudaSuccess) {
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  return TS_OK;
}

extern "C" ts_status ts_host_alloc(size_t bytes, void** host, void** dev) {
  if (!host || !dev || bytes == 0) return TS_ERR_INVALID_ARG;
  *host = nullptr;
  *dev = nullptr;
  void* h = nullptr;
  if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  if (cudaHostGetDevicePointer(dev, h, 0) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(h);
    return TS_ERR_CUDA;
  }
  *host = h;
  return TS_OK;
}

extern "C" ts_status ts_host_free(void* host) {
  if (!host) return TS_ERR_INVALID_ARG;
  if (cudaFreeHost(host) != cudaSuccess) {
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  return TS_OK;
}

extern "C" ts_status ts_read_error(int32_t* err, int32_t* bits, cudaStream_t stream) {
  if (!err || !bits) return TS_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof(int32_t), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return TS_ERR_CUDA;
  }
  *bits = v;
  return v ? TS_ERR_DEVICE_CHECK : TS_OK;
}
