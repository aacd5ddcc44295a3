// noalloc.cu -- a decode entry point for callers that cannot allocate device
// memory.
//
// mla_decode_fwd asks the caller for a workspace (the split partials and the
// status word).  Some callers have no way to provide one: a plugin inside an
// inference server or framework whose host owns all device memory through its
// own pool (a private cudaMalloc there bypasses the pool's accounting and can
// fail under its budget), or a latency-critical loop that must never call
// cudaMalloc / cudaFree because those calls can synchronise the device.
// mla_decode_fwd_noalloc takes only inputs and outputs: its scratch is one
// fixed array in this library's own device memory.
//
// The array is a file-scope __device__ object of kNoAllocScratchBytes
// (64 MiB), created on every GPU that loads the library and held there until
// the process exits.  Host code cannot hand the array's name to a kernel (on
// the host that name refers to a host-side stand-in, not device memory), so the
// first call made on each device looks up the device address with
// cudaGetSymbolAddress while that device is current and caches it.

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/mla_decode.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_fwd_noalloc(const mla_decode_plan_t* plan, const void* q,
                                      const void* kv_cache, int64_t num_pages,
                                      const float* kv_scale, const int32_t* block_table,
                                      int64_t bt_stride, const int32_t* seq_lens,
                                      float softmax_scale, void* out, float* lse, void* stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->workspace_bytes < 0 || (uint64_t)plan->workspace_bytes > kNoAllocScratchBytes)
    return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  int st = scratch_address(&ws);
  if (st != MLA_OK) return st;
  st = mla_decode_fwd(plan, q, kv_cache, num_pages, kv_scale, block_table, bt_stride, seq_lens,
                      softmax_scale, out, lse, ws, kNoAllocScratchBytes, stream);
  if (st != MLA_OK) return st;
  return mla_decode_combine(plan, seq_lens, ws, kNoAllocScratchBytes, out, lse, stream);
}
