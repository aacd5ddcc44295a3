// api.cu -- host side of the C ABI: argument validation, workspace carving and
// the launches of the fwd and combine kernels.  Nothing here allocates or
// synchronises (mla_decode_check excepted, by contract).

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/mla_decode.h"
#include "internal.h"

int mla_launch_fwd_sm103(const mla::FwdParams& p, void* stream);
int mla_launch_fwd_pipe_sm103(const mla::FwdParams& p, void* stream);

namespace {

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_plan(const mla_decode_plan_t* plan) {
  if (plan == nullptr || plan->version != MLA_DECODE_PLAN_VERSION) return MLA_ERR_INVALID_ARG;
  if (plan->batch < 1 || plan->rows < 1 || plan->rows != plan->num_heads * plan->sq)
    return MLA_ERR_INVALID_ARG;
  if (plan->num_splits < 1 || plan->chunk_len < 1 || plan->num_splits > mla::kMaxSplits)
    return MLA_ERR_INVALID_ARG;
  if (plan->kv_dtype != MLA_KV_BF16 && plan->kv_dtype != MLA_KV_FP8_E4M3)
    return MLA_ERR_INVALID_ARG;
  if (plan->wait_limit_us < 0) return MLA_ERR_INVALID_ARG;
  if (plan->key_tile != mla::kKeyTile && plan->key_tile != mla::kKeyTileSmall)
    return MLA_ERR_INVALID_ARG;
  if (plan->key_tile == mla::kKeyTileSmall && !mla_small_rows_fit(plan->rows, plan->kv_dtype))
    return MLA_ERR_INVALID_ARG;
  if (plan->chunk_len % plan->key_tile != 0) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int check_workspace(const mla_decode_plan_t* plan, const void* ws, size_t bytes) {
  if (ws == nullptr || !aligned(ws, 256)) return MLA_ERR_WORKSPACE;
  if ((int64_t)bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

// Validation and launch of the decode kernel.  reset_status: queue the
// status word's reset first (mla_decode_step resets it before the epilogue
// instead, so that no memset node sits between the epilogue and this kernel
// and the programmatic dependent launch can take effect).
int fwd_impl(const mla_decode_plan_t* plan, const void* q, const void* kv_cache,
             int64_t num_pages, const float* kv_scale, const int32_t* block_table,
             int64_t bt_stride, const int32_t* seq_lens, float softmax_scale, void* out,
             float* lse, void* workspace, size_t workspace_bytes, void* stream,
             bool reset_status) {
  int st = check_plan(plan);
  if (st != MLA_OK) return st;
  st = check_workspace(plan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (!q || !kv_cache || !block_table || !seq_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_pages < 1 || bt_stride < 1) return MLA_ERR_INVALID_ARG;
  if (num_pages * (int64_t)plan->page_size >= ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  if (bt_stride * (int64_t)plan->page_size < (int64_t)plan->max_ctx) return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale)) return MLA_ERR_INVALID_ARG;  // NaN

  char* ws = static_cast<char*>(workspace);
  mla::FwdParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.cache = kv_cache;
  p.num_pages = num_pages;
  p.kv_scale = plan->kv_dtype == MLA_KV_FP8_E4M3 ? kv_scale : nullptr;
  p.bt = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.softmax_scale = softmax_scale;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.part_o = plan->num_splits > 1 ? reinterpret_cast<float*>(ws + plan->ws_partial_o_offset) : nullptr;
  p.part_lse =
      plan->num_splits > 1 ? reinterpret_cast<float*>(ws + plan->ws_partial_lse_offset) : nullptr;
  p.status = reinterpret_cast<int32_t*>(ws + plan->ws_status_offset);
  p.wait_ns = plan->wait_limit_us > 0 ? (uint64_t)plan->wait_limit_us * 1000ull
                                      : kDefaultWaitNs;
  p.units = nullptr;
  p.n_units = nullptr;
  p.seq_info = nullptr;
  p.bt_indptr = nullptr;
  p.unit_capacity = 0;
  p.key_tile = plan->key_tile;
  p.batch = plan->batch;
  p.heads = plan->num_heads;
  p.sq = plan->sq;
  p.rows = plan->rows;
  p.page_size = plan->page_size;
  p.kv_dtype = plan->kv_dtype;
  p.causal = plan->causal;
  p.chunk_len = plan->chunk_len;
  p.num_splits = plan->num_splits;
  p.max_ctx = plan->max_ctx;
  p.row_blocks = plan->row_blocks;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (reset_status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (mla_launch_fwd(p, stream) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}

}  // namespace

extern "C" int mla_decode_fwd(const mla_decode_plan_t* plan, const void* q, const void* kv_cache,
                              int64_t num_pages, const float* kv_scale,
                              const int32_t* block_table, int64_t bt_stride,
                              const int32_t* seq_lens, float softmax_scale, void* out, float* lse,
                              void* workspace, size_t workspace_bytes, void* stream) {
  return fwd_impl(plan, q, kv_cache, num_pages, kv_scale, block_table, bt_stride, seq_lens,
                  softmax_scale, out, lse, workspace, workspace_bytes, stream, true);
}

extern "C" int mla_decode_step(const mla_decode_plan_t* plan, const void* ql_nope,
                               const void* q_pe, const void* kv_c, const void* k_pe,
                               const int64_t* slot_mapping, int32_t cache_inputs_early, void* q,
                               void* kv_cache, int64_t num_pages, const float* kv_scale,
                               const int32_t* block_table, int64_t bt_stride,
                               const int32_t* seq_lens, float softmax_scale, void* out, float* lse,
                               void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_plan(plan);
  if (st != MLA_OK) return st;
  st = check_workspace(plan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (plan->kv_dtype == MLA_KV_FP8_E4M3 && kv_scale == nullptr) return MLA_ERR_INVALID_ARG;
  int32_t* status =
      reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan->ws_status_offset);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
  st = mla_decode_epilogue(ql_nope, q_pe, kv_c, k_pe, slot_mapping, plan->batch * plan->sq,
                           plan->num_heads, q, kv_cache, num_pages, plan->page_size,
                           plan->kv_dtype, kv_scale, cache_inputs_early, status, stream);
  if (st != MLA_OK) return st;
  st = fwd_impl(plan, q, kv_cache, num_pages, kv_scale, block_table, bt_stride, seq_lens,
                softmax_scale, out, lse, workspace, workspace_bytes, stream, false);
  if (st != MLA_OK) return st;
  return mla_decode_combine(plan, seq_lens, workspace, workspace_bytes, out, lse, stream);
}

extern "C" int mla_decode_combine(const mla_decode_plan_t* plan, const int32_t* seq_lens,
                                  void* workspace, size_t workspace_bytes, void* out, float* lse,
                                  void* stream) {
  int st = check_plan(plan);
  if (st != MLA_OK) return st;
  st = check_workspace(plan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (!out || !lse || !seq_lens || !aligned(out, 16) || !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
  if (plan->num_splits == 1) return MLA_OK;
  char* ws = static_cast<char*>(workspace);
  mla::CombineParams c;
  c.part_o = reinterpret_cast<const float*>(ws + plan->ws_partial_o_offset);
  c.part_lse = reinterpret_cast<const float*>(ws + plan->ws_partial_lse_offset);
  c.out = static_cast<uint16_t*>(out);
  c.lse = lse;
  c.seq_info = nullptr;
  c.batch = plan->batch;
  c.rows = plan->rows;
  c.num_splits = plan->num_splits;
  if (mla_launch_combine(c, stream) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}

extern "C" int mla_decode_check(const mla_decode_plan_t* plan, const void* workspace,
                                void* stream, int32_t* host_status) {
  int st = check_plan(plan);
  if (st != MLA_OK) return st;
  if (workspace == nullptr || host_status == nullptr) return MLA_ERR_INVALID_ARG;
  int32_t v = 0;
  const char* ws = static_cast<const char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, ws + plan->ws_status_offset, sizeof v, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  *host_status = v;
  if (v & MLA_DEVFLAG_TIMEOUT) return MLA_ERR_TIMEOUT;
  if (v != 0) return MLA_ERR_DEVICE_CHECK;
  return MLA_OK;
}

namespace mla {

cudaError_t opt_in_smem(const void* kernel, int bytes, int dev, int slot) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static uint32_t done[kMaxDev] = {};
  if (dev < 0 || dev >= kMaxDev || slot < 0 || slot >= 32)
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev] & (1u << slot)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev] |= 1u << slot;
  return e;
}

}  // namespace mla

// Few-row blocks go to the 128-key-tile kernel; 128-row blocks with a bf16
// cache to the four-stage kernel (fp8 needs room for raw stages it lacks).
int mla_launch_fwd(const mla::FwdParams& p, void* stream) {
  if (p.key_tile == mla::kKeyTileSmall) return mla_launch_fwd_small_sm103(p, stream);
  if (p.kv_dtype == MLA_KV_BF16) return mla_launch_fwd_pipe_sm103(p, stream);
  return mla_launch_fwd_sm103(p, stream);
}
