// internal.h -- constants and launch parameters shared by the library's
// translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace mla {

constexpr int kDQK = 576;       // query/key row: 512 latent + 64 rope
constexpr int kDV = 512;        // value: first 512 dims of the same row
constexpr int kRowTile = 128;   // score rows per CTA pair (the MMA M)
constexpr int kKeyTile = 64;    // keys per pipeline stage (the QK^T MMA N)
constexpr int kKeyTileSmall = 128;  // the same for the few-row kernel
constexpr int kClusterSize = 2; // CTAs per work unit: each owns half the value dims
constexpr int kMaxRows = 1024;  // H * Sq limit
constexpr int kMaxSplits = 256; // split-count cap of the planner

// Everything a fwd kernel needs, resolved on the host from the plan and the
// caller's pointers.
struct FwdParams {
  const uint16_t* q;        // bf16 [B, Sq, H, 576]
  const void* cache;        // [num_pages, ps, 576] bf16 or e4m3
  int64_t num_pages;
  const float* kv_scale;    // device fp32[1] or nullptr
  const int32_t* bt;        // [B, bt_stride]
  int64_t bt_stride;
  const int32_t* seq_lens;  // [B]
  float softmax_scale;
  uint16_t* out;            // bf16 [B, Sq, H, 512]
  float* lse;               // [B, Sq, H]
  float* part_o;            // fp32 [B, S, rows, 512] (S > 1)
  float* part_lse;          // fp32 [B, S, rows]      (S > 1)
  int32_t* status;          // device status word
  uint64_t wait_ns;         // bound of every pipeline wait inside the kernel
  // Device-planned launches (nullptr otherwise): the unit list
  // {b, rb | chunk << 8, k0, k1}, its length, and per sequence
  // {clamped ctx, first partial slot, chunks, 0}.
  const int4* units;
  const int32_t* n_units;
  const int4* seq_info;
  const int32_t* bt_indptr;  // CSR row starts into bt (kv_indices), or nullptr
  int unit_capacity;         // device-planned: the grid's clusters (work-list capacity)
  int key_tile;              // 64: the 128-row kernel; 128: the few-row kernel
  int batch, heads, sq, rows, page_size, kv_dtype, causal;
  int chunk_len, num_splits, max_ctx, row_blocks;
};

// Raises a kernel's dynamic shared-memory limit to `bytes` on device `dev`,
// once per (device, kernel slot); thread-safe.  Slots name the library's
// kernels that need more than 48 KB (at most 32 of them).
cudaError_t opt_in_smem(const void* kernel, int bytes, int dev, int slot);

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  float* lse;
  const int4* seq_info;  // device-planned: per sequence {ctx, first partial, count, 0}
  int batch, rows, num_splits;
};

}  // namespace mla

// The few-row kernel (128-key tiles) takes problems of at most this many
// score rows per sequence: 64 with a bf16 cache, 16 with fp8.
bool mla_small_rows_fit(int rows, int kv_dtype);
int mla_launch_fwd_small_sm103(const mla::FwdParams& p, void* stream);

// Launchers (return a cudaError_t as int).
extern "C" int mla_decode_epilogue(const void* ql_nope, const void* q_pe, const void* kv_c,
                                   const void* k_pe, const int64_t* slot_mapping,
                                   int32_t num_tokens, int32_t num_heads, void* q_out,
                                   void* kv_cache, int64_t num_pages, int32_t page_size,
                                   int32_t kv_dtype, const float* kv_scale,
                                   int32_t cache_inputs_early, int32_t* status, void* stream);
int mla_launch_fwd(const mla::FwdParams& p, void* stream);
int mla_launch_combine(const mla::CombineParams& p, void* stream);
