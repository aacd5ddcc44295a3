// plan.cpp -- host-side split-KV planner (mla_decode_plan) and status strings.
//
// The planner is the "metadata" step of the three-call interface that "HK
// MLA: MI35x m16x8 retune, new m16x4 kernel, page_size + mask support" (aiter
// PR 3072, Summary track 2) describes: a host step that fixes the partition
// the launch then follows.  The partition itself is the one of "perf(mla):
// chunk the non-FP4 gather_kv_b_proj over KV" (aiter PR 4776, description):
// one program per (batch, head group, KV chunk), the grid sized from the
// longest sequence, programs past a sequence's last chunk returning at once.
//
// What is chosen here is only the chunk length.  For each candidate split
// count the planner replays the in-order dispatch of work units (one unit per
// CTA pair) onto the SM pairs with a list scheduler and keeps the split count
// with the smallest simulated makespan.  The cost of a unit is its keys at
// the per-pair streaming rate, plus a fixed prologue/epilogue cost, plus (when
// the result is split) the partial-output write and the combine's re-read.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <queue>
#include <vector>

#include "../../include/mla_decode.h"
#include "internal.h"

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
int64_t align256(int64_t a) { return round_up(a, 256); }

// Simulated time (ns) of one launch with a given chunk length.
double simulate(const int32_t* lens, int batch, int row_blocks, int chunk, int splits,
                int pairs, double ns_per_key, double ns_fixed, double ns_partial,
                double ns_empty, double ns_combine) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int p = 0; p < pairs; ++p) free_at.push(0.0);
  double makespan = 0.0;
  for (int b = 0; b < batch; ++b) {
    for (int rb = 0; rb < row_blocks; ++rb) {
      for (int s = 0; s < splits; ++s) {
        int64_t lo = (int64_t)s * chunk;
        int64_t keys = std::max<int64_t>(0, std::min<int64_t>(lens[b], lo + chunk) - lo);
        double cost = keys > 0 ? ns_fixed + keys * ns_per_key + (splits > 1 ? ns_partial : 0.0)
                               : ns_empty;
        double t = free_at.top();
        free_at.pop();
        t += cost;
        makespan = std::max(makespan, t);
        free_at.push(t);
      }
    }
  }
  return makespan + (splits > 1 ? ns_combine : 0.0);
}

}  // namespace

extern "C" int mla_decode_plan(const int32_t* seq_lens_host, int32_t batch, int32_t num_heads,
                               int32_t sq, int32_t page_size, int32_t kv_dtype, int32_t causal,
                               int32_t num_sms, mla_decode_plan_t* plan) {
  if (plan == nullptr || seq_lens_host == nullptr) return MLA_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535) return MLA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > 128 || sq < 1 || sq > 16) return MLA_ERR_INVALID_ARG;
  if (num_heads * sq > mla::kMaxRows) return MLA_ERR_INVALID_ARG;
  if (page_size < 1 || page_size > 4096) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return MLA_ERR_INVALID_ARG;
  int32_t max_ctx = 0;
  for (int b = 0; b < batch; ++b) {
    if (seq_lens_host[b] < 0) return MLA_ERR_INVALID_ARG;
    max_ctx = std::max(max_ctx, seq_lens_host[b]);
  }
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
  }

  mla_decode_plan_t p;
  std::memset(&p, 0, sizeof p);
  p.version = MLA_DECODE_PLAN_VERSION;
  p.batch = batch;
  p.num_heads = num_heads;
  p.sq = sq;
  p.page_size = page_size;
  p.kv_dtype = kv_dtype;
  p.causal = causal;
  p.rows = num_heads * sq;
  p.row_tile = mla::kRowTile;
  p.row_blocks = (int32_t)ceil_div(p.rows, p.row_tile);
  p.max_ctx = max_ctx;
  p.key_tile = mla::kKeyTile;
  p.num_sms = num_sms;
  p.cluster_size = mla::kClusterSize;

  // Per-pair cost model.  A pair streams keys at its share of HBM bandwidth,
  // or at its share of the tensor rate when that is slower (fp8 at 128 rows).
  const int pairs = std::max(1, num_sms / p.cluster_size);
  const double hbm_bytes_per_ns = 6700.0, tc_flop_per_ns = 1.9e6;
  const double key_bytes = kv_dtype == MLA_KV_BF16 ? 1152.0 : 576.0;
  const double rows_pad = (double)p.row_tile;
  const double ns_key_hbm = key_bytes * pairs / hbm_bytes_per_ns;
  const double ns_key_tc = 2.0 * rows_pad * (MLA_D_QK + MLA_D_V) * pairs / tc_flop_per_ns;
  const double ns_per_key = std::max(ns_key_hbm, ns_key_tc);
  const double ns_fixed = 2000.0, ns_empty = 400.0, ns_combine = 4000.0;
  const double partial_bytes = 2.0 * std::min(p.rows, p.row_tile) * (MLA_D_V * 4.0 + 4.0);
  const double ns_partial = partial_bytes * pairs / hbm_bytes_per_ns;

  int best_chunk = (int)round_up(std::max(max_ctx, 1), p.key_tile);
  int best_splits = 1;
  if (max_ctx > 0) {
    double best_t = simulate(seq_lens_host, batch, p.row_blocks, best_chunk, 1, pairs, ns_per_key,
                             ns_fixed, ns_partial, ns_empty, ns_combine);
    const int64_t max_splits =
        std::min<int64_t>(ceil_div(max_ctx, p.key_tile), mla::kMaxSplits);
    int last_splits = 1;
    for (int64_t s = 2; s <= max_splits; ++s) {
      int chunk = (int)round_up(ceil_div(max_ctx, s), p.key_tile);
      int splits = (int)ceil_div(max_ctx, chunk);
      if (splits == last_splits) continue;
      last_splits = splits;
      double t = simulate(seq_lens_host, batch, p.row_blocks, chunk, splits, pairs, ns_per_key,
                          ns_fixed, ns_partial, ns_empty, ns_combine);
      if (t < best_t * 0.99) {
        best_t = t;
        best_chunk = chunk;
        best_splits = splits;
      }
    }
  }
  p.chunk_len = best_chunk;
  p.num_splits = best_splits;
  p.grid_x = p.num_splits * p.cluster_size;
  p.grid_y = p.row_blocks;
  p.grid_z = batch;

  int64_t off = 0;
  if (p.num_splits > 1) {
    p.ws_partial_o_offset = off;
    off = align256(off + (int64_t)batch * p.num_splits * p.rows * MLA_D_V * 4);
    p.ws_partial_lse_offset = off;
    off = align256(off + (int64_t)batch * p.num_splits * p.rows * 4);
  } else {
    p.ws_partial_o_offset = -1;
    p.ws_partial_lse_offset = -1;
  }
  p.ws_status_offset = off;
  off = align256(off + 16);
  p.workspace_bytes = off;
  *plan = p;
  return MLA_OK;
}

extern "C" const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MLA_ERR_CUDA: return "CUDA call failed";
    case MLA_ERR_DEVICE_CHECK: return "device check failed (block-table entry or context out of range)";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

extern "C" const char* mla_decode_version(void) { return "mla_decode 0.1 sm_103a"; }
