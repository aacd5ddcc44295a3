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
                double ns_empty, double ns_combine_fixed, double ns_combine_per_unit) {
  std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
  for (int p = 0; p < pairs; ++p) free_at.push(0.0);
  double makespan = 0.0;
  int64_t units = 0;  // (sequence, row block, split) units with keys: partials the combine reads
  // Dispatch order of the launch grid (2 x row blocks, batch, splits): the
  // row block varies fastest, the split slowest.
  for (int s = 0; s < splits; ++s) {
    for (int b = 0; b < batch; ++b) {
      for (int rb = 0; rb < row_blocks; ++rb) {
        int64_t lo = (int64_t)s * chunk;
        int64_t keys = std::max<int64_t>(0, std::min<int64_t>(lens[b], lo + chunk) - lo);
        double cost = keys > 0 ? ns_fixed + keys * ns_per_key + (splits > 1 ? ns_partial : 0.0)
                               : ns_empty;
        units += keys > 0;
        double t = free_at.top();
        free_at.pop();
        t += cost;
        makespan = std::max(makespan, t);
        free_at.push(t);
      }
    }
  }
  return makespan + (splits > 1 ? ns_combine_fixed + ns_combine_per_unit * units : 0.0);
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
  // Few rows per sequence run on the 128-key-tile kernel (its chunks are
  // multiples of 128 keys); everything else on the 128-row, 64-key one.
  p.key_tile = mla_small_rows_fit(p.rows, kv_dtype) ? mla::kKeyTileSmall : mla::kKeyTile;
  p.num_sms = num_sms;
  p.cluster_size = mla::kClusterSize;

  // Per-pair cost model of the decode kernel on GB300.  Its pipeline is bound
  // by the latency of its per-tile chain (score contraction, score swap between
  // the two CTAs, softmax, value contraction), not by its share of HBM
  // bandwidth, so a pair's time per key does not depend on how many pairs run:
  // about 2.2 us per 64-key tile measured for 128 rows, bf16 or fp8.  A work
  // unit also pays its prologue, pipeline fill and epilogue (about 10 us), a
  // split result its partial write, and a split launch the combine pass over
  // all partials.
  const int pairs = std::max(1, num_sms / p.cluster_size);
  const double ns_per_key = 2200.0 / p.key_tile;
  const double ns_fixed = 10000.0, ns_empty = 400.0, ns_partial = 1000.0;
  // The combine reads every non-empty unit's partials once (about 5000
  // bytes/ns) after a launch gap.
  const double ns_combine_fixed = 12000.0;  // measured: launch, dependency wait and the LSE pass
  const double ns_combine_per_unit = std::min(p.rows, p.row_tile) * (MLA_D_V * 4.0 + 4.0) / 5000.0;
  int best_chunk = (int)round_up(std::max(max_ctx, 1), p.key_tile);
  int best_splits = 1;
  if (max_ctx > 0) {
    double best_t = simulate(seq_lens_host, batch, p.row_blocks, best_chunk, 1, pairs, ns_per_key,
                             ns_fixed, ns_partial, ns_empty, ns_combine_fixed,
                          ns_combine_per_unit);
    const int64_t max_splits =
        std::min<int64_t>(ceil_div(max_ctx, p.key_tile), mla::kMaxSplits);
    // The best split candidate is kept only if it beats one unit per
    // sequence clearly: the model leaves out that the pairs slow down a
    // little when all of them run, and that short tail units fill their
    // pipelines less well (measured: a 113 + 15 tile split of batch 64 x 8192
    // was 10% slower than one unit per sequence).
    const double unsplit_t = best_t;
    double split_t = 1e300;
    int split_chunk = best_chunk, split_n = 1;
    auto consider = [&](int chunk) {
      const int splits = (int)ceil_div(max_ctx, chunk);
      if (splits < 2 || splits > mla::kMaxSplits) return;
      double t = simulate(seq_lens_host, batch, p.row_blocks, chunk, splits, pairs, ns_per_key,
                          ns_fixed, ns_partial, ns_empty, ns_combine_fixed,
                          ns_combine_per_unit);
      if (t < split_t) {
        split_t = t;
        split_chunk = chunk;
        split_n = splits;
      }
    };
    // Even splits of the longest context ...
    int last_splits = 1;
    for (int64_t s = 2; s <= max_splits; ++s) {
      int chunk = (int)round_up(ceil_div(max_ctx, s), p.key_tile);
      int splits = (int)ceil_div(max_ctx, chunk);
      if (splits == last_splits) continue;
      last_splits = splits;
      consider(chunk);
    }
    // ... and, for short contexts, every chunk between half and all of it: a
    // long first chunk and a short tail lets the tails of all sequences fill
    // the SM pairs the first chunks leave idle (first chunks are dispatched
    // first).
    if (max_ctx <= 32768)
      for (int64_t chunk = round_up(ceil_div(max_ctx, 2), p.key_tile); chunk < max_ctx;
           chunk += p.key_tile)
        consider((int)chunk);
    if (split_t < unsplit_t * 0.9) {
      best_t = split_t;
      best_chunk = split_chunk;
      best_splits = split_n;
    }
  }
  p.chunk_len = best_chunk;
  p.num_splits = best_splits;
  p.grid_x = p.row_blocks * p.cluster_size;
  p.grid_y = batch;
  p.grid_z = p.num_splits;

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
