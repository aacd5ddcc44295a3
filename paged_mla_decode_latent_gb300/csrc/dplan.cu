// dplan.cu -- the device-planned decode: sizes fixed on the host from
// capacities only, the split-KV partition chosen on the GPU from the device
// context lengths, and the decode launched over a grid sized from the
// capacity whose clusters take their work unit from the device-written list.
//
// This is the three-call interface of "HK MLA: MI35x m16x8 retune, new m16x4
// kernel, page_size + mask support" (aiter PR 3072, Summary, track 2): a
// sizes query (get_mla_metadata_info_v1 there, mla_decode_dplan_info here), a
// metadata kernel on the device (get_mla_metadata_v1_2_device there,
// mla_decode_plan_device here) and the launch, which must agree on the
// number of work slots, tied to the SM count.  Because nothing launched
// depends on the context lengths' values, a CUDA graph of the three calls
// stays valid whatever the lengths become, up to the capacity.  The page
// tables may also come in the CSR form (kv_indptr / kv_indices) that page
// and "perf(mla): chunk the non-FP4 gather_kv_b_proj over KV" (aiter PR 4776,
// description: size the grid from the valid tokens, not kv_indices'
// capacity) use.
//
// The partition: with P = num_sms / 2 CTA pairs and K = sum of ceil(ctx/T)
// key tiles over the batch (T = 64, or 128 for the few-row kernel) (the fair share of a pair is ceil(K / P) tiles),
// every sequence is cut into chunks of max(ceil(share / 2), 2) tiles, unless
// no sequence is longer than 5/4 of the share, in which case none is cut
// (measured on the host-planned kernel: cutting batch 64 x 8192 into 113 +
// 15 tiles was slower than whole sequences).  Half the share keeps the
// greedy dispatch within 1.5 shares of the ideal and matches the host
// planner's simulated choice on the ragged batch (84-tile chunks there, 78
// here).  So at most 2P + B chunks exist, each a unit per 128-row block.
// Units are listed chunk by chunk (all first chunks, then all second ...),
// sequences with more chunks first, which is the longest-first order that
// list scheduling of the in-order block dispatch favours.  A sequence in one
// chunk writes its result directly; a cut one writes partial slots the
// merge reads.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/mla_decode.h"
#include "internal.h"

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMaxDplanBatch = 1024;
constexpr int kMaxChunksPerSeq = mla::kMaxSplits;  // chunks of one sequence: at most 2P <= 254
constexpr int kMinChunkTiles = 2;

int64_t align256(int64_t a) { return (a + 255) / 256 * 256; }

struct PlanArgs {
  const int32_t* seq_lens;
  const int32_t* kv_indptr;  // optional
  int4* units;
  int4* seq_info;
  int32_t* counts;  // [0] units, [1] chunk keys, [2] partial slots
  int32_t* status;
  int batch, row_blocks, pairs, page_size, ctx_capacity, max_units, tile_keys;
};

__global__ void __launch_bounds__(kPlanThreads) plan_device_kernel(PlanArgs a) {
  __shared__ int s_ctx[kMaxDplanBatch];
  __shared__ int s_n[kMaxDplanBatch];
  __shared__ int s_gt[kMaxChunksPerSeq];      // sequences with more than c chunks
  __shared__ int s_off[kMaxChunksPerSeq + 1];  // units listed before chunk level c
  __shared__ long long s_red[32];
  __shared__ int s_redi[32];
  __shared__ int s_chunk;
  const int tid = threadIdx.x, B = a.batch;
  // The lengths (and the CSR row starts) may come from the kernel this one
  // is launched behind.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  long long tiles = 0;
  int max_t = 0;
  for (int b = tid; b < B; b += kPlanThreads) {
    int ctx = a.seq_lens[b];
    int64_t cap = a.ctx_capacity;
    if (a.kv_indptr) {
      const int64_t pages = (int64_t)a.kv_indptr[b + 1] - a.kv_indptr[b];
      cap = pages < 0 ? 0 : min(cap, pages * a.page_size);
    }
    if (ctx < 0 || ctx > cap) {
      atomicOr(a.status, MLA_DEVFLAG_CTX_RANGE);
      ctx = ctx < 0 ? 0 : (int)cap;
    }
    s_ctx[b] = ctx;
    const int t = (ctx + a.tile_keys - 1) / a.tile_keys;
    tiles += t;
    max_t = max(max_t, t);
  }
  for (int o = 16; o > 0; o >>= 1) {
    tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
    max_t = max(max_t, __shfl_xor_sync(0xffffffffu, max_t, o));
  }
  if ((tid & 31) == 0) {
    s_red[tid >> 5] = tiles;
    s_redi[tid >> 5] = max_t;
  }
  for (int c = tid; c < kMaxChunksPerSeq; c += kPlanThreads) s_gt[c] = 0;
  __syncthreads();
  if (tid == 0) {
    long long total = 0;
    int mx = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) {
      total += s_red[w];
      mx = max(mx, s_redi[w]);
    }
    const long long fair = (total + a.pairs - 1) / a.pairs;
    const long long half = (fair + 1) / 2;
    long long chunk = mx <= fair + fair / 4 ? mx : (half > kMinChunkTiles ? half : kMinChunkTiles);
    if (chunk < 1) chunk = 1;
    s_chunk = (int)chunk * a.tile_keys;
  }
  __syncthreads();
  const int chunk_keys = s_chunk;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int n = max(1, (s_ctx[b] + chunk_keys - 1) / chunk_keys);
    s_n[b] = min(n, kMaxChunksPerSeq);
    for (int c = 0; c < s_n[b]; ++c) atomicAdd(&s_gt[c], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int c = 0; c < kMaxChunksPerSeq; ++c) {
      s_off[c] = acc;
      acc += s_gt[c] * a.row_blocks;
    }
    s_off[kMaxChunksPerSeq] = acc;
    a.counts[0] = min(acc, a.max_units);
    a.counts[1] = chunk_keys;
    if (acc > a.max_units) atomicOr(a.status, MLA_DEVFLAG_CTX_RANGE);
  }
  __syncthreads();
  int parts = 0;
  for (int b = tid; b < B; b += kPlanThreads) {
    const int n = s_n[b];
    // rank among sequences ordered by chunk count (more first), then index;
    // partial slots in sequence order for the sequences that are cut
    int rank = 0, part0 = 0;
    for (int x = 0; x < B; ++x) {
      const int nx = s_n[x];
      rank += (nx > n) || (nx == n && x < b);
      part0 += (x < b && nx > 1) ? nx : 0;
    }
    a.seq_info[b] = make_int4(s_ctx[b], part0, n, 0);
    parts += n > 1 ? n : 0;
    for (int c = 0; c < n; ++c) {
      const int k0 = c * chunk_keys;
      const int k1 = min(k0 + chunk_keys, s_ctx[b]);
      for (int rb = 0; rb < a.row_blocks; ++rb) {
        const int u = s_off[c] + rank * a.row_blocks + rb;
        if (u < a.max_units) a.units[u] = make_int4(b, rb | (c << 8), k0, k1);
      }
    }
  }
  for (int o = 16; o > 0; o >>= 1) parts += __shfl_xor_sync(0xffffffffu, parts, o);
  if ((tid & 31) == 0) s_redi[tid >> 5] = parts;
  __syncthreads();
  if (tid == 0) {
    int total = 0;
    for (int w = 0; w < kPlanThreads / 32; ++w) total += s_redi[w];
    a.counts[2] = total;
  }
}

int check_dplan(const mla_decode_dplan_t* d) {
  if (d == nullptr || d->version != MLA_DECODE_DPLAN_VERSION) return MLA_ERR_INVALID_ARG;
  if (d->batch < 1 || d->batch > kMaxDplanBatch || d->rows != d->num_heads * d->sq)
    return MLA_ERR_INVALID_ARG;
  if (d->pairs < 1 || d->max_units < 1 || d->max_parts < 1 || d->wait_limit_us < 0)
    return MLA_ERR_INVALID_ARG;
  if (d->key_tile != (mla_small_rows_fit(d->rows, d->kv_dtype) ? mla::kKeyTileSmall : mla::kKeyTile))
    return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

int check_ws(const mla_decode_dplan_t* d, const void* ws, size_t bytes) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255)) return MLA_ERR_WORKSPACE;
  if ((int64_t)bytes < d->workspace_bytes) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

template <typename T>
T* at(void* ws, int64_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

extern "C" int mla_decode_dplan_info(int32_t batch, int32_t num_heads, int32_t sq,
                                     int32_t page_size, int32_t kv_dtype, int32_t causal,
                                     int32_t ctx_capacity, int32_t num_sms,
                                     mla_decode_dplan_t* info) {
  if (info == nullptr) return MLA_ERR_INVALID_ARG;
  if (batch < 1 || batch > kMaxDplanBatch) return MLA_ERR_INVALID_ARG;
  if (num_heads < 1 || num_heads > 128 || sq < 1 || sq > 16 || num_heads * sq > mla::kMaxRows)
    return MLA_ERR_INVALID_ARG;
  if (page_size < 1 || page_size > 4096 || ctx_capacity < 0) return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return MLA_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  mla_decode_dplan_t d;
  std::memset(&d, 0, sizeof d);
  d.version = MLA_DECODE_DPLAN_VERSION;
  d.batch = batch;
  d.num_heads = num_heads;
  d.sq = sq;
  d.page_size = page_size;
  d.kv_dtype = kv_dtype;
  d.causal = causal;
  d.rows = num_heads * sq;
  d.row_blocks = (d.rows + mla::kRowTile - 1) / mla::kRowTile;
  d.ctx_capacity = ctx_capacity;
  d.num_sms = num_sms;
  d.pairs = num_sms / mla::kClusterSize < 1 ? 1 : num_sms / mla::kClusterSize;
  // a cut sequence has at most 2P chunks, which the merge holds in shared memory
  if (2 * d.pairs > kMaxChunksPerSeq - 1) d.pairs = (kMaxChunksPerSeq - 1) / 2;
  d.max_parts = 2 * d.pairs + batch;
  d.max_units = d.row_blocks * d.max_parts;
  d.key_tile = mla_small_rows_fit(d.rows, kv_dtype) ? mla::kKeyTileSmall : mla::kKeyTile;
  d.min_chunk_keys = kMinChunkTiles * d.key_tile;
  int64_t off = 0;
  d.ws_units_offset = off;
  off = align256(off + (int64_t)d.max_units * 16);
  d.ws_seq_offset = off;
  off = align256(off + (int64_t)batch * 16);
  d.ws_count_offset = off;
  off = align256(off + 16);
  d.ws_partial_o_offset = off;
  off = align256(off + (int64_t)d.max_parts * d.rows * MLA_D_V * 4);
  d.ws_partial_lse_offset = off;
  off = align256(off + (int64_t)d.max_parts * d.rows * 4);
  d.ws_status_offset = off;
  off = align256(off + 16);
  d.workspace_bytes = off;
  *info = d;
  return MLA_OK;
}

extern "C" int mla_decode_plan_device(const mla_decode_dplan_t* dplan, const int32_t* seq_lens,
                                      const int32_t* kv_indptr, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  int st = check_dplan(dplan);
  if (st != MLA_OK) return st;
  st = check_ws(dplan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (seq_lens == nullptr || (reinterpret_cast<uintptr_t>(seq_lens) & 3)) return MLA_ERR_INVALID_ARG;
  PlanArgs a;
  a.seq_lens = seq_lens;
  a.kv_indptr = kv_indptr;
  a.units = at<int4>(workspace, dplan->ws_units_offset);
  a.seq_info = at<int4>(workspace, dplan->ws_seq_offset);
  a.counts = at<int32_t>(workspace, dplan->ws_count_offset);
  a.status = at<int32_t>(workspace, dplan->ws_status_offset);
  a.batch = dplan->batch;
  a.row_blocks = dplan->row_blocks;
  a.pairs = dplan->pairs;
  a.page_size = dplan->page_size;
  a.ctx_capacity = dplan->ctx_capacity;
  a.max_units = dplan->max_units;
  a.tile_keys = dplan->key_tile;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word is reset here, before the planning kernel, so that only
  // kernels sit between the planner, the decode and the merge.
  if (cudaMemsetAsync(a.status, 0, sizeof(int32_t), s) != cudaSuccess) return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(kPlanThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, plan_device_kernel, a) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

extern "C" int mla_decode_fwd_dplan(const mla_decode_dplan_t* dplan, const void* q,
                                    const void* kv_cache, int64_t num_pages,
                                    const float* kv_scale, const int32_t* block_table,
                                    int64_t bt_stride, const int32_t* kv_indptr,
                                    float softmax_scale, void* out, float* lse, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  int st = check_dplan(dplan);
  if (st != MLA_OK) return st;
  st = check_ws(dplan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (!q || !kv_cache || !block_table || !out || !lse) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) & 15) || (reinterpret_cast<uintptr_t>(kv_cache) & 15) ||
      (reinterpret_cast<uintptr_t>(out) & 15) || (reinterpret_cast<uintptr_t>(lse) & 3) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3))
    return MLA_ERR_INVALID_ARG;
  if (num_pages < 1) return MLA_ERR_INVALID_ARG;
  if (num_pages * (int64_t)dplan->page_size >= ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  // Padded table: every row must hold the capacity.  CSR: the planner clamps
  // each context to its own row's pages.
  if (kv_indptr == nullptr &&
      (bt_stride < 1 || bt_stride * (int64_t)dplan->page_size < (int64_t)dplan->ctx_capacity))
    return MLA_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale)) return MLA_ERR_INVALID_ARG;
  mla::FwdParams p;
  std::memset(&p, 0, sizeof p);
  p.q = static_cast<const uint16_t*>(q);
  p.cache = kv_cache;
  p.num_pages = num_pages;
  p.kv_scale = dplan->kv_dtype == MLA_KV_FP8_E4M3 ? kv_scale : nullptr;
  p.bt = block_table;
  p.bt_stride = bt_stride;
  p.bt_indptr = kv_indptr;
  p.seq_lens = nullptr;
  p.softmax_scale = softmax_scale;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.part_o = at<float>(workspace, dplan->ws_partial_o_offset);
  p.part_lse = at<float>(workspace, dplan->ws_partial_lse_offset);
  p.status = at<int32_t>(workspace, dplan->ws_status_offset);
  p.wait_ns = dplan->wait_limit_us > 0 ? (uint64_t)dplan->wait_limit_us * 1000ull
                                       : 2000000000ull;
  p.units = at<int4>(workspace, dplan->ws_units_offset);
  p.n_units = at<int32_t>(workspace, dplan->ws_count_offset);
  p.seq_info = at<int4>(workspace, dplan->ws_seq_offset);
  p.batch = dplan->batch;
  p.unit_capacity = dplan->max_units;
  p.heads = dplan->num_heads;
  p.sq = dplan->sq;
  p.rows = dplan->rows;
  p.page_size = dplan->page_size;
  p.kv_dtype = dplan->kv_dtype;
  p.causal = dplan->causal;
  p.chunk_len = 0;
  p.num_splits = 1;
  p.max_ctx = dplan->ctx_capacity;
  p.row_blocks = dplan->row_blocks;
  p.key_tile = dplan->key_tile;
  if (mla_launch_fwd(p, stream) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}

extern "C" int mla_decode_combine_dplan(const mla_decode_dplan_t* dplan, void* workspace,
                                        size_t workspace_bytes, void* out, float* lse,
                                        void* stream) {
  int st = check_dplan(dplan);
  if (st != MLA_OK) return st;
  st = check_ws(dplan, workspace, workspace_bytes);
  if (st != MLA_OK) return st;
  if (!out || !lse || (reinterpret_cast<uintptr_t>(out) & 15) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return MLA_ERR_INVALID_ARG;
  mla::CombineParams c;
  c.part_o = at<const float>(workspace, dplan->ws_partial_o_offset);
  c.part_lse = at<const float>(workspace, dplan->ws_partial_lse_offset);
  c.out = static_cast<uint16_t*>(out);
  c.lse = lse;
  c.seq_info = at<const int4>(workspace, dplan->ws_seq_offset);
  c.batch = dplan->batch;
  c.rows = dplan->rows;
  c.num_splits = 0;
  if (mla_launch_combine(c, stream) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}
