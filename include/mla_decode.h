/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) paged MLA decode library
 * (libmla_decode.so).
 *
 * The operation: multi-head latent attention decode in the absorbed form over
 * a paged latent KV cache.  For sequence b, query token i < Sq and head
 * h < H, the 576-wide query row q[b,i,h,:] (512 latent + 64 rope dims) scores
 * every visible 576-wide latent row of sequence b, gathered through the block
 * table; a softmax over those scores weights the first 512 dims of the same
 * rows:
 *
 *   n      = causal ? ctx_b - Sq + i + 1 : ctx_b        (clamped to [0, ctx_b])
 *   row_j  = kv_scale * cache[block_table[b][j / page_size]][j % page_size][:]
 *   z_j    = softmax_scale * <q[b,i,h,:], row_j>                  j < n
 *   lse    = ln sum_j exp(z_j)                                     (natural log)
 *   out[d] = sum_j exp(z_j - lse) * row_j[d]                       d < 512
 *
 * n == 0 gives out = 0 and lse = -inf.
 *
 * Where each part comes from:
 *   - the 576-wide latent row whose first 512 dims are the value:
 *     "[Perf][Kimi-K3] Cut MLA decode concat/cache epilogue latency"
 *     (vLLM PR 54896), Purpose, item 1;
 *   - the paged cache at a variable page size and the causal mask over the
 *     1+MTP query tokens: "HK MLA: MI35x m16x8 retune, new m16x4 kernel,
 *     page_size + mask support" (aiter PR 3072), Summary, track 1;
 *   - the three-call interface (a sizes/plan step, a metadata step and the
 *     launch, which must all agree on the partition): same page, Summary,
 *     track 2 (get_mla_metadata_info_v1 / get_mla_metadata_v1_2_device and the
 *     kernel launch "all agree");
 *   - the split of each sequence's keys into chunks on the grid, with a grid
 *     sized from the longest sequence and chunks past a sequence's end
 *     returning at once: "perf(mla): chunk the non-FP4 gather_kv_b_proj over
 *     KV" (aiter PR 4776), description, second and third paragraphs.  The
 *     log-sum-exp merge of the chunk partials follows from the per-row LSE
 *     output; the pages do not write it out.
 *
 * Conventions for every entry point:
 *   - All pointers marked "device" are CUDA device pointers of the current
 *     device; "host" pointers are ordinary host memory.  The caller owns every
 *     buffer, the workspace included.  The library allocates nothing.
 *   - Work is queued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream).  No entry point synchronises the host except
 *     mla_decode_check, which says so.
 *   - Errors are returned as mla_status codes (never thrown, never printed).
 *     Arguments are validated on the host before anything is queued; when a
 *     call returns an error nothing was queued.
 *   - Conditions only the device can see (a block-table entry outside
 *     [0, num_pages), a context longer than the plan covers, a wait that ran
 *     past its iteration limit) never fault: the kernel clamps the access,
 *     sets a bit in the status word inside the workspace and carries on or
 *     stops early.  mla_decode_check reads that word.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,  /* a pointer, size or enum is out of range */
  MLA_ERR_UNSUPPORTED = -2,  /* valid request this build does not implement */
  MLA_ERR_WORKSPACE = -3,    /* workspace NULL, misaligned or too small */
  MLA_ERR_CUDA = -4,         /* a CUDA runtime/driver call failed */
  MLA_ERR_DEVICE_CHECK = -5, /* device status word: bad page id or context */
  MLA_ERR_TIMEOUT = -6       /* device status word: a bounded wait expired */
} mla_status;

/* Cache element types. */
typedef enum mla_kv_dtype {
  MLA_KV_BF16 = 0,     /* bfloat16 latent rows, 1152 bytes each */
  MLA_KV_FP8_E4M3 = 1  /* OCP fp8 E4M3FN codes, 576 bytes each, times kv_scale */
} mla_kv_dtype;

/* Bits of the device status word (OR-ed together by the kernels). */
#define MLA_DEVFLAG_BAD_PAGE 0x1   /* block-table entry outside [0, num_pages) */
#define MLA_DEVFLAG_CTX_RANGE 0x2  /* seq_lens[b] < 0 or beyond the plan's max_ctx
                                      (clamped to [0, max_ctx] on the device) */
#define MLA_DEVFLAG_TIMEOUT 0x4    /* a bounded barrier wait gave up         */
#define MLA_DEVFLAG_Q_RANGE 0x8    /* fp8 path: |q| beyond the fp16 range    */

#define MLA_DECODE_PLAN_VERSION 1
#define MLA_D_QK 576 /* query/key row width: 512 latent + 64 rope */
#define MLA_D_V 512  /* value width: the first 512 dims of the same row */

/*
 * The split-KV partition of one batch shape.  Plain old data: the caller owns
 * it, may copy or serialise it, and passes it unchanged to the calls below.
 * Fields are outputs of mla_decode_plan; callers do not edit them.
 */
typedef struct mla_decode_plan_t {
  int32_t version;      /* MLA_DECODE_PLAN_VERSION */
  int32_t batch;        /* B */
  int32_t num_heads;    /* H */
  int32_t sq;           /* query tokens per sequence, 1 + MTP */
  int32_t page_size;    /* keys per cache page */
  int32_t kv_dtype;     /* mla_kv_dtype */
  int32_t causal;       /* 0 or 1 */
  int32_t rows;         /* H * Sq: score rows per sequence */
  int32_t row_tile;     /* rows one CTA pair handles (128) */
  int32_t row_blocks;   /* ceil(rows / row_tile) */
  int32_t max_ctx;      /* longest context the plan covers */
  int32_t key_tile;     /* keys per pipeline tile: 128 when rows <= 64 (bf16) or <= 16
                           (fp8), the few-row kernel; 64 otherwise */
  int32_t chunk_len;    /* keys per split, a multiple of key_tile */
  int32_t num_splits;   /* splits per sequence = ceil(max_ctx / chunk_len) */
  int32_t num_sms;      /* SM count the partition was balanced for */
  int32_t cluster_size; /* CTAs cooperating on one (b, row block, split) */
  int32_t grid_x, grid_y, grid_z; /* launch grid of mla_decode_fwd: (2 x row_blocks, batch,
                                     num_splits); splits vary slowest */
  int32_t wait_limit_us; /* bound of every device-side wait, in microseconds; 0 (what
                            mla_decode_plan writes) means 2 s.  The one field a caller
                            may change: a short limit is how the timeout path is
                            exercised (waits then give up, MLA_ERR_TIMEOUT) */
  int64_t ws_partial_o_offset;   /* byte offset of fp32 [B, S, rows, 512] partials */
  int64_t ws_partial_lse_offset; /* byte offset of fp32 [B, S, rows] partial LSEs */
  int64_t ws_status_offset;      /* byte offset of the int32 device status word */
  int64_t workspace_bytes;       /* bytes the caller must provide */
} mla_decode_plan_t;

/*
 * mla_decode_plan -- choose the split-KV partition (the "metadata" step).
 *
 * seq_lens_host  host int32[batch]: keys per sequence, the Sq new tokens
 *                included (the cache insert precedes the decode).  0 allowed.
 * batch          1 .. 65535
 * num_heads      1 .. 128 with num_heads * sq <= 1024
 * sq             1 .. 16 query tokens per sequence
 * page_size      1 .. 4096 keys per page
 * kv_dtype       mla_kv_dtype
 * causal         0: every token sees all keys; 1: token i sees ctx - Sq + i + 1
 * num_sms        SMs to balance for; 0 queries the current device
 * plan           host out-parameter
 *
 * The chunk length is a multiple of the key tile, chosen by simulating
 * the in-order block dispatch over the SMs for each candidate split count
 * and keeping the fastest (partial-output traffic counted).  The plan stays
 * valid for later calls whose contexts are all <= plan->max_ctx; splits past
 * a shorter sequence's end exit at once.  Pure host code: queues nothing.
 * Returns MLA_OK or MLA_ERR_INVALID_ARG / MLA_ERR_CUDA (num_sms query).
 */
int mla_decode_plan(const int32_t* seq_lens_host, int32_t batch, int32_t num_heads,
                    int32_t sq, int32_t page_size, int32_t kv_dtype, int32_t causal,
                    int32_t num_sms, mla_decode_plan_t* plan);

/*
 * mla_decode_fwd -- the decode kernel: block-table gather, QK^T, masked
 * online softmax and PV for every (sequence, row block, split).
 *
 * plan            host, from mla_decode_plan
 * q               device bf16 [B, Sq, H, 576], contiguous, 16-byte aligned
 * kv_cache        device [num_pages, page_size, 576] bf16 or e4m3 codes,
 *                 contiguous, 16-byte aligned
 * num_pages       pages in kv_cache (block-table entries are checked against it)
 * kv_scale        device fp32[1]: dequant multiplier of the fp8 cache; NULL
 *                 means 1.0; ignored for bf16
 * block_table     device int32 [B, bt_stride]; entries past ceil(ctx_b /
 *                 page_size) are never read
 * bt_stride       int32 elements between consecutive sequences' tables
 * seq_lens        device int32[B]; each <= plan->max_ctx and <= bt_stride *
 *                 page_size
 * softmax_scale   multiplier of the raw dot product (e.g. 1/sqrt(192))
 * out             device bf16 [B, Sq, H, 512]
 * lse             device fp32 [B, Sq, H] (natural-log LSE of the scaled scores)
 * workspace       device, 256-byte aligned, >= plan->workspace_bytes; holds
 *                 the split partials and the status word; reused across calls
 * stream          cudaStream_t as void*
 *
 * With plan->num_splits == 1 this call writes out and lse itself.  Otherwise
 * it writes per-split partials into the workspace and mla_decode_combine must
 * follow on the same stream before out/lse are read.  Resets the status word
 * (an async memset on `stream`) before the kernel.
 */
int mla_decode_fwd(const mla_decode_plan_t* plan, const void* q, const void* kv_cache,
                   int64_t num_pages, const float* kv_scale, const int32_t* block_table,
                   int64_t bt_stride, const int32_t* seq_lens, float softmax_scale,
                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * mla_decode_combine -- log-sum-exp merge of the split partials:
 *   L = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - L) * o_s,  lse = L
 * over the splits of each row; splits with no keys (lse_s = -inf) carry no
 * weight, and a row with no keys at all gets out = 0, lse = -inf.
 *
 * Arguments as in mla_decode_fwd (same plan, seq_lens, workspace, out, lse,
 * stream).  A no-op returning MLA_OK when plan->num_splits == 1.
 */
int mla_decode_combine(const mla_decode_plan_t* plan, const int32_t* seq_lens,
                       void* workspace, size_t workspace_bytes, void* out, float* lse,
                       void* stream);

/*
 * mla_decode_check -- synchronously read the device status word of the last
 * call that used `workspace` on `stream`.  Blocks the host until `stream`
 * drains.  *host_status receives the MLA_DEVFLAG_* bits (0 = clean).
 * Returns MLA_OK, MLA_ERR_DEVICE_CHECK (a bad page id or context),
 * MLA_ERR_TIMEOUT (a wait gave up) or MLA_ERR_CUDA.
 */
int mla_decode_check(const mla_decode_plan_t* plan, const void* workspace, void* stream,
                     int32_t* host_status);

/*
 * Device-planned decode.  The three calls of "HK MLA: MI35x m16x8 retune, new
 * m16x4 kernel, page_size + mask support" (aiter PR 3072), Summary, track 2:
 * a sizes query, a metadata kernel on the device and the launch, agreeing on
 * the work-slot count tied to the SM count:
 *
 *   mla_decode_dplan_info      host: sizes from capacities only (no lengths)
 *   mla_decode_plan_device     device: the split-KV partition from the device
 *                              lengths, written into the workspace
 *   mla_decode_fwd_dplan       the decode over a grid of max_units CTA pairs,
 *                              each taking its unit from the list (slots past
 *                              the list's length exit at once)
 *   mla_decode_combine_dplan   the merge of the sequences that were cut
 *
 * Nothing queued depends on the lengths' values, so a CUDA graph of the last
 * three calls stays valid whatever the lengths become, up to ctx_capacity.
 * The partition: with P = num_sms / 2 pairs and K = the batch's 64-key tiles,
 * sequences are cut into chunks of max(ceil(ceil(K / P) / 2), 2) tiles unless
 * none is longer than 5/4 of the share ceil(K / P) (then none is cut); units
 * are listed chunk level by chunk level, sequences with more chunks first.
 * At most 2P + B chunks, so max_units = row_blocks * (2P + B).
 *
 * Page tables: the padded block table of mla_decode_fwd (kv_indptr NULL), or
 * the CSR form: kv_indptr device int32 [B + 1], sequence b's page ids are
 * block_table[kv_indptr[b] .. kv_indptr[b + 1]) (block_table is kv_indices,
 * bt_stride ignored) and its context is clamped, and flagged, to those pages.
 */
typedef struct mla_decode_dplan_t {
  int32_t version;        /* MLA_DECODE_DPLAN_VERSION */
  int32_t batch;          /* B, 1 .. 1024 */
  int32_t num_heads, sq, page_size, kv_dtype, causal;
  int32_t rows;           /* H * Sq */
  int32_t row_blocks;     /* ceil(rows / 128) */
  int32_t ctx_capacity;   /* longest context any call may bring */
  int32_t num_sms;        /* SMs the partition is balanced for */
  int32_t pairs;          /* P = num_sms / 2 (at most 127) */
  int32_t max_parts;      /* partial-slot capacity, 2P + B */
  int32_t max_units;      /* work-list capacity and launch size, row_blocks * (2P + B) */
  int32_t min_chunk_keys; /* shortest chunk a cut sequence gets (2 key tiles) */
  int32_t key_tile;       /* 64, or 128 for the few-row kernel (as mla_decode_plan_t) */
  int32_t wait_limit_us;  /* as in mla_decode_plan_t: 0 = 2 s; the one field a caller may set */
  int32_t reserved0;
  int64_t ws_units_offset;  /* int32x4 [max_units] {b, row block | chunk << 8, k0, k1} */
  int64_t ws_seq_offset;    /* int32x4 [B] {clamped ctx, first partial slot, chunks, 0} */
  int64_t ws_count_offset;  /* int32 [4] {units, chunk keys, partial slots used, 0} */
  int64_t ws_partial_o_offset;   /* fp32 [max_parts, rows, 512] */
  int64_t ws_partial_lse_offset; /* fp32 [max_parts, rows] */
  int64_t ws_status_offset;      /* int32 status word */
  int64_t workspace_bytes;
} mla_decode_dplan_t;

#define MLA_DECODE_DPLAN_VERSION 1

/* Sizes of the device-planned decode (pure host code; num_sms 0 queries the
 * current device).  Arguments as mla_decode_plan, with ctx_capacity in place
 * of the lengths.  Returns MLA_OK, MLA_ERR_INVALID_ARG or MLA_ERR_CUDA. */
int mla_decode_dplan_info(int32_t batch, int32_t num_heads, int32_t sq, int32_t page_size,
                          int32_t kv_dtype, int32_t causal, int32_t ctx_capacity,
                          int32_t num_sms, mla_decode_dplan_t* info);

/* The partition on the device: reads seq_lens (device int32 [B]) and, in the
 * CSR form, kv_indptr (else NULL); resets the status word and writes the
 * unit list into the workspace (256-byte aligned, >= workspace_bytes).
 * Lengths < 0 or beyond the capacity (or the sequence's CSR pages) are
 * clamped and set MLA_DEVFLAG_CTX_RANGE. */
int mla_decode_plan_device(const mla_decode_dplan_t* dplan, const int32_t* seq_lens,
                           const int32_t* kv_indptr, void* workspace, size_t workspace_bytes,
                           void* stream);

/* The decode over the device-written unit list: arguments as mla_decode_fwd
 * (the lengths come from the plan in the workspace) plus kv_indptr for the
 * CSR form.  Units of uncut sequences write out and lse; cut ones write
 * partials for mla_decode_combine_dplan, which must follow. */
int mla_decode_fwd_dplan(const mla_decode_dplan_t* dplan, const void* q, const void* kv_cache,
                         int64_t num_pages, const float* kv_scale, const int32_t* block_table,
                         int64_t bt_stride, const int32_t* kv_indptr, float softmax_scale,
                         void* out, float* lse, void* workspace, size_t workspace_bytes,
                         void* stream);

/* The log-sum-exp merge of the cut sequences (the others return at once). */
int mla_decode_combine_dplan(const mla_decode_dplan_t* dplan, void* workspace,
                             size_t workspace_bytes, void* out, float* lse, void* stream);

/*
 * mla_gather_kv_b_proj -- cached-prefix expansion of the paged latent into
 * full per-head keys and values through kv_b_proj ("perf(mla): chunk the
 * non-FP4 gather_kv_b_proj over KV", aiter PR 4776, description): for
 * sequence b, cached token j < seq_lens[b] and head h,
 *
 *   c_j = latent dims 0..511 of the token's cache row, r_j = rope dims 512..575
 *         (fp8 codes times kv_scale)
 *   k[t, h, 0:128]   = W[h, 0:128, :] c_j      k[t, h, 128:192] = r_j
 *   v[t, h, 0:128]   = W[h, 128:256, :] c_j
 *
 * with t = cu_seqlens[b] + j (the valid tokens, packed sequence by sequence).
 * One CTA per (sequence, 128-token chunk, group of 16 heads) on a grid sized
 * from max_ctx; chunks past a sequence's end return at once.  bf16 MMAs with
 * fp32 accumulation; k and v are rounded to bf16.
 *
 * kv_cache, num_pages, page_size, kv_dtype, kv_scale, block_table, bt_stride
 *              as mla_decode_fwd
 * seq_lens     device int32 [B], each <= max_ctx (larger values are clamped
 *              and set MLA_DEVFLAG_CTX_RANGE)
 * cu_seqlens   device int32 [B + 1], the exclusive prefix sums of seq_lens
 * max_ctx      host: the grid's extent, <= bt_stride * page_size
 * w_kv_b       device bf16 [H, 256, 512]: each head's 128 key rows, then its
 *              128 value rows (16-byte aligned)
 * k_out        device bf16 [cu_seqlens[B], H, 192]; v_out bf16 [.., H, 128]
 * status       device int32 status word (bad page ids, contexts, timeouts);
 *              the caller clears it
 * Returns MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED or MLA_ERR_CUDA.
 */
int mla_gather_kv_b_proj(const void* kv_cache, int64_t num_pages, int32_t page_size,
                         int32_t kv_dtype, const float* kv_scale, const int32_t* block_table,
                         int64_t bt_stride, const int32_t* seq_lens, const int32_t* cu_seqlens,
                         int32_t batch, int32_t max_ctx, const void* w_kv_b, int32_t num_heads,
                         void* k_out, void* v_out, int32_t* status, void* stream);

/*
 * mla_decode_epilogue -- the step just before the decode on every layer:
 * writes the 576-wide query rows and inserts each new token's latent row
 * into the paged cache.  "[Perf][Kimi-K3] Cut MLA decode concat/cache
 * epilogue latency" (vLLM PR 54896), Purpose items 1-3: the q-concat and
 * latent cache insert between the absorbed-q GEMM and the decode, bf16 or
 * fp8 cache, launched as a programmatic dependent of the GEMM.
 *
 *   q_out[t, h, 0:512]   = ql_nope[t, h, :]     q_out[t, h, 512:576] = q_pe[t, h, :]
 *   row                  = kv_c[t, :] || k_pe[t, :]                     (576 wide)
 *   cache[slot / page_size][slot % page_size][:] = row                  bf16 cache
 *                                              = e4m3(row / kv_scale)   fp8 cache
 * with slot = slot_mapping[t]; slot < 0 (a padding token) writes nothing.
 * The fp8 code is round-to-nearest-even of the fp32 quotient (correctly
 * rounded fp32 division), saturating to +-448.  q_pe and k_pe are taken as
 * already rotated (the rope is applied upstream).
 *
 * ql_nope      device bf16 [T, H, 512], contiguous, 16-byte aligned
 * q_pe         device bf16 [T, H, 64]
 * kv_c         device bf16 [T, 512]
 * k_pe         device bf16 [T, 64]
 * slot_mapping device int64 [T]: cache slot of token t (page * page_size + offset)
 * num_tokens   T >= 0 (0 queues nothing)
 * num_heads    H, 1 .. 128
 * q_out        device bf16 [T, H, 576]: the q of mla_decode_fwd
 * kv_cache     device [num_pages, page_size, 576] bf16 or e4m3 codes
 * kv_dtype     mla_kv_dtype of the cache; kv_scale device fp32[1] (fp8 only)
 * cache_inputs_early  1: kv_c and k_pe are older than the kernel this call
 *              is queued behind, so they are read before the dependency
 *              wait (as slot_mapping and kv_scale always are); 0: after it
 * status       optional device int32 status word (NULL = none): a slot
 *              >= num_pages * page_size is skipped and sets
 *              MLA_DEVFLAG_BAD_PAGE
 *
 * ql_nope and q_pe may be written by the kernel queued just before this one
 * (the dependency wait covers them); slot_mapping, kv_scale and, with
 * cache_inputs_early = 1, kv_c and k_pe must be older than that kernel.
 * Returns MLA_OK, MLA_ERR_INVALID_ARG or MLA_ERR_CUDA.
 */
int mla_decode_epilogue(const void* ql_nope, const void* q_pe, const void* kv_c,
                        const void* k_pe, const int64_t* slot_mapping, int32_t num_tokens,
                        int32_t num_heads, void* q_out, void* kv_cache, int64_t num_pages,
                        int32_t page_size, int32_t kv_dtype, const float* kv_scale,
                        int32_t cache_inputs_early, int32_t* status, void* stream);

/*
 * mla_decode_step -- one decode of the layer: mla_decode_epilogue for the
 * plan's batch * Sq new tokens (writing q and the new cache rows), then
 * mla_decode_fwd and mla_decode_combine, each kernel launched as a
 * programmatic dependent of the one before (the status word is reset before
 * the epilogue, so nothing but kernels sits between them on the stream).
 * The pages' chain of absorbed-q GEMM -> q-concat + cache insert -> decode,
 * "[Perf][Kimi-K3] Cut MLA decode concat/cache epilogue latency", Purpose.
 *
 * Arguments: the epilogue's inputs (T = plan->batch * plan->sq tokens in
 * sequence-major order, H = plan->num_heads), then those of mla_decode_fwd.
 * q is written here and read by the decode.  seq_lens count the new tokens,
 * whose rows this call inserts.  Returns as mla_decode_fwd.
 */
int mla_decode_step(const mla_decode_plan_t* plan, const void* ql_nope, const void* q_pe,
                    const void* kv_c, const void* k_pe, const int64_t* slot_mapping,
                    int32_t cache_inputs_early, void* q, void* kv_cache, int64_t num_pages,
                    const float* kv_scale, const int32_t* block_table, int64_t bt_stride,
                    const int32_t* seq_lens, float softmax_scale, void* out, float* lse,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_fwd_noalloc -- mla_decode_fwd followed by mla_decode_combine,
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart of this call.
 *
 * Who needs it: a plugin inside a server or framework whose host owns all
 * device memory through its own pool (a private cudaMalloc would bypass that
 * pool and its budget), or a latency-critical loop that must not call
 * cudaMalloc / cudaFree, which can synchronise the device.  Such a caller
 * cannot hand over a workspace; here the library uses its own scratch array.
 *
 * Arguments: as mla_decode_fwd, without workspace and workspace_bytes; the
 * caller still passes every input and both outputs.  out and lse are final on
 * return of the queued work (the combine is queued here too).
 *
 * Scratch: one fixed 64 MiB device array inside this library, created on
 * every GPU that loads it and held until the process exits.  Plans whose
 * plan->workspace_bytes exceed 64 MiB are rejected with MLA_ERR_WORKSPACE
 * (roughly batch * num_splits * H * Sq <= 32768 partial rows); a one-split
 * plan always fits.  The first call on each device looks the array's device
 * address up (cudaGetSymbolAddress, with that device current) and caches it;
 * make that first call before any stream capture.  Nothing is allocated or
 * freed, by this call or by anything it calls.
 *
 * All calls share the one array and it keeps the previous call's contents;
 * everything that must start at zero is reset on each call.  Calls whose work
 * overlaps on the GPU (different streams, no ordering between them) race on
 * the array: serialise them.  With no caller workspace there is no status
 * word to read back (mla_decode_check does not apply); out-of-range page ids
 * and contexts are still clamped on the device, never faulted.
 *
 * Returns MLA_OK, MLA_ERR_INVALID_ARG, MLA_ERR_WORKSPACE (plan too large for
 * the scratch), MLA_ERR_UNSUPPORTED (device ordinal >= 64) or MLA_ERR_CUDA.
 */
int mla_decode_fwd_noalloc(const mla_decode_plan_t* plan, const void* q, const void* kv_cache,
                           int64_t num_pages, const float* kv_scale, const int32_t* block_table,
                           int64_t bt_stride, const int32_t* seq_lens, float softmax_scale,
                           void* out, float* lse, void* stream);

/* Static text for a status code. */
const char* mla_status_string(int status);

/* Library version string, e.g. "mla_decode 0.1 sm_103a". */
const char* mla_decode_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
