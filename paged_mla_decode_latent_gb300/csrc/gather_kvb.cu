// gather_kvb.cu -- cached-prefix expansion of the paged latent into per-head
// keys and values ("gather_kv_b_proj"): for every cached token j of sequence
// b and head h,
//   k[t, h, 0:128]   = W[h][0:128]   . c_j       k[t, h, 128:192] = r_j
//   v[t, h, 0:128]   = W[h][128:256] . c_j
// with c_j / r_j the token's 512 latent / 64 rope dims read through the block
// table (fp8 codes times kv_scale), W = kv_b_proj [H][256][512] bf16 and
// t = cu_seqlens[b] + j the packed output row.
//
// Source: "perf(mla): chunk the non-FP4 gather_kv_b_proj over KV" (aiter PR
// 4776), description: the expansion over the whole cached context, one
// program per (batch, head group, KV chunk) on the grid instead of a serial
// loop over chunks, chunks past a sequence's end returning at once, each
// chunk storing its own slice.
//
// GB300 form: a CTA takes 128 tokens of one sequence (the MMA M) and a group
// of up to kGroup heads (fewer when that leaves SMs idle: see the launcher).  The 128 gathered latent rows go into TMEM as the A
// operand (256 columns of bf16 pairs; fp8 codes converted exactly on the
// way), so shared memory holds only the weights: each (head, key or value
// half) unit's 128 x 512 block streams through a ring of twelve 64-dim
// slabs (16 KB each, the B operand, K-major 128B-swizzled), each one TMA tile
// load of the weight tensor, about 192 KB in flight.  tcgen05 MMAs (M = 128, N = 128, K = 16, A from TMEM) accumulate a
// unit in one of two 128-column TMEM accumulators while four epilogue warps
// drain the other (fp32 -> bf16, x kv_scale for fp8).
//
// Warps: 0 weight loads (one thread issues the TMA loads), 1-2 idle, 3 MMA issue,
// 4-7 gather the rows into TMEM, write the rope dims and drain the
// accumulators (TMEM lane quarters 0-3).  Every wait is bounded (2 s): a
// wait that runs out sets MLA_DEVFLAG_TIMEOUT and the CTA winds down.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/mla_decode.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int kTok = 128;           // tokens per CTA (MMA M)
constexpr int kUnitN = 128;         // outputs per unit (MMA N): a head's keys or its values
constexpr int kLatent = 512;        // contraction (MMA K over 8 slabs)
constexpr int kSlabs = kLatent / 64;
constexpr int kGroup = 16;          // heads per CTA (the gathered rows serve them all)
constexpr int kStages = 12;         // weight slabs in flight (16 KB each)
constexpr int B_SLAB = kUnitN * 128;           // 16 KB
constexpr int OFF_B = 0;
constexpr int STG_W = 32 * 256;                    // a warp's 32 output rows of 256 B
constexpr int OFF_STG = OFF_B + kStages * B_SLAB;  // 192 KB: output staging, 4 x 8 KB
constexpr int OFF_BAR = OFF_STG + 4 * STG_W;       // 224 KB
constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;
static_assert(SMEM_BYTES <= 232448, "smem");
constexpr int kMmaWarp = 3;
constexpr int kThreads = 32 * 8;
constexpr uint32_t TM_A = 0;    // 256 columns: the 512 latent dims as bf16 pairs
constexpr uint32_t TM_D = 256;  // two 128-column accumulators
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint64_t kDrainNs = 500000000ull;

struct Bars {
  uint64_t a_full;            // rows in TMEM (128 gather threads)
  uint64_t b_full[kStages];   // weight slab landed (its loader warp's 32 lanes)
  uint64_t b_empty[kStages];  // weight slab consumed (MMA commit)
  uint64_t d_full[2];         // a unit's accumulator complete (MMA commit)
  uint64_t d_empty[2];        // accumulator drained (128 epilogue threads)
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 512, "barriers");

struct GkvParams {
  const void* cache;
  int64_t num_pages;
  const float* kv_scale;
  const int32_t* bt;
  int64_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* cu_seqlens;
  const uint16_t* w;  // bf16 [H, 256, 512]
  uint16_t* k_out;    // bf16 [T, H, 192]
  uint16_t* v_out;    // bf16 [T, H, 128]
  int32_t* status;
  int page_size, fp8, heads, max_ctx;
  int group;  // heads per CTA
};

struct Ctx {
  int32_t* status;
  volatile int32_t* abort;
};

__device__ __forceinline__ bool wait(const Ctx& c, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, 20000)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(c.status, MLA_DEVFLAG_TIMEOUT);
      *c.abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_all(const Ctx& c, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(c, bar, parity));
}

__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
  // e4m3 -> f16 is exact, and so is f16 -> bf16 for every e4m3 value
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two_codes));
  const float lo = __half2float(__ushort_as_half((uint16_t)(h & 0xFFFF)));
  const float hi = __half2float(__ushort_as_half((uint16_t)(h >> 16)));
  return (__float_as_uint(hi) & 0xFFFF0000u) | (__float_as_uint(lo) >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// K-major, 128B-swizzled operand: rows 128 B apart, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return ptx::smem_desc(addr, 16, 1024, 2); }

__global__ void __launch_bounds__(kThreads, 1)
    gather_kvb_kernel(GkvParams p, const __grid_constant__ CUtensorMap wmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, group = blockIdx.y, b = blockIdx.z;

  ptx::grid_dependency_wait();
  int ctx = p.seq_lens[b];
  if (ctx < 0 || ctx > p.max_ctx) {
    if (threadIdx.x == 0 && chunk == 0 && group == 0) atomicOr(p.status, MLA_DEVFLAG_CTX_RANGE);
    ctx = ctx < 0 ? 0 : p.max_ctx;
  }
  const int j0 = chunk * kTok;
  if (j0 >= ctx) return;  // past this sequence's last chunk
  const int n_tok = min(kTok, ctx - j0);
  const int h0 = group * p.group;
  const int n_heads = min(p.group, p.heads - h0);
  const int n_units = 2 * n_heads;  // (head, keys or values)
  const int n_slabs = n_units * kSlabs;
  const int64_t t0 = (int64_t)p.cu_seqlens[b] + j0;
  const float s_kv = p.fp8 && p.kv_scale ? *p.kv_scale : 1.f;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars.a_full), 128);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars.b_full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.b_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.d_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.d_empty[i]), 128);
    }
    ptx::mbar_init(ptx::smem_u32(&bars.drain), 1);
    bars.abort = 0;
    ptx::fence_mbar_init_cluster();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars.tmem_base), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars.tmem_base;
  Ctx c{p.status, &bars.abort};

  if (warp == 0) {
    // ------------------------------------------------- weight loader ---
    // One thread fills slab i (slab k = i % 8 of unit i / 8: 128 weight rows
    // x 64 dims) into stage i % 12 with one TMA tile load (the map's 128-byte
    // swizzle gives the K-major operand layout), counted on the stage's
    // barrier; a stage is refilled once the MMAs that read it are done.
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < n_slabs; ++i) {
        const int s = i % kStages;
        if (i >= kStages && !wait(c, ptx::smem_u32(&bars.b_empty[s]), ((i / kStages) - 1) & 1)) break;
        const int unit = i / kSlabs, k = i % kSlabs;
        const int h = h0 + (unit >> 1), x = unit & 1;
        ptx::mbar_arrive_expect_tx(ptx::smem_u32(&bars.b_full[s]), B_SLAB);
        ptx::tma_load_2d(sbase + OFF_B + s * B_SLAB, &wmap, k * 64, h * 256 + x * kUnitN,
                         ptx::smem_u32(&bars.b_full[s]));
        ++issued;
      }
      // No copy may still be landing when the CTA leaves (after a wind-down
      // the MMA warp may not have consumed them): wait for the last ones.
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        const uint32_t bar = ptx::smem_u32(&bars.b_full[i % kStages]);
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, (i / kStages) & 1))
          if (ptx::globaltimer_ns() - t0 > kDrainNs) break;
      }
    }
    __syncwarp();
  } else if (warp < kMmaWarp) {
    // warps 1 and 2: no work
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_f16(128, kUnitN, 1u, false, false);
      bool ok = wait(c, ptx::smem_u32(&bars.a_full), 0);
      ptx::tc_fence_after();
      for (int uu = 0; ok && uu < n_units; ++uu) {
        const int buf = uu & 1;
        if (uu >= 2 && !wait(c, ptx::smem_u32(&bars.d_empty[buf]), ((uu >> 1) - 1) & 1)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + TM_D + buf * kUnitN;
        for (int k = 0; k < kSlabs; ++k) {
          const int i = uu * kSlabs + k, s = i % kStages;
          if (!wait(c, ptx::smem_u32(&bars.b_full[s]), (i / kStages) & 1)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t bb = sbase + OFF_B + s * B_SLAB;
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ts(d, tmem + TM_A + k * 32 + kk * 8, kdesc(bb + kk * 32), idesc, (k | kk) != 0);
          ptx::mma_commit(ptx::smem_u32(&bars.b_empty[s]));
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&bars.d_full[buf]));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------- gather and epilogue ---
    // Thread i of warp w (4..7) owns TMEM lane 32 (w % 4) + i, i.e. token row
    // r of the chunk.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const bool valid = r < n_tok;
    const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
    const char* cache = static_cast<const char*>(p.cache);
    int64_t row = 0;
    if (valid) {
      const int j = j0 + r;
      int64_t page = p.bt[(size_t)b * p.bt_stride + j / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
        page = 0;
      }
      row = page * p.page_size + j % p.page_size;
    }
    // The row's 512 latent dims -> TMEM (columns = dims / 2), 128 dims a batch.
    for (int bq = 0; bq < 4; ++bq) {
      uint32_t w[64];
      if (!p.fp8) {
        const uint4* src = reinterpret_cast<const uint4*>(cache + (row * MLA_D_QK + bq * 128) * 2);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const uint4 x = valid ? src[v] : make_uint4(0, 0, 0, 0);
          w[4 * v] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(cache + row * MLA_D_QK + bq * 128);
        uint4 x[8];
#pragma unroll
        for (int v = 0; v < 8; ++v) x[v] = valid ? src[v] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint32_t cw[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            w[8 * v + 2 * e] = e4m3x2_to_bf16x2(cw[e]);
            w[8 * v + 2 * e + 1] = e4m3x2_to_bf16x2(cw[e] >> 16);
          }
        }
      }
      ptx::tmem_st32(tmem + lanes + TM_A + bq * 64, *reinterpret_cast<uint32_t(*)[32]>(w));
      ptx::tmem_st32(tmem + lanes + TM_A + bq * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(w + 32));
    }
    ptx::tmem_st_wait();
    ptx::tc_fence_before();
    ptx::mbar_arrive(ptx::smem_u32(&bars.a_full));

    // Output rows are H * 384 B (keys) or H * 256 B (values) apart, so a
    // thread writing its own token's row would touch 32 lines per warp
    // store.  Instead the warp's 32 rows go through its staging tile (8 KB,
    // 16-byte chunks swizzled by the row) and leave as whole rows: lanes
    // 16 k .. 16 k + 15 write 16 bytes each of one row, two rows per store.
    const uint32_t stg = sbase + OFF_STG + q4 * STG_W;
    const int half = lane >> 4, cl = lane & 15;
    // The rope dims, once per head: 8 lanes per 128-byte rope row, 4 rows a
    // store, each chunk read once from the cache and written for every head.
    {
      const int c8 = lane & 7;
      for (int it = 0; it < 8; ++it) {
        const int rr = q4 * 32 + it * 4 + (lane >> 3);
        if (rr >= n_tok) continue;
        const int j = j0 + rr;
        int64_t page = p.bt[(size_t)b * p.bt_stride + j / p.page_size];
        if (page < 0 || page >= p.num_pages) page = 0;
        const int64_t crow = page * p.page_size + j % p.page_size;
        uint4 v;
        if (p.fp8) {
          const uint2 codes = *reinterpret_cast<const uint2*>(cache + crow * MLA_D_QK + 512 + c8 * 8);
          const uint32_t cw[2] = {codes.x, codes.y};
          uint32_t o4[4];
          for (int e = 0; e < 2; ++e) {
            const uint32_t bf0 = e4m3x2_to_bf16x2(cw[e]), bf1 = e4m3x2_to_bf16x2(cw[e] >> 16);
            o4[2 * e] = pack_bf16(__uint_as_float(bf0 << 16) * s_kv,
                                  __uint_as_float(bf0 & 0xFFFF0000u) * s_kv);
            o4[2 * e + 1] = pack_bf16(__uint_as_float(bf1 << 16) * s_kv,
                                      __uint_as_float(bf1 & 0xFFFF0000u) * s_kv);
          }
          v = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        } else {
          v = *reinterpret_cast<const uint4*>(cache + (crow * MLA_D_QK + 512 + c8 * 8) * 2);
        }
        for (int hh = 0; hh < n_heads; ++hh)
          *reinterpret_cast<uint4*>(p.k_out + ((t0 + rr) * p.heads + h0 + hh) * 192 + 128 + c8 * 8) = v;
      }
    }
    // Drain each unit: keys to k[t, h, 0:128], values to v[t, h, 0:128].
    for (int uu = 0; uu < n_units; ++uu) {
      const int buf = uu & 1;
      if (!wait_all(c, ptx::smem_u32(&bars.d_full[buf]), (uu >> 1) & 1)) break;
      ptx::tc_fence_after();
      const int h = h0 + (uu >> 1);
      // All four 32-column loads in flight before one wait.
      uint32_t x[4][32];
#pragma unroll
      for (int part = 0; part < kUnitN / 32; ++part)
        ptx::tmem_ld32(tmem + lanes + TM_D + buf * kUnitN + part * 32, x[part]);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int part = 0; part < kUnitN / 32; ++part) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = pack_bf16(__uint_as_float(x[part][8 * v + 2 * e]) * s_kv,
                             __uint_as_float(x[part][8 * v + 2 * e + 1]) * s_kv);
          const int chunk = part * 4 + v;  // 16-byte chunk of this row (0..15)
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(
                           stg + lane * 256 + ((chunk ^ (lane & 15)) * 16)),
                       "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
      }
      // The accumulator is read: the MMAs may reuse it while the rows leave.
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.d_empty[buf]));
      __syncwarp();
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const int lr = 2 * k + half;  // the warp's row
        const int rr = q4 * 32 + lr;
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(stg + lr * 256 + ((cl ^ (lr & 15)) * 16))
                     : "memory");
        if (rr < n_tok) {
          uint16_t* dst = buf == 0 ? p.k_out + ((t0 + rr) * p.heads + h) * 192
                                   : p.v_out + ((t0 + rr) * p.heads + h) * 128;
          reinterpret_cast<uint4*>(dst)[cl] = v;
        }
      }
      __syncwarp();
    }
  }

  // ------------------------------------------------------------ teardown ---
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    if (bars.abort) {
      if (lane == 0) {
        ptx::mma_commit(ptx::smem_u32(&bars.drain));
        const uint64_t t1 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(ptx::smem_u32(&bars.drain), 0))
          if (ptx::globaltimer_ns() - t1 > kWaitNs / 4) break;
      }
      __syncwarp();
    }
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

namespace {

// The driver's tensor-map encoder, looked up once through the runtime (no
// link-time dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static void* fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
  });
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

}  // namespace

extern "C" int mla_gather_kv_b_proj(const void* kv_cache, int64_t num_pages, int32_t page_size,
                                    int32_t kv_dtype, const float* kv_scale,
                                    const int32_t* block_table, int64_t bt_stride,
                                    const int32_t* seq_lens, const int32_t* cu_seqlens,
                                    int32_t batch, int32_t max_ctx, const void* w_kv_b,
                                    int32_t num_heads, void* k_out, void* v_out, int32_t* status,
                                    void* stream) {
  if (!kv_cache || !block_table || !seq_lens || !cu_seqlens || !w_kv_b || !k_out || !v_out ||
      !status)
    return MLA_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || num_heads < 1 || num_heads > 128 || page_size < 1 ||
      page_size > 4096 || num_pages < 1 || bt_stride < 1 || max_ctx < 0)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (bt_stride * (int64_t)page_size < (int64_t)max_ctx) return MLA_ERR_INVALID_ARG;
  if (num_pages * (int64_t)page_size >= ((int64_t)1 << 31)) return MLA_ERR_UNSUPPORTED;
  auto mis = [](const void* x, uintptr_t a) { return (reinterpret_cast<uintptr_t>(x) % a) != 0; };
  if (mis(kv_cache, 16) || mis(w_kv_b, 16) || mis(k_out, 16) || mis(v_out, 16) ||
      mis(block_table, 4) || mis(seq_lens, 4) || mis(cu_seqlens, 4) || mis(status, 4))
    return MLA_ERR_INVALID_ARG;
  if (max_ctx == 0) return MLA_OK;
  GkvParams p;
  p.cache = kv_cache;
  p.num_pages = num_pages;
  p.kv_scale = kv_dtype == MLA_KV_FP8_E4M3 ? kv_scale : nullptr;
  p.bt = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.cu_seqlens = cu_seqlens;
  p.w = static_cast<const uint16_t*>(w_kv_b);
  p.k_out = static_cast<uint16_t*>(k_out);
  p.v_out = static_cast<uint16_t*>(v_out);
  p.status = status;
  p.page_size = page_size;
  p.fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  p.heads = num_heads;
  p.max_ctx = max_ctx;
  int dev = 0, num_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (mla::opt_in_smem(reinterpret_cast<const void*>(gather_kvb_kernel), SMEM_BYTES, dev, 2) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  // Heads per CTA.  A CTA's (head, keys / values) units run one after the
  // other, so its time is about (gather + g heads) and the launch takes
  // ceil(CTAs / SMs) such rounds (one CTA per SM).  Few chunks (short
  // contexts) leave most SMs idle with all heads in one CTA; smaller groups
  // spread the heads, each CTA gathering the same rows again (from L2).
  // The cost is counted in heads, the gather and fill taken as half a head.
  const int64_t chunks = (int64_t)((max_ctx + kTok - 1) / kTok) * batch;
  int group = std::min(kGroup, num_heads);
  double best = 1e300;
  for (int g = std::min(kGroup, num_heads); g >= 1; --g) {
    const int64_t ctas = chunks * ((num_heads + g - 1) / g);
    const double t = (double)((ctas + num_sms - 1) / num_sms) * (0.5 + g);
    if (t < best * 0.97) {  // a smaller group only for a clear gain
      best = t;
      group = g;
    }
  }
  p.group = group;
  // The weights [H, 256, 512] as a 2-D tensor of H * 256 rows of 512 bf16,
  // read in boxes of 128 rows x 64 dims with the 128-byte swizzle of the
  // K-major operand.
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return MLA_ERR_CUDA;
  CUtensorMap wmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)kLatent, (cuuint64_t)num_heads * 256};
  const cuuint64_t gstride[1] = {(cuuint64_t)kLatent * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kUnitN};
  const cuuint32_t estride[2] = {1, 1};
  if (encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_kv_b), gdim, gstride,
             box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_ctx + kTok - 1) / kTok, (num_heads + group - 1) / group, batch);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gather_kvb_kernel, p, wmap) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}
