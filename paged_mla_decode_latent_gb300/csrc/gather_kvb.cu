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
// of up to kGroup heads.  The 128 gathered latent rows stay in shared memory
// for the whole group as the A operand (K-major, 128B-swizzled, 8 slabs of 64
// dims; fp8 codes converted to bf16 on the way in, exactly).  Each head's
// 256 x 512 weight block streams through a ring of 64-dim slabs (the B
// operand, 256 rows N); tcgen05 MMAs (M = 128, N = 256, K = 16) accumulate
// one head in 256 TMEM columns while four epilogue warps drain the previous
// head from the other 256 (fp32 -> bf16, x kv_scale for fp8).
//
// Warps: 0-2 weight loaders (one per ring stage), 3 MMA issue, 4-7 epilogue
// (TMEM lane quarters 0-3); the MMA and epilogue warps gather the latent
// rows first while the loaders start on the weights.  Every wait is
// bounded (2 s): a wait that runs out sets MLA_DEVFLAG_TIMEOUT and the CTA
// winds down.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla_decode.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int kTok = 128;           // tokens per CTA (MMA M)
constexpr int kN = 256;             // outputs per head (MMA N): 128 key + 128 value
constexpr int kLatent = 512;        // contraction (MMA K over 8 slabs)
constexpr int kSlabs = kLatent / 64;
constexpr int kGroup = 16;          // heads per CTA (the gathered rows serve them all)
constexpr int kStages = 3;          // weight slabs in flight
constexpr int A_SLAB = kTok * 128;  // 16 KB
constexpr int B_SLAB = kN * 128;    // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B = kSlabs * A_SLAB;           // 128 KB
constexpr int OFF_BAR = OFF_B + kStages * B_SLAB;  // 224 KB
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
static_assert(SMEM_BYTES <= 232448, "smem");
constexpr int kLoaders = kStages;  // weight loader warps, one per ring stage
constexpr int kWarps = kLoaders + 1 + 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kMmaWarp = kLoaders;
constexpr int kGatherThreads = kThreads - 32 * kLoaders;  // MMA + epilogue warps gather A
constexpr uint64_t kWaitNs = 2000000000ull;

struct Bars {
  uint64_t a_full;           // latent rows gathered (all threads)
  uint64_t b_full[kStages];  // weight slab landed (its loader warp's 32 lanes)
  uint64_t b_empty[kStages]; // weight slab consumed (MMA commit)
  uint64_t d_full[2];        // a head's accumulator complete (MMA commit)
  uint64_t d_empty[2];       // accumulator drained (128 epilogue threads)
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
};
static_assert(sizeof(Bars) <= 256, "barriers");

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

__global__ void __launch_bounds__(kThreads, 1) gather_kvb_kernel(GkvParams p) {
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
  const int h0 = group * kGroup;
  const int n_heads = min(kGroup, p.heads - h0);
  const int64_t t0 = (int64_t)p.cu_seqlens[b] + j0;
  const float s_kv = p.fp8 && p.kv_scale ? *p.kv_scale : 1.f;

  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bars.a_full), kGatherThreads);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars.b_full[s]), 32);
      ptx::mbar_init(ptx::smem_u32(&bars.b_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.d_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.d_empty[i]), 128);
    }
    ptx::mbar_init(ptx::smem_u32(&bars.drain), 1);
    bars.abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
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

  const int n_slabs = n_heads * kSlabs;
  if (warp >= kMmaWarp) {
    // ---- MMA and epilogue warps: gather the chunk's latent rows into A ----
    // A piece is 16 bytes of bf16 operand (8 dims), 64 per row, stored
    // 128B-swizzled in its 64-dim slab.  bf16: 16-byte cp.async copies, all
    // in flight at once.  fp8: 8 codes per piece loaded in batches of 8 and
    // converted (exactly) by the loading thread.  Rows past the sequence are
    // zero (their outputs are not stored).
    const int gt = threadIdx.x - 32 * kMmaWarp;
    const char* cache = static_cast<const char*>(p.cache);
    const int32_t* bt = p.bt + (size_t)b * p.bt_stride;
    bool bad = false;
    auto row_of = [&](int r) -> int64_t {
      const int j = j0 + r;
      int64_t page = bt[j / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        bad = true;
        page = 0;
      }
      return page * p.page_size + j % p.page_size;
    };
    auto dst_of = [&](int i) -> uint32_t {
      const int r = i >> 6, piece = i & 63;
      return sbase + OFF_A + (piece >> 3) * A_SLAB + r * 128 + (((piece & 7) ^ (r & 7)) * 16);
    };
    auto zero = [&](uint32_t dst) {
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
    };
    constexpr int kPieces = kTok * 64;
    if (!p.fp8) {
      for (int i = gt; i < kPieces; i += kGatherThreads) {
        const int r = i >> 6;
        if (r < n_tok)
          ptx::cp_async_16(dst_of(i), cache + (row_of(r) * MLA_D_QK + (i & 63) * 8) * 2);
        else
          zero(dst_of(i));
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
    } else {
      for (int i0 = gt; i0 < kPieces; i0 += 8 * kGatherThreads) {
        uint2 codes[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kGatherThreads, r = i >> 6;
          codes[u] = (i < kPieces && r < n_tok)
                         ? *reinterpret_cast<const uint2*>(cache + row_of(r) * MLA_D_QK + (i & 63) * 8)
                         : make_uint2(0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u * kGatherThreads;
          if (i >= kPieces) break;
          const uint32_t x = e4m3x2_to_bf16x2(codes[u].x), y = e4m3x2_to_bf16x2(codes[u].x >> 16);
          const uint32_t z = e4m3x2_to_bf16x2(codes[u].y), w = e4m3x2_to_bf16x2(codes[u].y >> 16);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst_of(i)), "r"(x),
                       "r"(y), "r"(z), "r"(w)
                       : "memory");
        }
      }
    }
    if (bad) atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(ptx::smem_u32(&bars.a_full));
  }

  if (warp < kLoaders) {
    // ------------------------------------------------- weight loaders ---
    // Loader warp w owns ring stage w and fills slabs w, w + kStages, ...:
    // 256 rows x 128 B of one head's block, 16-byte pieces into the
    // 128B-swizzled K-major layout; it waits for its own copies, fences them
    // for the tensor cores and arrives on the stage's barrier.
    for (int i = warp; i < n_slabs; i += kStages) {
      const int s = warp;
      if (i >= kStages && !wait_all(c, ptx::smem_u32(&bars.b_empty[s]), ((i / kStages) - 1) & 1))
        break;
      const int h = h0 + i / kSlabs, k = i % kSlabs;
      const uint16_t* src = p.w + ((size_t)h * kN) * kLatent + k * 64;
      const uint32_t dst = sbase + OFF_B + s * B_SLAB;
#pragma unroll 4
      for (int q = lane; q < kN * 8; q += 32) {
        const int o = q >> 3, piece = q & 7;
        ptx::cp_async_16(dst + o * 128 + ((piece ^ (o & 7)) * 16), src + (size_t)o * kLatent + piece * 8);
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&bars.b_full[s]));
    }
    ptx::cp_async_wait<0>();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_f16(128, kN, 1u, false, false);
      bool ok = wait(c, ptx::smem_u32(&bars.a_full), 0);
      ptx::tc_fence_after();
      for (int hh = 0; ok && hh < n_heads; ++hh) {
        const int buf = hh & 1;
        if (hh >= 2 && !wait(c, ptx::smem_u32(&bars.d_empty[buf]), ((hh >> 1) - 1) & 1)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * kN;
        for (int k = 0; k < kSlabs; ++k) {
          const int i = hh * kSlabs + k, s = i % kStages;
          if (!wait(c, ptx::smem_u32(&bars.b_full[s]), (i / kStages) & 1)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a = sbase + OFF_A + k * A_SLAB, bb = sbase + OFF_B + s * B_SLAB;
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ss(d, kdesc(a + kk * 32), kdesc(bb + kk * 32), idesc, (k | kk) != 0);
          ptx::mma_commit(ptx::smem_u32(&bars.b_empty[s]));
        }
        if (!ok) break;
        ptx::mma_commit(ptx::smem_u32(&bars.d_full[buf]));
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue ---
    // Thread i of epilogue warp w owns TMEM lane 32 (w % 4) + i, i.e. token
    // row r of the chunk; it writes that token's rope dims once per head,
    // then each head's 128 key and 128 value dims.
    const int q4 = warp & 3;  // warps 4-7: lane quarters 0-3
    const int r = q4 * 32 + lane;
    const bool valid = r < n_tok;
    const int64_t t = t0 + r;
    if (valid) {
      const int j = j0 + r;
      int64_t page = p.bt[(size_t)b * p.bt_stride + j / p.page_size];
      if (page < 0 || page >= p.num_pages) page = 0;
      const int64_t row = page * p.page_size + j % p.page_size;
      uint4 rope[8];
      const char* cache = static_cast<const char*>(p.cache);
      if (p.fp8) {
        const uint4* src = reinterpret_cast<const uint4*>(cache + row * MLA_D_QK + 512);
        for (int v = 0; v < 4; ++v) {
          const uint4 x = src[v];
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
          uint32_t o8[8];
          for (int e = 0; e < 4; ++e) {
            const uint32_t bf0 = e4m3x2_to_bf16x2(w4[e]), bf1 = e4m3x2_to_bf16x2(w4[e] >> 16);
            o8[2 * e] = pack_bf16(__uint_as_float(bf0 << 16) * s_kv,
                                  __uint_as_float(bf0 & 0xFFFF0000u) * s_kv);
            o8[2 * e + 1] = pack_bf16(__uint_as_float(bf1 << 16) * s_kv,
                                      __uint_as_float(bf1 & 0xFFFF0000u) * s_kv);
          }
          rope[2 * v] = make_uint4(o8[0], o8[1], o8[2], o8[3]);
          rope[2 * v + 1] = make_uint4(o8[4], o8[5], o8[6], o8[7]);
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(cache + (row * MLA_D_QK + 512) * 2);
        for (int v = 0; v < 8; ++v) rope[v] = src[v];
      }
      for (int hh = 0; hh < n_heads; ++hh) {
        uint4* dst = reinterpret_cast<uint4*>(p.k_out + (t * p.heads + h0 + hh) * 192 + 128);
        for (int v = 0; v < 8; ++v) dst[v] = rope[v];
      }
    }
    const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
    for (int hh = 0; hh < n_heads; ++hh) {
      const int buf = hh & 1;
      if (!wait_all(c, ptx::smem_u32(&bars.d_full[buf]), (hh >> 1) & 1)) break;
      ptx::tc_fence_after();
      const int h = h0 + hh;
#pragma unroll 1
      for (int part = 0; part < kN / 32; ++part) {
        uint32_t x[32];
        ptx::tmem_ld32(tmem + lanes + buf * kN + part * 32, x);
        ptx::tmem_ld_wait();
        if (valid) {
          uint16_t* dst = part < 4 ? p.k_out + (t * p.heads + h) * 192 + part * 32
                                   : p.v_out + (t * p.heads + h) * 128 + (part - 4) * 32;
          uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_bf16(__uint_as_float(x[8 * v + 2 * e]) * s_kv,
                               __uint_as_float(x[8 * v + 2 * e + 1]) * s_kv);
            d4[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.d_empty[buf]));
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
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (mla::opt_in_smem(reinterpret_cast<const void*>(gather_kvb_kernel), SMEM_BYTES, dev, 2) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((max_ctx + kTok - 1) / kTok, (num_heads + kGroup - 1) / kGroup, batch);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, gather_kvb_kernel, p) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}
