// epilogue.cu -- the step before the decode on every layer: the 576-wide
// query rows (ql_nope || q_pe) and the insert of each new token's latent row
// (kv_c || k_pe) into the paged cache through slot_mapping, as bf16 or as
// fp8 E4M3 codes of x / kv_scale.
//
// Source: "[Perf][Kimi-K3] Cut MLA decode concat/cache epilogue latency"
// (vLLM PR 54896), Purpose items 1-3.  Kept from it: one 8-element
// load -> convert -> store per thread (16 bytes of bf16 in, 16 bytes of bf16
// or 8 bytes of fp8 out); the inputs that are older than the producing GEMM
// (slot_mapping, kv_scale and, when the caller says so, the cache-row inputs)
// read before the programmatic dependency wait, the query inputs after it;
// the dependent launch triggered right after that wait so the decode's
// prologue overlaps this kernel's last round trip.  Different from it: the
// page's kernel splits a row over 3 warps up to 64 tokens and keeps one warp
// per row beyond; here every size uses the flat form, one thread per 16-byte
// piece of a row (72 per row), so no token-count dispatch is needed.
//
// Rows: token t has H query rows and one cache row.  Thread i of the grid
// handles piece i % 72 of row i / 72, rows ordered (token, H query rows +
// the cache row).  Pieces 0..63 come from the 512 latent dims, 64..71 from
// the 64 rope dims.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla_decode.h"
#include "internal.h"

namespace {

constexpr int kPieces = 72;  // 16-byte pieces of a 576-wide bf16 row
constexpr int kThreads = 256;

struct EpiParams {
  const uint16_t* ql_nope;  // bf16 [T, H, 512]
  const uint16_t* q_pe;     // bf16 [T, H, 64]
  const uint16_t* kv_c;     // bf16 [T, 512]
  const uint16_t* k_pe;     // bf16 [T, 64]
  const int64_t* slot_mapping;  // [T]; < 0 = no insert
  uint16_t* q_out;          // bf16 [T, H, 576]
  void* cache;              // [num_pages, page_size, 576] bf16 or e4m3
  const float* kv_scale;    // fp8 only
  int32_t* status;          // optional
  int64_t num_slots;        // num_pages * page_size
  int tokens, heads, fp8, cache_early;
};

// Two fp32 -> two e4m3 codes (round to nearest even, saturating to +-448;
// the first value in the low byte).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float first, float second) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

__global__ void __launch_bounds__(kThreads) epilogue_kernel(EpiParams p) {
  const int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t rows_per_token = p.heads + 1;
  const int64_t n = (int64_t)p.tokens * rows_per_token * kPieces;
  const bool active = i < n;
  const int piece = (int)(i % kPieces);
  const int64_t row = i / kPieces;
  const int t = (int)(row / rows_per_token);
  const int h = (int)(row % rows_per_token);  // h == heads: the cache row
  const bool cache_row = active && h == p.heads;

  // Older inputs first: the slot and, if the caller allows it, the cache row.
  int64_t slot = -1;
  uint4 v = make_uint4(0, 0, 0, 0);
  if (cache_row) {
    slot = p.slot_mapping[t];
    if (p.cache_early) {
      v = piece < 64 ? reinterpret_cast<const uint4*>(p.kv_c + (int64_t)t * 512)[piece]
                     : reinterpret_cast<const uint4*>(p.k_pe + (int64_t)t * 64)[piece - 64];
    }
  }
  // ql_nope / q_pe may come from the kernel this one is launched behind.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!active) return;
  if (!cache_row) {
    const int64_t qrow = (int64_t)t * p.heads + h;
    const uint4 x = piece < 64 ? reinterpret_cast<const uint4*>(p.ql_nope + qrow * 512)[piece]
                               : reinterpret_cast<const uint4*>(p.q_pe + qrow * 64)[piece - 64];
    reinterpret_cast<uint4*>(p.q_out + qrow * MLA_D_QK)[piece] = x;
    return;
  }
  if (!p.cache_early) {
    v = piece < 64 ? reinterpret_cast<const uint4*>(p.kv_c + (int64_t)t * 512)[piece]
                   : reinterpret_cast<const uint4*>(p.k_pe + (int64_t)t * 64)[piece - 64];
  }
  if (slot < 0) return;  // padding token: no insert
  if (slot >= p.num_slots) {
    if (piece == 0 && p.status) atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
    return;
  }
  if (!p.fp8) {
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.cache) + slot * MLA_D_QK)[piece] = v;
    return;
  }
  const float s = *p.kv_scale;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t codes[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t word = w[2 * k + e];
      const float lo = __fdiv_rn(__uint_as_float(word << 16), s);
      const float hi = __fdiv_rn(__uint_as_float(word & 0xFFFF0000u), s);
      c |= (uint32_t)f32x2_to_e4m3x2(lo, hi) << (16 * e);
    }
    codes[k] = c;
  }
  reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.cache) + slot * MLA_D_QK)[piece] =
      make_uint2(codes[0], codes[1]);
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; }

}  // namespace

extern "C" int mla_decode_epilogue(const void* ql_nope, const void* q_pe, const void* kv_c,
                                   const void* k_pe, const int64_t* slot_mapping,
                                   int32_t num_tokens, int32_t num_heads, void* q_out,
                                   void* kv_cache, int64_t num_pages, int32_t page_size,
                                   int32_t kv_dtype, const float* kv_scale,
                                   int32_t cache_inputs_early, int32_t* status, void* stream) {
  if (num_tokens < 0 || num_heads < 1 || num_heads > 128 || page_size < 1 || num_pages < 1)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (cache_inputs_early != 0 && cache_inputs_early != 1) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (!ql_nope || !q_pe || !kv_c || !k_pe || !slot_mapping || !q_out || !kv_cache)
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !kv_scale) return MLA_ERR_INVALID_ARG;
  if (!aligned16(ql_nope) || !aligned16(q_pe) || !aligned16(kv_c) || !aligned16(k_pe) ||
      !aligned16(q_out) || !aligned16(kv_cache) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7))
    return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && (reinterpret_cast<uintptr_t>(kv_scale) & 3))
    return MLA_ERR_INVALID_ARG;
  EpiParams p;
  p.ql_nope = static_cast<const uint16_t*>(ql_nope);
  p.q_pe = static_cast<const uint16_t*>(q_pe);
  p.kv_c = static_cast<const uint16_t*>(kv_c);
  p.k_pe = static_cast<const uint16_t*>(k_pe);
  p.slot_mapping = slot_mapping;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.cache = kv_cache;
  p.kv_scale = kv_scale;
  p.status = status;
  p.num_slots = num_pages * (int64_t)page_size;
  p.tokens = num_tokens;
  p.heads = num_heads;
  p.fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  p.cache_early = cache_inputs_early;
  const int64_t threads = (int64_t)num_tokens * (num_heads + 1) * kPieces;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((threads + kThreads - 1) / kThreads), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, epilogue_kernel, p) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}
