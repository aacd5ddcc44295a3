// combine.cu -- log-sum-exp merge of the split-KV partials.
//
// Each split s of a row produced o_s (normalised over its own keys) and its
// log-sum-exp lse_s; the row's result is
//     L = ln sum_s exp(lse_s),   out = sum_s exp(lse_s - L) * o_s.
// The per-chunk slices come from the KV-chunk grid of "perf(mla): chunk the
// non-FP4 gather_kv_b_proj over KV" (aiter PR 4776, description); the merge
// itself follows from the per-row LSE output and is not written out on the
// pages.  Splits with no keys carry lse_s = -inf and are skipped (their o_s
// is never read, so it may hold anything).
//
// One 128-thread CTA per (row, sequence); each thread owns 4 of the 512
// value dims, so every partial row is read as one coalesced 2 KB sweep.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace {

__global__ void __launch_bounds__(128) combine_kernel(mla::CombineParams p) {
  const int r = blockIdx.x;
  const int b = blockIdx.y;
  __shared__ float w_s[mla::kMaxSplits];
  __shared__ float red[4];
  __shared__ float L_s;

  // Let the producing fwd kernel finish before reading its partials (a no-op
  // unless this grid was launched as a programmatic dependent launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // Splits of this sequence and the first one's partial slot: every
  // sequence has num_splits slots (host plan), or the device plan's count
  // (a sequence in one piece was written to out by the decode itself).
  int S = p.num_splits;
  size_t part0 = (size_t)b * S;
  if (p.seq_info != nullptr) {
    const int4 si = p.seq_info[b];
    if (si.z <= 1) return;
    S = si.z;
    part0 = (size_t)si.y;
  }
  const float* lse_row = p.part_lse + part0 * p.rows + r;
  float m = -INFINITY;
  for (int s = threadIdx.x; s < S; s += blockDim.x) m = fmaxf(m, lse_row[(size_t)s * p.rows]);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  __syncthreads();

  float sum = 0.f;
  for (int s = threadIdx.x; s < S; s += blockDim.x) {
    float ls = lse_row[(size_t)s * p.rows];
    float e = (ls == -INFINITY) ? 0.f : expf(ls - m);
    w_s[s] = e;
    sum += e;
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = red[0] + red[1] + red[2] + red[3];
    L_s = (m == -INFINITY) ? -INFINITY : m + logf(tot);
    red[0] = (m == -INFINITY) ? 0.f : 1.f / tot;
  }
  __syncthreads();
  const float inv = red[0];

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* o_base =
      reinterpret_cast<const float4*>(p.part_o + (part0 * p.rows + r) * mla::kDV) + threadIdx.x;
  const size_t stride = (size_t)p.rows * (mla::kDV / 4);
  // Eight splits' partial rows in flight at a time.  An empty split's row
  // holds anything (it was never written): its load is skipped and its
  // weight is zero.
  for (int s0 = 0; s0 < S; s0 += 8) {
    float4 v[8];
    float w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = s0 + u;
      w[u] = s < S ? w_s[s] : 0.f;
      v[u] = w[u] != 0.f ? o_base[(size_t)s * stride] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wu = w[u] * inv;
      acc.x += wu * v[u].x;
      acc.y += wu * v[u].y;
      acc.z += wu * v[u].z;
      acc.w += wu * v[u].w;
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  reinterpret_cast<uint2*>(p.out + ((size_t)b * p.rows + r) * mla::kDV)[threadIdx.x] = packed;
  if (threadIdx.x == 0) p.lse[(size_t)b * p.rows + r] = L_s;
}

}  // namespace

int mla_launch_combine(const mla::CombineParams& p, void* stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows, p.batch, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, combine_kernel, p);
}
