// fwd_simt.cu -- first, plain CUDA-core version of the decode kernel.
//
// One CTA per (split, 16-row block, sequence).  Keys are streamed through
// shared memory 32 at a time; scores and the value sums run on the CUDA cores
// in fp32 with an online softmax in the log2 domain.  It computes exactly what
// the tcgen05 kernel computes and is the bring-up path of the library.

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/mla_decode.h"
#include "internal.h"

namespace {

constexpr int kRows = 16;
constexpr int kKeys = 32;
constexpr int kKStride = mla::kDQK + 1;
constexpr int kThreads = 256;
constexpr size_t kSmem = sizeof(float) * (kRows * mla::kDQK + kKeys * kKStride + kRows * kKeys);

__device__ __forceinline__ float bf16_to_f(uint16_t v) {
  return __uint_as_float(((uint32_t)v) << 16);
}

__device__ __forceinline__ float e4m3_to_f(uint8_t v) {
  __nv_fp8_e4m3 x;
  x.__x = v;
  return float(x);
}

__global__ void __launch_bounds__(kThreads) fwd_simt_kernel(mla::FwdParams p) {
  extern __shared__ float smem[];
  float* q_s = smem;                     // [16][576]
  float* k_s = q_s + kRows * mla::kDQK;  // [32][577]
  float* p_s = k_s + kKeys * kKStride;   // [16][32]
  __shared__ float m_s[kRows], l_s[kRows], alpha_s[kRows];

  const int split = blockIdx.x, rb = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int ctx = p.seq_lens[b];
  const int covered = p.num_splits * p.chunk_len;
  if (ctx > covered || ctx < 0) {
    if (tid == 0) atomicOr(p.status, MLA_DEVFLAG_CTX_RANGE);
    ctx = ctx < 0 ? 0 : covered;
  }
  const int k0 = split * p.chunk_len;
  const int k1 = min(k0 + p.chunk_len, ctx);
  const int r0 = rb * kRows;
  const float s_kv = (p.kv_dtype == MLA_KV_FP8_E4M3 && p.kv_scale) ? *p.kv_scale : 1.f;
  const float sl2 = p.softmax_scale * s_kv * 1.4426950408889634f;

  for (int i = tid; i < kRows * mla::kDQK; i += kThreads) {
    int r = r0 + i / mla::kDQK;
    q_s[i] = r < p.rows ? bf16_to_f(p.q[((size_t)b * p.rows + r) * mla::kDQK + i % mla::kDQK])
                        : 0.f;
  }
  if (tid < kRows) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }

  float acc[kRows][2];
#pragma unroll
  for (int r = 0; r < kRows; ++r) acc[r][0] = acc[r][1] = 0.f;

  const int lr = tid / 16;  // the row this thread scores
  const int row_lr = r0 + lr;
  int nvis = 0;
  if (row_lr < p.rows) {
    int i = row_lr / p.heads;
    nvis = p.causal ? ctx - p.sq + i + 1 : ctx;
    nvis = max(0, min(nvis, ctx));
  }

  for (int t0 = k0; t0 < k1; t0 += kKeys) {
    const int nk = min(kKeys, k1 - t0);
    __syncthreads();
    for (int i = tid; i < nk * mla::kDQK; i += kThreads) {
      int kk = i / mla::kDQK, d = i % mla::kDQK;
      int j = t0 + kk;
      int64_t page = p.bt[(size_t)b * p.bt_stride + j / p.page_size];
      if (page < 0 || page >= p.num_pages) {
        atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
        page = 0;
      }
      size_t idx = ((size_t)page * p.page_size + j % p.page_size) * mla::kDQK + d;
      k_s[kk * kKStride + d] =
          p.kv_dtype == MLA_KV_BF16 ? bf16_to_f(static_cast<const uint16_t*>(p.cache)[idx])
                                    : e4m3_to_f(static_cast<const uint8_t*>(p.cache)[idx]);
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int kk = (tid % 16) + 16 * h;
      float z = -INFINITY;
      if (kk < nk && t0 + kk < nvis) {
        float dot = 0.f;
        const float* qr = q_s + lr * mla::kDQK;
        const float* kr = k_s + kk * kKStride;
        for (int d = 0; d < mla::kDQK; ++d) dot = fmaf(qr[d], kr[d], dot);
        z = dot * sl2;
      }
      p_s[lr * kKeys + kk] = z;
    }
    __syncthreads();
    // online softmax: warp w owns rows 2w and 2w+1, one key per lane
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int r = warp * 2 + h;
      float v = p_s[r * kKeys + lane];
      float mt = v;
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      float m_old = m_s[r];
      float m_new = fmaxf(m_old, mt);
      float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
      float pv = (v == -INFINITY) ? 0.f : exp2f(v - m_new);
      float ps = pv;
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      p_s[r * kKeys + lane] = pv;
      __syncwarp();
      if (lane == 0) {
        m_s[r] = m_new;
        l_s[r] = l_s[r] * alpha + ps;
        alpha_s[r] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float alpha = alpha_s[r];
      acc[r][0] *= alpha;
      acc[r][1] *= alpha;
      for (int kk = 0; kk < nk; ++kk) {
        float w = p_s[r * kKeys + kk];
        acc[r][0] = fmaf(w, k_s[kk * kKStride + tid], acc[r][0]);
        acc[r][1] = fmaf(w, k_s[kk * kKStride + tid + 256], acc[r][1]);
      }
    }
  }
  __syncthreads();

#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int row = r0 + r;
    if (row >= p.rows) break;
    const float l = l_s[r], m = m_s[r];
    const float inv = l > 0.f ? s_kv / l : 0.f;
    const float lse = l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
    if (p.num_splits == 1) {
      uint16_t* o = p.out + ((size_t)b * p.rows + row) * mla::kDV;
      __nv_bfloat16 v0 = __float2bfloat16_rn(acc[r][0] * inv);
      __nv_bfloat16 v1 = __float2bfloat16_rn(acc[r][1] * inv);
      o[tid] = *reinterpret_cast<uint16_t*>(&v0);
      o[tid + 256] = *reinterpret_cast<uint16_t*>(&v1);
      if (tid == 0) p.lse[(size_t)b * p.rows + row] = lse;
    } else {
      size_t pr = ((size_t)b * p.num_splits + split) * p.rows + row;
      float* o = p.part_o + pr * mla::kDV;
      o[tid] = acc[r][0] * inv;
      o[tid + 256] = acc[r][1] * inv;
      if (tid == 0) p.part_lse[pr] = lse;
    }
  }
}

}  // namespace

int mla_launch_fwd_simt(const mla::FwdParams& p, void* stream) {
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmem);
  if (e != cudaSuccess) return (int)e;
  dim3 grid(p.num_splits, (p.rows + kRows - 1) / kRows, p.batch);
  fwd_simt_kernel<<<grid, kThreads, kSmem, static_cast<cudaStream_t>(stream)>>>(p);
  return (int)cudaGetLastError();
}
