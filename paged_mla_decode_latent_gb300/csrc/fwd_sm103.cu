// fwd_sm103.cu -- the decode kernel on the 5th-generation tensor cores.
//
// Work unit: one (sequence b, 128-row block, KV split) handled by a cluster of
// two CTAs; grid (2 x row blocks, sequences, splits).  Rows are the Sq*H query rows of the sequence (token-major, as q
// is laid out), padded to the MMA M of 128.  The fp32 output accumulator of
// 128 rows x 512 value dims would fill all 512 TMEM columns of one SM, so the
// two CTAs split the value dims: CTA r owns value dims [256r, 256r+256) and,
// for the score contraction, the same 256 latent dims and half of the 64
// rope dims (CTA r: rope dims [32r, 32r+32)), so both CTAs issue the same
// number of MMAs.  Each CTA therefore reads only its part of every latent row.
//
// Per 64-key tile, in each CTA:
//   loader warps  : three warps take turns by tile, one per
//                   operand stage: block-table lookup, then
//                   16-byte cp.async of the tile's rows in 128-byte pieces
//                   (one 64-dim slab of one key; of the rope slab, the CTA's
//                   64-byte half) straight into a 128B-swizzled
//                   K-major stage (bf16), or into a raw stage the same lanes
//                   convert to f16 (fp8); each lane fences its own copies for
//                   the tensor cores and arrives on the stage's barrier.
//   MMA warp      : S_part = Q_part K_part^T  (tcgen05, A = Q from TMEM,
//                   the rope part's A from shared memory), then
//                   O_half += P V_half        (A = P from TMEM, B = the same
//                   stage read MN-major as V).
//   softmax warps : eight warps of 16 whole rows each (TMEM 16-lane access
//                   shapes; a row's keys spread over a quad of threads).
//                   Each sends its partial scores, rounded to 24 bits and
//                   packed, to the same warp of the partner CTA over
//                   distributed shared memory (st.async counted on the
//                   partner's mbarrier), adds the partner's block to its own
//                   exact partial scores, then runs the online
//                   softmax with a lazily rescaled running max and writes its
//                   weights to TMEM over the consumed score columns (bf16: a
//                   high part and, on tiles where one key carries much of a
//                   row's weight, a low part).
// The epilogue normalises O and writes bf16 output (one split) or fp32
// partials plus the per-row log-sum-exp (several splits).
//
// Sources: the 576-wide latent row whose first 512 dims are the value
// ("[Perf][Kimi-K3] Cut MLA decode concat/cache epilogue latency", Purpose
// item 1); paged cache at any page size and the causal MTP mask ("HK MLA:
// MI35x m16x8 retune, new m16x4 kernel, page_size + mask support", Summary
// track 1; its MI35x retune interleaves the output rescale with the PV GEMM
// and uses 64-key blocks, which this kernel keeps); one program per (batch,
// head group, KV chunk) with chunks past a sequence's end returning at once
// ("perf(mla): chunk the non-FP4 gather_kv_b_proj over KV", description).
//
// Every wait is bounded (2 s of wall time unless the plan sets another
// limit).  A wait that runs out sets MLA_DEVFLAG_TIMEOUT in the status word
// and the CTA winds down instead of hanging the GPU: it stops issuing, drains
// its copies and MMAs, frees TMEM and meets its partner at the final cluster
// barrier (the partner's own waits run out in turn).

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla_decode.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int T = mla::kKeyTile;       // 64 keys per tile
constexpr int ATOM = T * 128;          // one 64-dim slab of a 16-bit stage: 64 keys x 128 B
constexpr int ATOM8 = T * 64;          // the same slab of raw fp8 codes: 64 keys x 64 B
constexpr int SLOTS = 5;               // slabs per stage: 4 value + 1 rope (half of it used)
constexpr int STAGE = SLOTS * ATOM;    // 40 KB of 16-bit operands (36 KB of it filled)
constexpr int RAW_STAGE = SLOTS * ATOM8;  // 20 KB of fp8 codes
constexpr int QROPE = 128 * 128;       // rope dims of Q, 128 rows x 128 B
// Exchange with the partner CTA: each softmax warp sends and receives the
// partial scores of its 16 rows x 64 keys per tile (1024 scores), each
// rounded to 24 bits (16 significant bits) and packed four to three words.
constexpr int kSoftmaxWarps = 8;
constexpr int RECV_W = 32 * 32 * 3;                  // one warp's block (3 KB)
constexpr int RECV = kSoftmaxWarps * RECV_W;         // one tile (24 KB), one buffer
constexpr int X_FREE = RECV;                         // [8] words the "buffer free" signals land in
constexpr int XCHG = X_FREE + 128;
// Warps: 0..2 loaders (warp w owns operand stage w), 3 MMA, 4..11 softmax;
// 12 warps leave 168 registers a thread.
constexpr int kSoftmaxWarp0 = 4;
constexpr int kMmaWarp = 3;
constexpr int kThreads = 32 * 12;

// Shared-memory plan.  Each operand stage has its own loader warp, so every
// stage barrier is waited on by one warp, in order.  bf16 cache: 3 operand
// stages filled with cp.async.  fp8 cache: 3 f16 operand stages, each with a
// raw stage of codes its loader warp copies into and converts from.  (A
// fourth bf16 stage needs a 13th warp, which cuts the registers to 128 a
// thread; measured, the 12-warp kernel with 3 stages is faster.)
template <bool kFp8>
struct Layout {
  static constexpr int NS = 3;              // operand stages = loader warps
  static constexpr int NR = kFp8 ? 3 : 0;   // raw fp8 stages (one per loader warp)
  static constexpr int OFF_STAGE = 0;
  static constexpr int OFF_RAW = OFF_STAGE + NS * STAGE;
  static constexpr int OFF_QROPE = OFF_RAW + NR * RAW_STAGE;
  static constexpr int OFF_RECV = OFF_QROPE + QROPE;
  static constexpr int OFF_BAR = OFF_RECV + XCHG;
  static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + barriers + alignment slack
};
static_assert(Layout<false>::SMEM_BYTES <= 232448, "bf16 smem");
static_assert(Layout<true>::SMEM_BYTES <= 232448, "fp8 smem");

// TMEM columns
constexpr uint32_t TM_O = 0;     // 256 fp32 columns: this CTA's value half
constexpr uint32_t TM_Q = 256;   // 128 columns: 256 bf16 of Q, packed in pairs
constexpr uint32_t TM_S = 384;   // two 64-column score buffers; P overwrites them (bf16:
                                 // cols 0..31 high-order, 32..63 low-order weights)
constexpr uint32_t TM_COLS = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before a rescale
constexpr float kMaxSentinel = -1.0e30f;
constexpr uint64_t kDrainNs = 500000000ull;  // bound of the wind-down waits after an abort
constexpr uint32_t kSleepNs = 20000;  // suspend-time hint of a waiting thread

struct Bars {
  uint64_t kv_full[4];    // operand stage ready (the 32 threads of its loader warp arrive)
  uint64_t kv_empty[4];   // operand stage consumed by the MMAs
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t recv_full[kSoftmaxWarps];  // the partner warp's partial scores landed (3 KB)
  uint64_t recv_free[kSoftmaxWarps];  // the partner warp has read what this warp sent
  uint64_t o_done;
  uint64_t o_final;  // the last PV has drained (one phase)
  uint64_t q_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  uint64_t heavy[2];  // bf16: per score buffer, one byte per softmax warp (see the softmax)
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct Ctx {
  int32_t* status;
  volatile int32_t* abort;
  uint64_t limit_ns;  // bound of every pipeline wait (FwdParams::wait_ns)
  uint32_t sleep_ns;  // suspend hint of a wait: no longer than the limit, so any limit is reachable
};

// Wait used only while winding down after an abort: ignores the abort word,
// gives up after 0.5 s.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kDrainNs) return false;
  }
  return true;
}

// Bounded wait on an mbarrier phase.  Returns false (and flags the status
// word and the CTA's abort word) if the phase did not complete in time or
// another warp of this CTA already gave up.
__device__ __forceinline__ bool wait(const Ctx& c, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    // Sleep on the barrier rather than spin: waiting warps would otherwise
    // take issue slots from the warps that share their sub-partition.  A
    // failed try suspends the thread for up to kSleepNs (the wait limit
    // if that is shorter), so reading the timer after each one costs
    // nothing that matters.
    if (ptx::mbar_try_wait_sleep(bar, parity, c.sleep_ns)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.limit_ns) {
      atomicOr(c.status, MLA_DEVFLAG_TIMEOUT);
      *c.abort = 1;
      return false;
    }
  }
}

// The same, decided for the whole warp: true only if every lane's wait
// succeeded, so warp-collective tcgen05 instructions stay convergent.
__device__ __forceinline__ bool wait_all(const Ctx& c, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(c, bar, parity));
}

// 2^x with the SFU's approximate exp2 (inputs below -126 flush to +0, -inf
// gives +0).  Its relative error is far below the 16-bit rounding the
// weights get next.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 codes (low byte = first) -> two f16 (exact: every e4m3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_codes));
  return r;
}

// fp32 bits + half a unit of the 24-bit value: the top three bytes are the
// value rounded to 16 significant bits (half away from zero on the magnitude).
__device__ __forceinline__ uint32_t round_up_bits(float x) { return __float_as_uint(x) + 0x80u; }

// Four values -> three words (the upper three bytes of each).
__device__ __forceinline__ void pack24(uint32_t A, uint32_t B, uint32_t C, uint32_t D, uint32_t* w) {
  w[0] = __byte_perm(A, B, 0x5321);
  w[1] = __byte_perm(B, C, 0x6532);
  w[2] = __byte_perm(C, D, 0x7653);
}

__device__ __forceinline__ void unpack24(const uint32_t* w, float* u) {
  u[0] = __uint_as_float(__byte_perm(w[0], 0u, 0x2104));
  u[1] = __uint_as_float(__byte_perm(w[0], w[1], 0x5430) & 0xFFFFFF00u);
  u[2] = __uint_as_float(__byte_perm(w[1], w[2], 0x4320) & 0xFFFFFF00u);
  u[3] = __uint_as_float(w[2] & 0xFFFFFF00u);
}

__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Eight bf16 -> eight f16 (exact for |x| in [2^-14, 65504]; flags larger values).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 x, bool& out_of_range) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16), hi = __uint_as_float(w[i] & 0xFFFF0000u);
    out_of_range |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
    w[i] = pack_f16(lo, hi);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// K-major, 128B-swizzled operand: rows 128 B apart, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t addr) {
  return ptx::smem_desc(addr, 16, 1024, 2);
}

// The same stage read MN-major as V (N = 256 value dims over 4 slabs 8 KB
// apart, K = keys in 8-row groups 1 KB apart).
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t addr) {
  return ptx::smem_desc(addr, ATOM, 1024, 2);
}

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_sm103_kernel(mla::FwdParams p) {
  using L = Layout<kFp8>;
  constexpr int NS = L::NS;
  constexpr int OFF_STAGE = L::OFF_STAGE, OFF_RAW = L::OFF_RAW, OFF_QROPE = L::OFF_QROPE;
  constexpr int OFF_RECV = L::OFF_RECV, OFF_BAR = L::OFF_BAR;
  constexpr uint32_t kAB = kFp8 ? 0u : 1u;  // operand type: f16 (fp8 cache) or bf16
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = ptx::smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  // The work unit: (sequence b, row block rb, key range [k0, k1)), its
  // context, and where its result goes (the final output when the unit
  // covers the whole sequence, else partial slot `part` for the merge).
  int rb, b, ctx, k0, k1;
  bool single;
  size_t part;
  if (p.units != nullptr) {
    // Device-planned: the unit list was written by the planning kernel this
    // one is launched behind, so wait for it first.  Both CTAs of a pair
    // read the same unit and take the same branches.
    ptx::grid_dependency_wait();
    const int u = blockIdx.x >> 1;
    if (u >= *p.n_units) return;
    const int4 d = p.units[u];
    const int4 si = p.seq_info[d.x];
    b = d.x;
    rb = d.y & 0xFF;
    k0 = d.z;
    k1 = d.w;
    ctx = si.x;  // already clamped to what the table holds
    single = si.z == 1;
    part = (size_t)si.y + (d.y >> 8);
  } else {
    rb = blockIdx.x >> 1;
    b = blockIdx.y;
    const int split = blockIdx.z;
    // A context the plan does not cover is clamped to [0, max_ctx] and
    // flagged.  max_ctx keys fit the block table (bt_stride * page_size >=
    // max_ctx is checked on the host) and the splits (num_splits *
    // chunk_len >= max_ctx), so no table entry past the sequence's row is
    // read.
    ctx = p.seq_lens[b];
    if (ctx < 0 || ctx > p.max_ctx) {
      if (threadIdx.x == 0 && rank == 0 && split == 0) atomicOr(p.status, MLA_DEVFLAG_CTX_RANGE);
      ctx = ctx < 0 ? 0 : p.max_ctx;
    }
    k0 = split * p.chunk_len;
    k1 = min(k0 + p.chunk_len, ctx);
    single = p.num_splits == 1;
    part = (size_t)b * p.num_splits + split;
  }
  const int n_tiles = k1 > k0 ? (k1 - k0 + T - 1) / T : 0;
  const int vdim0 = (int)rank * 256;  // this CTA's value dims
  const float s_kv = (p.kv_dtype == MLA_KV_FP8_E4M3 && p.kv_scale) ? *p.kv_scale : 1.f;

  if (n_tiles == 0) {
    // No key of this split: the row results are out = 0, lse = -inf.  Both
    // CTAs of the pair take this branch together, before any cluster traffic.
    ptx::grid_dependency_wait();
    for (int i = threadIdx.x; i < mla::kRowTile; i += kThreads) {
      const int row = rb * mla::kRowTile + i;
      if (row >= p.rows) break;
      if (single) {
        uint4* o = reinterpret_cast<uint4*>(p.out + ((size_t)b * p.rows + row) * mla::kDV + vdim0);
        for (int c = 0; c < 32; ++c) o[c] = make_uint4(0, 0, 0, 0);
        if (rank == 0) p.lse[(size_t)b * p.rows + row] = -INFINITY;
      } else if (rank == 0) {
        p.part_lse[part * p.rows + row] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(ptx::smem_u32(&bars.kv_full[s]), 32);
      ptx::mbar_init(ptx::smem_u32(&bars.kv_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.p_full[i]), 32 * kSoftmaxWarps);
    }
    for (int w = 0; w < kSoftmaxWarps; ++w) {
      ptx::mbar_init(ptx::smem_u32(&bars.recv_full[w]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.recv_free[w]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars.o_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars.o_final), 1);
    ptx::mbar_init(ptx::smem_u32(&bars.q_ready), 32 * kSoftmaxWarps);
    ptx::mbar_init(ptx::smem_u32(&bars.drain), 1);
    bars.abort = 0;
    ptx::fence_mbar_init_cluster();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(ptx::smem_u32(&bars.tmem_base), TM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();  // barriers of both CTAs initialised before any remote arrive
  ptx::tc_fence_after();
  // q and the newest cache rows may come from the kernel this one is
  // launched behind (the decode epilogue): nothing past this point reads
  // them, or writes an output, before that kernel has completed.  A no-op
  // when the launch is not a programmatic dependent one.
  ptx::grid_dependency_wait();
  const uint32_t tmem = bars.tmem_base;
  Ctx c{p.status, &bars.abort, p.wait_ns,
        (uint32_t)(p.wait_ns < (uint64_t)kSleepNs ? p.wait_ns : (uint64_t)kSleepNs)};

  if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t id_qk = ptx::idesc_f16(128, T, kAB, false, false);
      const uint32_t id_pv = ptx::idesc_f16(128, 256, kAB, false, true);
      bool ok = wait(c, ptx::smem_u32(&bars.q_ready), 0);
      ptx::tc_fence_after();
      // Operand descriptors from bases: the start address is the low field in
      // 16-byte units, so a stage, a slab or a 16-key step of V is an add (no
      // carry: every address is below 256 KB).
      const uint64_t dk = kmajor_desc(sbase + OFF_STAGE);  // slab 0 of stage 0
      const uint64_t dv = vmajor_desc(sbase + OFF_STAGE);  // V of stage 0
      const uint64_t dqr = kmajor_desc(sbase + OFF_QROPE);
      constexpr uint32_t kStageU = STAGE >> 4, kAtomU = ATOM >> 4;
      auto issue_qk = [&](int u, int s) {  // tile u from stage s (u % NS)
        const uint32_t d = tmem + TM_S + (u & 1) * T;
        const uint64_t k0 = dk + s * kStageU;
        for (int a = 0; a < 4; ++a)
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ts(d, tmem + TM_Q + a * 32 + kk * 8, k0 + a * kAtomU + 2 * kk, id_qk,
                        (a | kk) != 0);
        // this CTA's 32 rope dims: 16-dim steps 2 rank, 2 rank + 1 of the rope slab
        for (int kk = 2 * (int)rank; kk < 2 * (int)rank + 2; ++kk)
          ptx::mma_ss(d, dqr + 2 * kk, k0 + 4 * kAtomU + 2 * kk, id_qk, 1);
        ptx::mma_commit(ptx::smem_u32(&bars.s_full[u & 1]));
      };
      auto issue_pv = [&](int t, int s, bool second) {  // tile t from stage s (t % NS)
        const uint32_t pa = tmem + TM_S + (t & 1) * T;
        const uint64_t v0 = dv + s * kStageU;
        for (int kk = 0; kk < T / 16; ++kk)
          ptx::mma_ts(tmem + TM_O, pa + kk * 8, v0 + kk * (2048 >> 4), id_pv, (t | kk) != 0);
        if (!kFp8 && second) {  // second-order weights (see the softmax)
          for (int kk = 0; kk < T / 16; ++kk)
            ptx::mma_ts(tmem + TM_O, pa + 32 + kk * 8, v0 + kk * (2048 >> 4), id_pv, 1);
        }
        ptx::mma_commit(ptx::smem_u32(&bars.o_done));
        if (t == n_tiles - 1) ptx::mma_commit(ptx::smem_u32(&bars.o_final));
        ptx::mma_commit(ptx::smem_u32(&bars.kv_empty[s]));
      };
      // Issue whichever is ready: QK^T of tile nq (its stage has landed and
      // its score buffer is free, i.e. the PV of tile nq-2 is issued; the
      // tensor pipe runs one thread's MMAs in order) or PV of tile np (its
      // weights are written).  A late stage never holds back a ready PV.
      // The stage ring's positions and phases are counted, not divided out.
      int nq = 0, np = 0;
      int sq = 0, sp = 0;     // stages of tiles nq and np (t % NS)
      uint32_t phq = 0;       // phase parity of tile nq's stage barrier
      uint64_t t_last = ptx::globaltimer_ns();
      uint32_t idle = 0;
      while (ok && np < n_tiles) {
        bool progress = false;
        if (nq < n_tiles && nq <= np + 1 &&
            ptx::mbar_test_wait(ptx::smem_u32(&bars.kv_full[sq]), phq)) {
          ptx::tc_fence_after();
          issue_qk(nq++, sq);
          if (sq == NS - 1) {
            sq = 0;
            phq ^= 1u;
          } else {
            ++sq;
          }
          progress = true;
        }
        if (np < nq && ptx::mbar_test_wait(ptx::smem_u32(&bars.p_full[np & 1]), (np >> 1) & 1)) {
          ptx::tc_fence_after();
          const bool second = *reinterpret_cast<volatile uint64_t*>(&bars.heavy[np & 1]) != 0;
          issue_pv(np++, sp, second);
          sp = sp == NS - 1 ? 0 : sp + 1;
          progress = true;
        }
        if (progress) {
          idle = 0;
          t_last = 0;
          continue;
        }
        // Nothing ready.  Do not spin on the issue slots the softmax and
        // loader warps of this sub-partition need: when only the weights of
        // tile np can unblock the pipe, sleep on their barrier (the phase is
        // tested again above); otherwise back off briefly.
        if (nq < n_tiles && nq <= np + 1) __nanosleep(32);
        else (void)ptx::mbar_try_wait(ptx::smem_u32(&bars.p_full[np & 1]), (np >> 1) & 1);
        if ((++idle & 15) == 0) {
          const uint64_t now = ptx::globaltimer_ns();
          if (t_last == 0) t_last = now;
          if (*c.abort) ok = false;
          else if (now - t_last > c.limit_ns) {
            atomicOr(c.status, MLA_DEVFLAG_TIMEOUT);
            *c.abort = 1;
            ok = false;
          }
        }
      }
      (void)ok;
    }
    __syncwarp();
  } else if (warp < NS) {
    // ------------------------------------------------------------ loader ---
    // Gather of a tile's cache rows with 16-byte cp.async (L2 only).  The
    // operand layout keeps a key's 64-dim slab contiguous only over 128 B, so
    // every copy is a 128-byte piece of one row (of the rope slab, the CTA's
    // 64-byte half): 8 lanes per (key, slab) piece for bf16, written straight
    // into the 128B-swizzled stage; 4 lanes per 64-byte piece of fp8 codes,
    // written into the warp's raw stage and converted to f16 by the same
    // lanes.  Loader warp w
    // owns operand stage w and copies tiles w, w+NS, ...: it issues a tile,
    // waits for its own copies, fences them for the tensor cores' async proxy
    // and arrives on the stage's full barrier, while the other loader warps
    // have their tiles in flight.  Block-table entries for the warp's next
    // tile are read before it waits.
    constexpr int LPI = kFp8 ? 4 : 8;        // lanes per piece
    constexpr int IPI = 32 / LPI;            // pieces per warp instruction
    constexpr int NK = T / IPI;              // keys per lane: 16 (bf16) or 8 (fp8)
    const int lw = warp;  // the operand stage this warp owns
    const int g = lane / LPI, sub = lane % LPI;
    constexpr int n_slots = SLOTS;
    // In the rope slab a CTA copies only its 32 dims: the lanes of 16-byte
    // pieces 4 rank .. 4 rank + 3 (bf16) or of 16-code pieces 2 rank, 2 rank + 1 (fp8).
    const bool rope_lane = (kFp8 ? (sub >> 1) : (sub >> 2)) == (int)rank;
    // This sequence's page ids: a row of the padded table, or (CSR form)
    // kv_indices from kv_indptr[b] on.
    const int32_t* bt = p.bt + (p.bt_indptr ? (size_t)p.bt_indptr[b] : (size_t)b * p.bt_stride);
    const char* cache = static_cast<const char*>(p.cache);
    auto key_of = [&](int tile, int i) -> int {  // i-th key of this lane, clamped to the split
      const int start = k0 + tile * T;
      return start + min(i * IPI + g, min(T, k1 - start) - 1);
    };
    // key / page_size by a multiply and shifts: the unsigned form of
    // Granlund and Montgomery, "Division by invariant integers using
    // multiplication" (PLDI 1994), exact for every 32-bit key.  With
    // l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
    // q = (t + ((n - t) >> 1)) >> (l - 1) where t = mulhi(m, n); d = 1 is n.
    const uint32_t pdiv = (uint32_t)p.page_size;
    const uint32_t plog = 32u - __clz(pdiv - 1u);
    const uint32_t pmul = (uint32_t)(((1ull << 32) * ((1ull << plog) - pdiv)) / pdiv) + 1u;
    const uint32_t pshift = plog > 0 ? plog - 1u : 0u;
    auto page_of = [&](uint32_t key) -> uint32_t {
      const uint32_t t = __umulhi(pmul, key);
      return pdiv == 1u ? key : (t + ((key - t) >> 1)) >> pshift;
    };
    int pg[NK];
    auto load_pages = [&](int tile) {
      if (tile >= n_tiles) return;
#pragma unroll
      for (int i = 0; i < NK; ++i) pg[i] = __ldg(&bt[page_of((uint32_t)key_of(tile, i))]);
    };
    load_pages(lw);
    for (int t = lw; t < n_tiles; t += NS) {
      const int s = lw;
      const char* row[NK];
      bool bad = false;
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        int64_t page = pg[i];
        if (page < 0 || page >= p.num_pages) {
          bad = true;
          page = 0;
        }
        const uint32_t key = (uint32_t)key_of(t, i);
        const int64_t r = page * p.page_size + (int64_t)(key - page_of(key) * pdiv);
        row[i] = cache + r * (kFp8 ? mla::kDQK : mla::kDQK * 2);
      }
      if (bad) atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
      load_pages(t + NS);
      if constexpr (!kFp8) {
        if (t >= NS && !wait_all(c, ptx::smem_u32(&bars.kv_empty[s]), ((t / NS) - 1) & 1))
          break;
      }
      const uint32_t dst = sbase + (kFp8 ? OFF_RAW + lw * RAW_STAGE : OFF_STAGE + s * STAGE);
      for (int sl = 0; sl < n_slots; ++sl) {
        if (sl == 4 && !rope_lane) continue;
        const int dim = sl < 4 ? vdim0 + sl * 64 : 512;
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int kk = i * IPI + g;
          if constexpr (kFp8) {
            ptx::cp_async_16(dst + sl * ATOM8 + kk * 64 + sub * 16, row[i] + dim + sub * 16);
          } else {
            ptx::cp_async_16(dst + sl * ATOM + kk * 128 + ((sub ^ (kk & 7)) * 16),
                             row[i] + (dim + sub * 8) * 2);
          }
        }
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
      if constexpr (kFp8) {
        // e4m3 codes -> f16 operands (exact); the per-tensor scale is applied
        // to the scores and the output instead.
        if (t >= NS && !wait_all(c, ptx::smem_u32(&bars.kv_empty[s]), ((t / NS) - 1) & 1))
          break;
        const uint32_t out = sbase + OFF_STAGE + s * STAGE;
        for (int sl = 0; sl < n_slots; ++sl) {
          if (sl == 4 && !rope_lane) continue;
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            const int kk = i * IPI + g;
            const uint4 codes = ld_shared_u4(dst + sl * ATOM8 + kk * 64 + sub * 16);
            uint4 lo, hi;
            lo.x = e4m3x2_to_f16x2(codes.x);
            lo.y = e4m3x2_to_f16x2(codes.x >> 16);
            lo.z = e4m3x2_to_f16x2(codes.y);
            lo.w = e4m3x2_to_f16x2(codes.y >> 16);
            hi.x = e4m3x2_to_f16x2(codes.z);
            hi.y = e4m3x2_to_f16x2(codes.z >> 16);
            hi.z = e4m3x2_to_f16x2(codes.w);
            hi.w = e4m3x2_to_f16x2(codes.w >> 16);
            const uint32_t rowp = out + sl * ATOM + kk * 128;
            st_shared_u4(rowp + (((2 * sub) ^ (kk & 7)) * 16), lo);
            st_shared_u4(rowp + (((2 * sub + 1) ^ (kk & 7)) * 16), hi);
          }
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&bars.kv_full[s]));
    }
    ptx::cp_async_wait<0>();  // nothing of this warp is in flight when it leaves
  } else if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + kSoftmaxWarps) {
    // ----------------------------------------------------------- softmax ---
    // Softmax warp sw (0..7) owns 16 whole rows of the 128-row block: TMEM
    // lanes lbase .. lbase + 15 with lbase = 32 (warp % 4) + 16 (sw / 4) (a
    // warp reaches the lane quarter warp % 4 only).  Through the 16x256b
    // access shape thread i holds rows rA = lbase + i/4 and rB = rA + 8, and
    // of every 8-key group j the keys 8j + 2(i%4) and 8j + 2(i%4) + 1: a row's
    // 64 keys are spread over the 4 threads of a quad, whose shuffles give the
    // row max and sum.  The partner CTA's warp sw holds the same elements.
    const int sw = warp - kSoftmaxWarp0;
    const int q4 = warp & 3;                   // TMEM lane quarter of this warp
    const int g = sw >> 2;                     // which half of the quarter
    const int lbase = q4 * 32 + g * 16;
    const int cq = lane & 3;                   // column pair within each 8-key group
    const int rA = lbase + (lane >> 2), rB = rA + 8;
    const uint32_t lanes16 = (uint32_t)lbase << 16;
    auto visible = [&](int r) {  // keys [k0, visible) of this split that row r sees
      const int row = rb * mla::kRowTile + r;
      if (row >= p.rows) return 0;
      const int tok = row / p.heads;
      int nvis = p.causal ? ctx - p.sq + tok + 1 : ctx;
      nvis = max(0, min(nvis, ctx));
      return min(nvis, k1);
    };
    const int visA = visible(rA), visB = visible(rB);

    // Q (this CTA's 256 latent dims) -> TMEM as 16-bit pairs: thread i of
    // the two warps of a lane quarter writes row 32 q4 + i, two 64-dim chunks
    // each; in both CTAs the second warp also puts the 64 rope dims into shared
    // memory (128B-swizzled K-major).
    {
      const int r = q4 * 32 + lane;
      const int row = rb * mla::kRowTile + r;
      const bool valid_row = row < p.rows;
      const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
      const uint4* qv = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.rows + row) * mla::kDQK);
      uint32_t buf[32];
      bool q_range = false;
      for (int chunk = 2 * g; chunk < 2 * g + 2; ++chunk) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = valid_row ? qv[(vdim0 + chunk * 64) / 8 + v] : make_uint4(0, 0, 0, 0);
          if (kFp8) x = bf16x8_to_f16x8(x, q_range);
          buf[v * 4 + 0] = x.x;
          buf[v * 4 + 1] = x.y;
          buf[v * 4 + 2] = x.z;
          buf[v * 4 + 3] = x.w;
        }
        ptx::tmem_st32(tmem + lanes + TM_Q + chunk * 32, buf);
      }
      if (g == 1) {
        uint8_t* qr = smem + OFF_QROPE + r * 128;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x = valid_row ? qv[512 / 8 + v] : make_uint4(0, 0, 0, 0);
          if (kFp8) x = bf16x8_to_f16x8(x, q_range);
          *reinterpret_cast<uint4*>(qr + ((v ^ (r & 7)) * 16)) = x;
        }
        ptx::fence_proxy_async_smem();
      }
      if (kFp8 && q_range) atomicOr(p.status, MLA_DEVFLAG_Q_RANGE);
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.q_ready));
    }

    const float c2 = p.softmax_scale * s_kv * 1.4426950408889634f;
    float mA = kMaxSentinel, mB = kMaxSentinel;  // running maxima (log2 domain), quad-uniform
    float lA = 0.f, lB = 0.f;                     // exact row sums over this thread's keys
    const uint32_t my_recv = sbase + OFF_RECV + sw * RECV_W;
    const uint32_t peer_recv = ptx::mapa(my_recv, peer);
    const uint32_t peer_free = ptx::mapa(sbase + OFF_RECV + X_FREE + sw * 4, peer);
    const uint32_t recv_full = ptx::smem_u32(&bars.recv_full[sw]);
    const uint32_t recv_free = ptx::smem_u32(&bars.recv_free[sw]);
    // A warp whose 16 rows are all past the problem's rows (fewer than 128
    // rows) swaps nothing and computes nothing; it only keeps the barrier
    // phases moving.  Both CTAs skip the same warps.  Its TMEM lanes hold
    // garbage that no output reads (the MMAs keep rows apart).
    const bool live = rb * mla::kRowTile + lbase < p.rows;
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int buf = t & 1;
      if (!wait_all(c, ptx::smem_u32(&bars.s_full[buf]), (t >> 1) & 1)) { ok = false; break; }
      if (!live) {
        if (!kFp8 && lane == 0) reinterpret_cast<volatile uint8_t*>(&bars.heavy[buf])[sw] = 0;
        ptx::mbar_arrive(ptx::smem_u32(&bars.p_full[buf]));
        continue;
      }
      ptx::tc_fence_after();
      const uint32_t scol = tmem + lanes16 + TM_S + buf * T;
      float s[32];  // s[4j + e]: e = 0, 1 -> row A keys 8j + 2cq + e; e = 2, 3 -> row B
      {
        uint32_t raw[32];
        ptx::tmem_ld16x256b_x8(scol, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(raw[i]);
      }
      // Swap partial-score blocks with the same warp of the partner CTA.  The
      // block of tile t goes into the partner's (single) buffer once the
      // partner has read tile t - 1 from it.
      if (t >= 1) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(recv_free, 4);
        if (!wait_all(c, recv_free, (t - 1) & 1)) { ok = false; break; }
      }
      {
        const uint32_t dst = peer_recv + lane * 16;
        const uint32_t bar = ptx::mapa(recv_full, peer);
#pragma unroll
        for (int qd = 0; qd < 2; ++qd) {  // 16 scores -> 12 words -> 3 stores
          uint32_t w[12];
#pragma unroll
          for (int k = 0; k < 4; ++k)  // rounded to 24 bits: the top 3 bytes of x + 0x80
            pack24(round_up_bits(s[16 * qd + 4 * k]), round_up_bits(s[16 * qd + 4 * k + 1]),
                   round_up_bits(s[16 * qd + 4 * k + 2]), round_up_bits(s[16 * qd + 4 * k + 3]),
                   w + 3 * k);
#pragma unroll
          for (int v = 0; v < 3; ++v)
            ptx::st_async_u4(dst + (3 * qd + v) * 512, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                             w[4 * v + 3], bar);
        }
      }
      {
        if (lane == 0) ptx::mbar_arrive_expect_tx(recv_full, RECV_W);
        if (!wait_all(c, recv_full, t & 1)) { ok = false; break; }
        const uint32_t src = my_recv + lane * 16;
        uint32_t fold = 0;
#pragma unroll
        for (int qd = 0; qd < 2; ++qd) {
          uint32_t w[12];
#pragma unroll
          for (int v = 0; v < 3; ++v) {
            const uint4 x = ld_shared_u4(src + (3 * qd + v) * 512);
            w[4 * v] = x.x;
            w[4 * v + 1] = x.y;
            w[4 * v + 2] = x.z;
            w[4 * v + 3] = x.w;
            fold ^= x.x ^ x.y ^ x.z ^ x.w;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float u[4];
            unpack24(w + 3 * k, u);
#pragma unroll
            for (int e = 0; e < 4; ++e) s[16 * qd + 4 * k + e] += u[e];
          }
        }
        // The buffer is read (the vote needs every lane's loaded words): the
        // partner may send its next tile.
        const bool any = __any_sync(0xffffffffu, fold == 0x9E3779B9u);
        if (t + 1 < n_tiles && lane == 0)
          ptx::st_async_b32(peer_free, any ? 1u : 0u, ptx::mapa(recv_free, peer));
      }
      // Row maxima over the visible keys of this tile (log2 domain).  Only the
      // last tile of a split and causal rows need the mask.
      const int tile0 = k0 + t * T;
      const int limA = visA - tile0, limB = visB - tile0;  // visible keys of this tile
      const bool fullA = limA >= T, fullB = limB >= T;
      // Every key of the tile visible to every row of the warp (all tiles but
      // a split's last, outside causal masking): the mask-free path.
      const bool all_full = __all_sync(0xffffffffu, fullA && fullB);
      float mxA = -INFINITY, mxB = -INFINITY;
      if (all_full) {
        float xa[4], xb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          xa[u] = fmaxf(fmaxf(s[8 * u], s[8 * u + 1]), fmaxf(s[8 * u + 4], s[8 * u + 5]));
          xb[u] = fmaxf(fmaxf(s[8 * u + 2], s[8 * u + 3]), fmaxf(s[8 * u + 6], s[8 * u + 7]));
        }
        mxA = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
        mxB = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 8 * j + 2 * cq + e;
            if (k < limA) mxA = fmaxf(mxA, s[4 * j + e]);
            if (k < limB) mxB = fmaxf(mxB, s[4 * j + 2 + e]);
          }
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      const float mtA = limA > 0 ? mxA * c2 : -INFINITY;
      const float mtB = limB > 0 ? mxB * c2 : -INFINITY;
      const bool needA = mtA > mA + kRescaleThreshold, needB = mtB > mB + kRescaleThreshold;
      if (__any_sync(0xffffffffu, needA || needB)) {
        const float nA = needA ? fmaxf(mA, mtA) : mA, nB = needB ? fmaxf(mB, mtB) : mB;
        const float alA = exp2f(mA - nA), alB = exp2f(mB - nB);
        if (t > 0) {
          // This warp's rows of the CTA's O half; the PV of the previous tile
          // must have finished accumulating.  One parity wait on o_done is
          // enough: QK^T of this tile was issued after PV of tile t - 2 and
          // the pipe runs in order, so that PV has finished and o_done is at
          // most one phase short.  (A deeper score ring breaks this.)
          if (!wait_all(c, ptx::smem_u32(&bars.o_done), (t - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t o[32];
            const uint32_t col = tmem + lanes16 + TM_O + ch * 64;
            ptx::tmem_ld16x256b_x8(col, o);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * ((i & 2) ? alB : alA));
            ptx::tmem_st16x256b_x8(col, o);
          }
        }
        lA *= alA;
        lB *= alB;
        mA = nA;
        mB = nB;
      }
      // Weights p = 2^(s*c2 - m) (s now holds them); the row sums are exact.
      uint32_t pk[32];  // [0, 16): weights as 16-bit pairs (16x128b order); [16, 32): low-order terms
      {
        const float nmA = -mA, nmB = -mB;
        float sA = 0.f, sB = 0.f;
        if (all_full) {
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s[i] = fast_exp2(fmaf(s[i], c2, (i & 2) ? nmB : nmA));
            ps[i & 3] += s[i];
          }
          sA = ps[0] + ps[1];
          sB = ps[2] + ps[3];
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int k = 8 * j + 2 * cq;
            const float a0 = fast_exp2(fmaf(s[4 * j], c2, nmA));
            const float a1 = fast_exp2(fmaf(s[4 * j + 1], c2, nmA));
            const float b0 = fast_exp2(fmaf(s[4 * j + 2], c2, nmB));
            const float b1 = fast_exp2(fmaf(s[4 * j + 3], c2, nmB));
            s[4 * j] = k < limA ? a0 : 0.f;
            s[4 * j + 1] = k + 1 < limA ? a1 : 0.f;
            s[4 * j + 2] = k < limB ? b0 : 0.f;
            s[4 * j + 3] = k + 1 < limB ? b1 : 0.f;
            sA += s[4 * j] + s[4 * j + 1];
            sB += s[4 * j + 2] + s[4 * j + 3];
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pk[2 * j] = kFp8 ? pack_f16(s[4 * j], s[4 * j + 1]) : pack_bf16(s[4 * j], s[4 * j + 1]);
          pk[2 * j + 1] =
              kFp8 ? pack_f16(s[4 * j + 2], s[4 * j + 3]) : pack_bf16(s[4 * j + 2], s[4 * j + 3]);
        }
        lA += sA;
        lB += sB;
      }
      // P columns of this tile: key pair (2m, 2m + 1) at column m; thread i
      // holds pairs 4j + i%4, which is where the 16x128b shape writes.
      const uint32_t pcol = tmem + lanes16 + TM_S + buf * T;
      ptx::tmem_st16x128b_x8(pcol, pk);
      if constexpr (!kFp8) {
        // bf16 keeps 8 significant bits.  Where one key carries a sizeable
        // share of a row's weight (more than 1/16 of the row sum so far), the
        // rounding would show in O, so the warp's rows also get a second bf16
        // term with what the first rounded away (P = P_hi + P_lo to ~16 bits)
        // and the MMA warp adds a second PV for the tile.  Below that share a
        // key's rounding moves O by at most 2^-9 / 16 of its value (5e-3 for
        // a value of 40), and the rounding errors of many small weights
        // average out.  Each warp votes
        // with one byte; a warp that votes no writes zeros as its second
        // term, so the second PV is right whichever warps voted.
        const float pmA = limA > 0 ? fast_exp2(mtA - mA) : 0.f;
        const float pmB = limB > 0 ? fast_exp2(mtB - mB) : 0.f;
        float rsA = lA + __shfl_xor_sync(0xffffffffu, lA, 1);  // row sums over the quad
        float rsB = lB + __shfl_xor_sync(0xffffffffu, lB, 1);
        rsA += __shfl_xor_sync(0xffffffffu, rsA, 2);
        rsB += __shfl_xor_sync(0xffffffffu, rsB, 2);
        const bool heavy = __any_sync(0xffffffffu, pmA * 16.f > rsA || pmB * 16.f > rsB);
        if (heavy) {  // warp-uniform
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = __uint_as_float(pk[j] << 16), h1 = __uint_as_float(pk[j] & 0xFFFF0000u);
            const int e = (j & 1) ? 2 : 0;
            pk[16 + j] = pack_bf16(s[4 * (j >> 1) + e] - h0, s[4 * (j >> 1) + e + 1] - h1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[16 + j] = 0u;
        }
        ptx::tmem_st16x128b_x8(pcol + 32, pk + 16);
        if (lane == 0) reinterpret_cast<volatile uint8_t*>(&bars.heavy[buf])[sw] = heavy ? 1 : 0;
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.p_full[buf]));
    }

    // ---------------------------------------------------------- epilogue ---
    // Row sums over the quad, in the same order in both CTAs.
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    if (ok && live && wait_all(c, ptx::smem_u32(&bars.o_final), 0)) {
      // O is final once the last PV has drained (a barrier of its own: a
      // parity wait on o_done only tells the current phase from the one
      // before it, and o_done may be one phase short or already complete).
      ptx::tc_fence_after();
      const float invA = lA > 0.f ? s_kv / lA : 0.f, invB = lB > 0.f ? s_kv / lB : 0.f;
      const int rowA = rb * mla::kRowTile + rA, rowB = rb * mla::kRowTile + rB;
      const bool okA = rowA < p.rows, okB = rowB < p.rows;
      const size_t pA = part * p.rows + rowA;
      const size_t pB = part * p.rows + rowB;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t o[32];
        ptx::tmem_ld16x256b_x8(tmem + lanes16 + TM_O + ch * 64, o);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int dim = vdim0 + ch * 64 + 8 * j + 2 * cq;
          const float a0 = __uint_as_float(o[4 * j]) * invA, a1 = __uint_as_float(o[4 * j + 1]) * invA;
          const float b0 = __uint_as_float(o[4 * j + 2]) * invB, b1 = __uint_as_float(o[4 * j + 3]) * invB;
          if (single) {
            if (okA) *reinterpret_cast<uint32_t*>(p.out + ((size_t)b * p.rows + rowA) * mla::kDV + dim) = pack_bf16(a0, a1);
            if (okB) *reinterpret_cast<uint32_t*>(p.out + ((size_t)b * p.rows + rowB) * mla::kDV + dim) = pack_bf16(b0, b1);
          } else {
            if (okA) *reinterpret_cast<float2*>(p.part_o + pA * mla::kDV + dim) = make_float2(a0, a1);
            if (okB) *reinterpret_cast<float2*>(p.part_o + pB * mla::kDV + dim) = make_float2(b0, b1);
          }
        }
      }
      if (rank == 0 && cq == 0) {
        const float lseA = lA > 0.f ? (mA + log2f(lA)) * 0.6931471805599453f : -INFINITY;
        const float lseB = lB > 0.f ? (mB + log2f(lB)) * 0.6931471805599453f : -INFINITY;
        if (single) {
          if (okA) p.lse[(size_t)b * p.rows + rowA] = lseA;
          if (okB) p.lse[(size_t)b * p.rows + rowB] = lseB;
        } else {
          if (okA) p.part_lse[pA] = lseA;
          if (okB) p.part_lse[pB] = lseB;
        }
      }
    }
    ptx::tc_fence_before();
  }

  // ------------------------------------------------------------ teardown ---
  __syncthreads();
  if (warp == kMmaWarp) {
    if (bars.abort) {
      // wait for every tcgen05 op this CTA issued before giving TMEM back
      if (lane == 0) {
        ptx::mma_commit(ptx::smem_u32(&bars.drain));
        wait_drain(ptx::smem_u32(&bars.drain), 0);
      }
      __syncwarp();
    }
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TM_COLS);
  }
  ptx::cluster_sync_all();  // no CTA leaves while its partner may still write into it
}

}  // namespace

int mla_launch_fwd_sm103(const mla::FwdParams& p, void* stream) {
  const bool fp8 = p.kv_dtype == MLA_KV_FP8_E4M3;
  auto kernel = fp8 ? fwd_sm103_kernel<true> : fwd_sm103_kernel<false>;
  const int smem = fp8 ? Layout<true>::SMEM_BYTES : Layout<false>::SMEM_BYTES;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = mla::opt_in_smem(reinterpret_cast<const void*>(kernel), smem, dev, fp8 ? 1 : 0);
  if (e != cudaSuccess) return (int)e;
  // Splits vary slowest, so every sequence's first chunk is dispatched
  // before any second chunk (the planner simulates this order).  Launched as
  // a programmatic dependent: behind the decode epilogue the prologue
  // (barrier set-up, TMEM allocation) overlaps that kernel's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.units != nullptr ? dim3(2 * p.unit_capacity, 1, 1)
                                  : dim3(p.row_blocks * 2, p.batch, p.num_splits);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, kernel, p);
}
