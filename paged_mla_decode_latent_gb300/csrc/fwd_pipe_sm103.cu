// fwd_pipe_sm103.cu -- the decode kernel for 65 to 128 score rows per block
// with a bf16 cache: the 128-row pair design of fwd_sm103.cu with a deeper
// pipeline (four operand stages, three score buffers).
//
// Work unit and split of the work between the two CTAs of a cluster are those
// of fwd_sm103.cu: CTA r owns value dims [256r, 256r + 256) and contracts the
// same 256 latent dims plus rope dims [32r, 32r + 32); the two swap 24-bit
// partial scores over distributed shared memory.  The arithmetic, and so
// every output bit, is that of fwd_sm103.cu; what differs is where the
// operands live:
//   TMEM  : O half (256 columns) | Q latent dims [0, 128) of the CTA's 256
//           (64 columns) | three 64-column score buffers (P overwrites its
//           own: high-order weights in columns 0..31, low-order in 32..63).
//   smem  : four 36 KB operand stages (four 64-dim latent slabs, 128B
//           swizzle, and the CTA's 32 rope dims in a 64B-swizzled slab), Q
//           latent dims [128, 256) (two 16 KB slabs) and Q's rope half (8 KB,
//           64B swizzle), a 24 KB receive buffer.
// A stage is held from the start of its copy until the PV of its tile has
// finished, and QK^T of tile t waits for a free score buffer (the PV of tile
// t - 3 issued).  With three stages and two buffers both rings were closed
// loops about as long as two or three tiles of softmax work; one more of
// each lets the copies and QK^T run a tile further ahead of the softmax.
//
// Per 64-key tile, in each CTA:
//   loader warps 0-2 : tiles dealt round robin (warp w takes tiles w, w + 3,
//                      ...; tile t goes to stage t % 4), 16-byte cp.async of
//                      the CTA's latent half and rope half of each key;
//   MMA warp 3       : S = Q K^T (8 MMAs with A from TMEM, 8 + 2 with A from
//                      shared memory; N = 64) into score buffer t % 3 once
//                      the PV of tile t - 3 is issued; O += P V (4 MMAs, N =
//                      256, plus 4 with the low-order weights on heavy tiles);
//   softmax warps 4-11 : send this CTA's partial scores, receive the
//                      partner's, add, online softmax with a lazily rescaled
//                      running max, weights to TMEM.
//
// The rescale of O at tile t must follow the PV of tile t - 1: PV completions
// are counted on a ring of three barriers (tile t on o_done[t % 3]); QK^T of
// tile t was issued after PV of tile t - 3, so when the softmax reaches tile t
// the barrier of tile t - 1 is at most one phase short and one parity wait
// decides.  The same holds for the stage barriers a loader waits on (see the
// loader).
//
// Every wait is bounded (2 s unless the plan sets another limit); a wait that
// runs out sets MLA_DEVFLAG_TIMEOUT and the CTA winds down as in
// fwd_sm103.cu.
//
// Sources: as fwd_sm103.cu ("HK MLA: MI35x m16x8 retune, new m16x4 kernel,
// page_size + mask support", Summary track 1 and 2; "[Perf][Kimi-K3] Cut MLA
// decode concat/cache epilogue latency", Purpose item 1; "perf(mla): chunk
// the non-FP4 gather_kv_b_proj over KV", description).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla_decode.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int T = mla::kKeyTile;       // 64 keys per tile
constexpr int NB = 3;                  // score buffers (2 or 3)
constexpr int QT = NB == 3 ? 2 : 4;    // 64-dim latent slabs of Q in TMEM (the rest in shared memory)
constexpr int NS = 4;                  // operand stages (a power of two)
constexpr int kLoaders = 3;            // loader warps (tiles dealt round robin)
constexpr int ATOM = T * 128;          // one 64-dim latent slab of a stage: 8 KB
constexpr int RATOM = T * 64;          // the CTA's 32 rope dims of a stage, 64-byte rows: 4 KB
constexpr int STAGE = 4 * ATOM + RATOM;  // 36 KB
constexpr int QSLAB = 128 * 128;       // one 64-dim slab of Q in shared memory (128 rows)
constexpr int QROPE = 128 * 64;        // Q's rope half, 64-byte rows
constexpr int kSoftmaxWarps = 8;
constexpr int RECV_W = 32 * 32 * 3;    // one warp's partial scores of a tile (3 KB)
constexpr int RECV = kSoftmaxWarps * RECV_W;  // one receive buffer (24 KB)
constexpr int OFF_STAGE = 0;
constexpr int OFF_QS = OFF_STAGE + NS * STAGE;    // Q latent dims [128, 256): 2 slabs
constexpr int OFF_QROPE = OFF_QS + (4 - QT) * QSLAB;
constexpr int OFF_RECV = OFF_QROPE + QROPE;       // the receive buffer
constexpr int OFF_XFREE = OFF_RECV + RECV;         // [8 warps] "read" words
constexpr int OFF_BAR = OFF_XFREE + 128;
constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + barriers + alignment slack
static_assert(SMEM_BYTES <= 232448, "smem");
static_assert(OFF_QS % 1024 == 0 && OFF_QROPE % 512 == 0 && STAGE % 1024 == 0, "swizzle atoms");

// Warps: 0..2 loaders (warp w owns stage w), 3 MMA, 4..11 softmax.
constexpr int kSoftmaxWarp0 = 4;
constexpr int kMmaWarp = 3;
constexpr int kThreads = 32 * 12;

// TMEM columns
constexpr uint32_t TM_O = 0;     // 256 fp32 columns: this CTA's value half
constexpr uint32_t TM_Q = 256;   // 32 QT columns: Q latent dims [0, 64 QT) of the CTA's, 16-bit pairs
constexpr uint32_t TM_S = TM_Q + 32 * QT;  // NB 64-column score buffers
static_assert(TM_S + NB * T <= 512, "TMEM columns");
static_assert((NS & (NS - 1)) == 0, "stage ring indexed by masking");
constexpr uint32_t TM_COLS = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before a rescale
constexpr float kMaxSentinel = -1.0e30f;
constexpr uint64_t kDrainNs = 500000000ull;
constexpr uint32_t kSleepNs = 20000;

struct Bars {
  uint64_t kv_full[NS];    // operand stage ready (the 32 threads of one loader warp arrive)
  uint64_t kv_empty[NS];   // operand stage consumed by the MMAs
  uint64_t s_full[NB];     // scores of the buffer's tile written
  uint64_t p_full[NB];     // weights of the buffer's tile written (every softmax thread)
  uint64_t recv_full[kSoftmaxWarps];  // the partner warp's block landed
  uint64_t recv_free[kSoftmaxWarps];  // the partner warp has read what this warp sent
  uint64_t o_done[NB];     // PV of the tile (t % 3) has finished
  uint64_t o_final;        // the last PV has finished (one phase)
  uint64_t q_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  uint64_t heavy[NB];      // per score buffer, one byte per softmax warp
};
static_assert(sizeof(Bars) <= 512, "barrier block");

struct Ctx {
  int32_t* status;
  volatile int32_t* abort;
  uint64_t limit_ns;
  uint32_t sleep_ns;  // suspend hint of a wait: no longer than the limit, so any limit is reachable
};

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity))
    if (ptx::globaltimer_ns() - t0 > kDrainNs) return false;
  return true;
}

__device__ __forceinline__ bool wait(const Ctx& c, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait_sleep(bar, parity, c.sleep_ns)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer_ns() - t0 > c.limit_ns) {
      atomicOr(c.status, MLA_DEVFLAG_TIMEOUT);
      *c.abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_all(const Ctx& c, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait(c, bar, parity));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

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

// K-major, 128B-swizzled operand: rows 128 B apart, 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t kdesc128(uint32_t addr) { return ptx::smem_desc(addr, 16, 1024, 2); }
// K-major, 64B-swizzled operand (the rope halves): rows 64 B apart, 8-row groups 512 B apart.
__device__ __forceinline__ uint64_t kdesc64(uint32_t addr) { return ptx::smem_desc(addr, 16, 512, 4); }
// The stage read MN-major as V: N = 256 value dims over 4 slabs ATOM apart,
// K = keys in 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t vdesc(uint32_t addr) { return ptx::smem_desc(addr, ATOM, 1024, 2); }

// Byte offset of 16-byte chunk c of row r in a 128B-swizzled slab (c < 8) and
// in a 64B-swizzled one (c < 4).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) * 16); }
__device__ __forceinline__ uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) * 16); }

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    fwd_pipe_kernel(mla::FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + OFF_BAR);
  const uint32_t sbase = ptx::smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  // The work unit (as in fwd_sm103.cu): sequence b, row block rb, keys
  // [k0, k1), and where the result goes.
  int rb, b, ctx, k0, k1;
  bool single;
  size_t part;
  if (p.units != nullptr) {
    ptx::grid_dependency_wait();
    const int u = blockIdx.x >> 1;
    if (u >= *p.n_units) return;
    const int4 d = p.units[u];
    const int4 si = p.seq_info[d.x];
    b = d.x;
    rb = d.y & 0xFF;
    k0 = d.z;
    k1 = d.w;
    ctx = si.x;
    single = si.z == 1;
    part = (size_t)si.y + (d.y >> 8);
  } else {
    rb = blockIdx.x >> 1;
    b = blockIdx.y;
    const int split = blockIdx.z;
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
  const int vdim0 = (int)rank * 256;

  if (n_tiles == 0) {
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
    for (int i = 0; i < NS; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.kv_full[i]), 32);
      ptx::mbar_init(ptx::smem_u32(&bars.kv_empty[i]), 1);
    }
    for (int i = 0; i < NB; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.p_full[i]), 32 * kSoftmaxWarps);
      ptx::mbar_init(ptx::smem_u32(&bars.o_done[i]), 1);
    }
    for (int w = 0; w < kSoftmaxWarps; ++w) {
      ptx::mbar_init(ptx::smem_u32(&bars.recv_full[w]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.recv_free[w]), 1);
    }
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
  ptx::grid_dependency_wait();
  const uint32_t tmem = bars.tmem_base;
  Ctx c{p.status, &bars.abort, p.wait_ns,
        (uint32_t)(p.wait_ns < (uint64_t)kSleepNs ? p.wait_ns : (uint64_t)kSleepNs)};

  if (warp == kMmaWarp) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t id_qk = ptx::idesc_f16(128, T, 1u, false, false);
      const uint32_t id_pv = ptx::idesc_f16(128, 256, 1u, false, true);
      bool ok = wait(c, ptx::smem_u32(&bars.q_ready), 0);
      ptx::tc_fence_after();
      // Operand descriptors from bases: the start address is the low field in
      // 16-byte units, so a stage (STAGE bytes), a slab (ATOM) or a 16-key
      // step of V (2048) is an add (no carry: every address is below 256 KB).
      const uint64_t dk = kdesc128(sbase + OFF_STAGE);          // latent slab 0 of stage 0
      const uint64_t dr = kdesc64(sbase + OFF_STAGE + 4 * ATOM);  // rope slab of stage 0
      const uint64_t dv = vdesc(sbase + OFF_STAGE);             // V of stage 0
      const uint64_t dq = kdesc128(sbase + OFF_QS);             // Q's shared-memory slabs
      const uint64_t dqr = kdesc64(sbase + OFF_QROPE);          // Q's rope half
      constexpr uint32_t kStageU = STAGE >> 4, kAtomU = ATOM >> 4, kQSlabU = QSLAB >> 4;
      auto issue_qk = [&](int sb, int sg) {  // into score buffer sb from stage sg
        const uint32_t d = tmem + TM_S + sb * T;
        const uint64_t k0 = dk + sg * kStageU, r0 = dr + sg * kStageU;
        for (int a = 0; a < QT; ++a)  // latent dims [0, 64 QT): A from TMEM
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ts(d, tmem + TM_Q + a * 32 + kk * 8, k0 + a * kAtomU + 2 * kk, id_qk, (a | kk) != 0);
        for (int a = QT; a < 4; ++a)  // latent dims [64 QT, 256): A from shared memory
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ss(d, dq + (a - QT) * kQSlabU + 2 * kk, k0 + a * kAtomU + 2 * kk, id_qk, 1);
        for (int kk = 0; kk < 2; ++kk)  // this CTA's 32 rope dims
          ptx::mma_ss(d, dqr + 2 * kk, r0 + 2 * kk, id_qk, 1);
        ptx::mma_commit(ptx::smem_u32(&bars.s_full[sb]));
      };
      auto issue_pv = [&](int t, int sb, int sg, bool second) {
        const uint32_t pa = tmem + TM_S + sb * T;
        const uint64_t v0 = dv + sg * kStageU;
        for (int kk = 0; kk < T / 16; ++kk)
          ptx::mma_ts(tmem + TM_O, pa + kk * 8, v0 + kk * (2048 >> 4), id_pv, (t | kk) != 0);
        if (second)
          for (int kk = 0; kk < T / 16; ++kk)
            ptx::mma_ts(tmem + TM_O, pa + 32 + kk * 8, v0 + kk * (2048 >> 4), id_pv, 1);
        ptx::mma_commit(ptx::smem_u32(&bars.o_done[sb]));
        if (t == n_tiles - 1) ptx::mma_commit(ptx::smem_u32(&bars.o_final));
        ptx::mma_commit(ptx::smem_u32(&bars.kv_empty[sg]));
      };
      // Ready-first issue: QK^T of tile nq once its stage has landed and its
      // score buffer is free (the PV of tile nq - 3 is issued; one thread's
      // MMAs run in order), PV of tile np once its weights are written.  The
      // ring positions and phases are counted, not divided out.
      int nq = 0, np = 0;
      int bq = 0, bp = 0;            // score buffers of tiles nq and np (t % NB)
      uint32_t pp = 0;               // phase parity of tile np's weights barrier
      uint64_t t_last = ptx::globaltimer_ns();
      uint32_t idle = 0;
      while (ok && np < n_tiles) {
        bool progress = false;
        if (nq < n_tiles && nq <= np + NB - 1 &&
            ptx::mbar_test_wait(ptx::smem_u32(&bars.kv_full[nq & (NS - 1)]), (nq / NS) & 1)) {
          ptx::tc_fence_after();
          issue_qk(bq, nq & (NS - 1));
          ++nq;
          bq = bq == NB - 1 ? 0 : bq + 1;
          progress = true;
        }
        if (np < nq && ptx::mbar_test_wait(ptx::smem_u32(&bars.p_full[bp]), pp)) {
          ptx::tc_fence_after();
          const bool second = *reinterpret_cast<volatile uint64_t*>(&bars.heavy[bp]) != 0;
          issue_pv(np, bp, np & (NS - 1), second);
          ++np;
          if (bp == NB - 1) {
            bp = 0;
            pp ^= 1u;
          } else {
            ++bp;
          }
          progress = true;
        }
        if (progress) {
          idle = 0;
          t_last = 0;
          continue;
        }
        if (nq < n_tiles && nq <= np + NB - 1) __nanosleep(32);
        else (void)ptx::mbar_try_wait(ptx::smem_u32(&bars.p_full[bp]), pp);
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
  } else if (warp < kLoaders) {
    // ------------------------------------------------------------ loader ---
    // Loader warp w owns stage w and copies tiles w, w + 3, ...: block-table
    // lookup, 16-byte cp.async of 128-byte row pieces (8 lanes a piece; of
    // the rope, the CTA's 64-byte half, 4 lanes) into the swizzled stage,
    // then a fence for the tensor cores and an arrival on the stage's
    // barrier.  The next tile's block-table entries are read before the warp
    // waits for its stage.
    constexpr int LPI = 8;            // lanes per 128-byte piece
    constexpr int IPI = 32 / LPI;     // keys per warp instruction
    constexpr int NK = T / IPI;       // keys per lane: 16
    const int lw = warp;
    const int g = lane / LPI, sub = lane % LPI;
    const int32_t* bt = p.bt + (p.bt_indptr ? (size_t)p.bt_indptr[b] : (size_t)b * p.bt_stride);
    const char* cache = static_cast<const char*>(p.cache);
    auto key_of = [&](int tile, int i) -> int {  // i-th key of this lane, clamped to the split
      const int start = k0 + tile * T;
      return start + min(i * IPI + g, min(T, k1 - start) - 1);
    };
    // key / page_size by a multiply and shifts (Granlund and Montgomery,
    // "Division by invariant integers using multiplication", PLDI 1994).
    const uint32_t pdiv = (uint32_t)p.page_size;
    const uint32_t plog = 32u - __clz(pdiv - 1u);
    const uint32_t pmul = (uint32_t)(((1ull << 32) * ((1ull << plog) - pdiv)) / pdiv) + 1u;
    const uint32_t pshift = plog > 0 ? plog - 1u : 0u;
    auto page_of = [&](uint32_t key) -> uint32_t {
      const uint32_t q = __umulhi(pmul, key);
      return pdiv == 1u ? key : (q + ((key - q) >> 1)) >> pshift;
    };
    int pg[NK];
    auto load_pages = [&](int tile) {
      if (tile >= n_tiles) return;
#pragma unroll
      for (int i = 0; i < NK; ++i) pg[i] = __ldg(&bt[page_of((uint32_t)key_of(tile, i))]);
    };
    load_pages(lw);
    for (int t = lw; t < n_tiles; t += kLoaders) {
      const int s = t % NS;
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
        row[i] = cache + r * (mla::kDQK * 2);
      }
      if (bad) atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
      load_pages(t + kLoaders);
      // The stage's previous tile is t - NS.  This warp's own previous wait
      // (tile t - kLoaders) saw the PV of tile t - kLoaders - NS finish, so the
      // barrier is at most one phase short and one parity wait decides.
      if (t >= NS && !wait_all(c, ptx::smem_u32(&bars.kv_empty[s]), ((t / NS) - 1) & 1)) break;
      const uint32_t dst = sbase + OFF_STAGE + s * STAGE;
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        const int kk = i * IPI + g;
#pragma unroll
        for (int sl = 0; sl < 4; ++sl)
          ptx::cp_async_16(dst + sl * ATOM + sw128(kk, sub), row[i] + (vdim0 + sl * 64 + sub * 8) * 2);
        if (sub < 4)  // the CTA's rope half: dims 512 + 32 rank + 8 sub
          ptx::cp_async_16(dst + 4 * ATOM + sw64(kk, sub), row[i] + (512 + 32 * (int)rank + sub * 8) * 2);
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<0>();
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&bars.kv_full[s]));
    }
    ptx::cp_async_wait<0>();  // nothing of this warp is in flight when it leaves
  } else if (warp >= kSoftmaxWarp0) {
    // ----------------------------------------------------------- softmax ---
    // Softmax warp sw (0..7) owns 16 whole rows: TMEM lanes lbase .. lbase +
    // 15 with lbase = 32 (warp % 4) + 16 (sw / 4).  Through the 16x256b access
    // thread i holds rows rA = lbase + i/4 and rB = rA + 8 and, of every 8-key
    // group j, keys 8j + 2(i%4) and + 1; a row's 64 keys lie in a quad of
    // threads.  The partner CTA's warp sw holds the same elements.
    const int sw = warp - kSoftmaxWarp0;
    const int q4 = warp & 3;
    const int g = sw >> 2;
    const int lbase = q4 * 32 + g * 16;
    const int cq = lane & 3;
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

    // Q: thread i of the two warps of lane quarter q4 stages row 32 q4 + i.
    // Warp g takes the 64-dim latent slabs a = g and g + 2 of the CTA's 256
    // dims: slab a < QT into TMEM, the others into shared memory slab a - QT
    // (128B swizzle); warp 1 also the CTA's 32 rope dims (64B swizzle).
    {
      const int r = q4 * 32 + lane;
      const int row = rb * mla::kRowTile + r;
      const bool valid_row = row < p.rows;
      const uint32_t lanes = (uint32_t)(q4 * 32) << 16;
      const uint4* qv = reinterpret_cast<const uint4*>(p.q + ((size_t)b * p.rows + row) * mla::kDQK);
#pragma unroll
      for (int a = g; a < 4; a += 2) {
        if (a < QT) {
          uint32_t buf[32];
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = valid_row ? qv[(vdim0 + a * 64) / 8 + v] : make_uint4(0, 0, 0, 0);
            buf[v * 4 + 0] = x.x;
            buf[v * 4 + 1] = x.y;
            buf[v * 4 + 2] = x.z;
            buf[v * 4 + 3] = x.w;
          }
          ptx::tmem_st32(tmem + lanes + TM_Q + a * 32, buf);
        } else {
          const uint32_t qs = sbase + OFF_QS + (a - QT) * QSLAB;
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const uint4 x = valid_row ? qv[(vdim0 + a * 64) / 8 + v] : make_uint4(0, 0, 0, 0);
            st_shared_u4(qs + sw128(r, v), x);
          }
        }
      }
      if (g == 1) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 x = valid_row ? qv[(512 + 32 * (int)rank) / 8 + v] : make_uint4(0, 0, 0, 0);
          st_shared_u4(sbase + OFF_QROPE + sw64(r, v), x);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.q_ready));
    }

    const float c2 = p.softmax_scale * 1.4426950408889634f;
    float mA = kMaxSentinel, mB = kMaxSentinel;  // running maxima (log2 domain), quad-uniform
    float lA = 0.f, lB = 0.f;                     // exact row sums over this thread's keys
    const uint32_t my_recv = sbase + OFF_RECV + sw * RECV_W;
    const uint32_t recv_full = ptx::smem_u32(&bars.recv_full[sw]);
    const uint32_t recv_free = ptx::smem_u32(&bars.recv_free[sw]);
    // A warp whose 16 rows are all past the problem's rows swaps and computes
    // nothing; it keeps the barrier phases moving.  Both CTAs skip the same warps.
    const bool live = rb * mla::kRowTile + lbase < p.rows;

    // Tile t's partial scores -> the partner warp's receive buffer, rounded
    // to 24 bits and packed four to three words, once the partner has read
    // tile t - 1 from it.
    // (bt3, ph3: tile t's score buffer, t % 3, and that barrier's phase parity.)
    auto send = [&](int t, int bt3, uint32_t ph3) -> bool {
      if (!wait_all(c, ptx::smem_u32(&bars.s_full[bt3]), ph3)) return false;
      ptx::tc_fence_after();
      if (t >= 1) {
        if (lane == 0) ptx::mbar_arrive_expect_tx(recv_free, 4);
        if (!wait_all(c, recv_free, (t - 1) & 1)) return false;
      }
      uint32_t raw[32];
      ptx::tmem_ld16x256b_x8(tmem + lanes16 + TM_S + bt3 * T, raw);
      ptx::tmem_ld_wait();
      const uint32_t dst = ptx::mapa(my_recv, peer) + lane * 16;
      const uint32_t bar = ptx::mapa(recv_full, peer);
#pragma unroll
      for (int qd = 0; qd < 2; ++qd) {  // 16 scores -> 12 words -> 3 stores
        uint32_t w[12];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          pack24(raw[16 * qd + 4 * k] + 0x80u, raw[16 * qd + 4 * k + 1] + 0x80u,
                 raw[16 * qd + 4 * k + 2] + 0x80u, raw[16 * qd + 4 * k + 3] + 0x80u, w + 3 * k);
#pragma unroll
        for (int v = 0; v < 3; ++v)
          ptx::st_async_u4(dst + (3 * qd + v) * 512, w[4 * v], w[4 * v + 1], w[4 * v + 2],
                           w[4 * v + 3], bar);
      }
      return true;
    };

    bool ok = true;
    int bt3 = 0;       // t % NB, counted
    uint32_t ph3 = 0;  // (t / NB) & 1
    for (int t = 0; ok && t < n_tiles; ++t, ph3 ^= (bt3 == NB - 1), bt3 = bt3 == NB - 1 ? 0 : bt3 + 1) {
      if (!live) {
        if (!wait_all(c, ptx::smem_u32(&bars.s_full[bt3]), ph3)) { ok = false; break; }
        if (lane == 0) reinterpret_cast<volatile uint8_t*>(&bars.heavy[bt3])[sw] = 0;
        ptx::mbar_arrive(ptx::smem_u32(&bars.p_full[bt3]));
        continue;
      }
      if (!send(t, bt3, ph3)) { ok = false; break; }
      // Tile t: the partner's block and this CTA's own exact partial scores
      // (still in score buffer t % 3).
      if (lane == 0) ptx::mbar_arrive_expect_tx(recv_full, RECV_W);
      if (!wait_all(c, recv_full, t & 1)) { ok = false; break; }
      ptx::tc_fence_after();
      float s[32];  // s[4j + e]: e = 0, 1 -> row A keys 8j + 2cq + e; e = 2, 3 -> row B
      {
        uint32_t raw[32];
        ptx::tmem_ld16x256b_x8(tmem + lanes16 + TM_S + bt3 * T, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(raw[i]);
      }
      {
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
        // partner may send tile t + 1 into it.
        const bool any = __any_sync(0xffffffffu, fold == 0x9E3779B9u);
        if (t + 1 < n_tiles && lane == 0)
          ptx::st_async_b32(ptx::mapa(sbase + OFF_XFREE + sw * 4, peer), any ? 1u : 0u,
                            ptx::mapa(recv_free, peer));
      }
      // Row maxima over the visible keys of this tile (log2 domain); only the
      // last tile of a split and causal rows need the mask.
      const int tile0 = k0 + t * T;
      const int limA = visA - tile0, limB = visB - tile0;
      const bool all_full = __all_sync(0xffffffffu, limA >= T && limB >= T);
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
          // The PV of tile t - 1 must have finished accumulating: its barrier
          // in the ring is at most one phase short (see the file comment).
          const int bprev = bt3 == 0 ? NB - 1 : bt3 - 1;  // tile t - 1's ring slot and phase
          const uint32_t pprev = bt3 == 0 ? ph3 ^ 1u : ph3;
          if (!wait_all(c, ptx::smem_u32(&bars.o_done[bprev]), pprev)) { ok = false; break; }
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
      uint32_t pk[32];  // [0, 16): weights as bf16 pairs (16x128b order); [16, 32): low-order terms
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
          pk[2 * j] = pack_bf16(s[4 * j], s[4 * j + 1]);
          pk[2 * j + 1] = pack_bf16(s[4 * j + 2], s[4 * j + 3]);
        }
        lA += sA;
        lB += sB;
      }
      // P over the consumed scores: key pair (2m, 2m + 1) at column m.
      const uint32_t pcol = tmem + lanes16 + TM_S + bt3 * T;
      ptx::tmem_st16x128b_x8(pcol, pk);
      {
        // The low-order terms and the second PV where one key carries more
        // than 1/16 of a row's sum so far (as in fwd_sm103.cu).
        const float pmA = limA > 0 ? fast_exp2(mtA - mA) : 0.f;
        const float pmB = limB > 0 ? fast_exp2(mtB - mB) : 0.f;
        float rsA = lA + __shfl_xor_sync(0xffffffffu, lA, 1);
        float rsB = lB + __shfl_xor_sync(0xffffffffu, lB, 1);
        rsA += __shfl_xor_sync(0xffffffffu, rsA, 2);
        rsB += __shfl_xor_sync(0xffffffffu, rsB, 2);
        const bool heavy = __any_sync(0xffffffffu, pmA * 16.f > rsA || pmB * 16.f > rsB);
        if (heavy) {
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
        if (lane == 0) reinterpret_cast<volatile uint8_t*>(&bars.heavy[bt3])[sw] = heavy ? 1 : 0;
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.p_full[bt3]));
    }

    // ---------------------------------------------------------- epilogue ---
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    if (ok && live && wait_all(c, ptx::smem_u32(&bars.o_final), 0)) {
      ptx::tc_fence_after();
      const float invA = lA > 0.f ? 1.f / lA : 0.f, invB = lB > 0.f ? 1.f / lB : 0.f;
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

int mla_launch_fwd_pipe_sm103(const mla::FwdParams& p, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = mla::opt_in_smem(reinterpret_cast<const void*>(fwd_pipe_kernel), SMEM_BYTES, dev, 6);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.units != nullptr ? dim3(2 * p.unit_capacity, 1, 1)
                                  : dim3(p.row_blocks * 2, p.batch, p.num_splits);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, fwd_pipe_kernel, p);
}
