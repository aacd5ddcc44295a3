// fwd_small_sm103.cu -- the decode kernel for problems with few score rows
// per sequence (H * Sq <= 64 with a bf16 cache, <= 16 with fp8): the
// product-64 shapes (64,1), (32,2), (16,4) and the TP-local 16-head fp8
// decode.
//
// Source: "HK MLA: MI35x m16x8 retune, new m16x4 kernel, page_size + mask
// support" (aiter PR 3072), Summary, track 2: a separate kernel for the
// shapes whose num_heads x max_seqlen_qo is 64, with a different tiling and
// occupancy from the 128-row one.
//
// Why a second kernel on GB300.  Every tcgen05 MMA of M = 128 costs about 64
// cycles whatever its N up to 128, so with few rows the work per key is set
// by how many keys one MMA covers, not by the rows.  The 128-row kernel
// scores 64 keys per MMA (its TMEM holds Q, so only two 64-column score
// buffers fit next to the output half); here the tile is 128 keys, which
// halves the MMA issue per key.  TMEM then holds the output half (256
// columns) and two 128-column score buffers, so Q moves to shared memory:
// with at most 64 real rows its slabs are small (the MMA reads 128 rows of
// A; rows past the problem's land in the memory that follows and are never
// used).  The rope half of each key (32 dims, 64 bytes per CTA) is kept in a
// 64-byte-swizzled slab instead of half of a 128-byte one, which brings an
// operand stage to 72 KB and lets two of them, the fp8 raw slots and Q fit.
//
// The rest is the 128-row kernel's design: a CTA pair per (sequence, split)
// splits the value dims (CTA r owns dims [256r, 256r + 256) and contracts
// its 256 latent + 32 rope dims), swaps 24-bit partial scores with the
// partner over distributed shared memory, and runs a lazily rescaled online
// softmax in the softmax warps whose 16-row block holds real rows.
//
// Per 128-key tile:
//   loader warps  : L warps (4 in the narrow form, 3 in the wide one), loader
//                   l owning parts Li + l of the tile sequence (64 keys for
//                   bf16, 32 for fp8): block-table lookup, 16-byte cp.async
//                   of the part's row pieces into the tile's stage (bf16) or
//                   into one of the loader's raw slots, converted to f16 by
//                   the same lanes (fp8, the next part's copy already in
//                   flight); every part arrives on the stage's barrier, and
//                   a part's stage rows are refilled as soon as the last
//                   value MMA that reads them is done.
//   MMA warp      : S_part = Q_part K_part^T (18 MMAs, N = 128, A = Q from
//                   shared memory), then O_half += P V_half (8 MMAs, N =
//                   256, A = P from TMEM, B = the same stage read MN-major;
//                   up to 8 more with the low-order weights, one for each
//                   16-key group that holds a heavy key).
//   softmax warps : as in the 128-row kernel, two warps per 16-row quarter,
//                   each over one 64-key half of the tile: 32 scores a
//                   thread, 3 KB swapped per warp and tile, row maxima and
//                   sums traded with the other warp of the quarter.
//
// Every wait is bounded (2 s unless the plan sets another limit); a wait
// that runs out sets MLA_DEVFLAG_TIMEOUT and the CTA winds down.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mla_decode.h"
#include "internal.h"
#include "ptx.cuh"

namespace {

constexpr int T = mla::kKeyTileSmall;   // 128 keys per tile
constexpr int ATOM = T * 128;           // one 64-dim latent slab of a stage: 16 KB
constexpr int RATOM = T * 64;           // the CTA's rope half, 64-byte rows: 8 KB
constexpr int STAGE = 4 * ATOM + RATOM; // 72 KB
constexpr int NS = 2;                   // operand stages (one tile each)
template <bool kFp8>
struct LoadPart {
  static constexpr int keys = kFp8 ? 32 : 64;  // keys of one loader part
};
constexpr int RAW_PART = 32 * (256 + 32);      // fp8 codes of a 32-key part: 9 KB
// Raw slots: two for each loader warp but the first, which owns a tile's
// first part (the first the value MMAs release) and has one.
constexpr int NR = 7;
// Rows and warps: a warp reaches only the TMEM lane quarter warp % 4, and
// each quarter belongs to one SM sub-partition.  So that all four
// sub-partitions share the softmax, the (at most 64) rows are spread 16 to a
// quarter: row 16 q + i of the problem is row 32 q + i of the MMA's A and of
// every accumulator (lanes 32 q + 16 .. 32 q + 31 hold unused rows).
//
// Key split: the two warps that reach a quarter (q and q + 4) share each
// 128-key tile, 64 keys each (key half kh = warp / 4), and trade their row
// maxima and sums through shared memory, so a softmax warp holds 32 scores a
// thread.  Two forms:
//   narrow (at most 16 rows, quarter 0 only): 8 warps; 0 and 4 softmax,
//     6, 1, 2, 3 load (loader index 0..3, so with 32-key parts warp 1 + i
//     owns part i of every tile and the two parts that share a sub-partition
//     are released first and third), 5 idle, 7 issues the MMAs;
//   wide (17 to 64 rows, bf16): 12 warps; 0-7 softmax (two per quarter),
//     8-10 load, 11 issues the MMAs (168 registers a thread).
template <bool kWide>
struct Warps {
  static constexpr int count = kWide ? 12 : 8;
  static constexpr int softmax = kWide ? 8 : 2;
  static constexpr int loaders = kWide ? 3 : 4;
  static constexpr int mma = kWide ? 11 : 7;
};
template <bool kWide>
__device__ __forceinline__ bool is_softmax_warp(int w) { return kWide ? w < 8 : (w == 0 || w == 4); }
template <bool kWide>
__device__ __forceinline__ bool is_loader_warp(int w) {
  return kWide ? (w >= 8 && w <= 10) : ((w >= 1 && w <= 3) || w == 6);
}
template <bool kWide>
__device__ __forceinline__ int loader_index(int w) { return kWide ? w - 8 : (w == 6 ? 0 : w); }
__device__ __forceinline__ int mma_row(int r) { return 32 * (r >> 4) + (r & 15); }
constexpr int RECV_W = 32 * 16 * 6;     // one warp's partial scores: 16 rows x 64 keys x 3 B (3 KB)

template <bool kFp8>
struct Layout {
  // Q as the A operand (128 MMA rows, K-major; the MMA reads all 128 rows of
  // a slab, 16 KB, and the unused ones may hold anything).  bf16 (up to 64
  // rows, at MMA rows 32 q + i): the real rows of a latent slab are its
  // 8-row groups 4q and 4q + 1, so slabs 2k and 2k + 1 interleave 2 KB
  // apart in one 16 KB span (each one's unused groups are the other's rows):
  // 32 KB of latent slabs, then the rope slab (64-byte rows, 8 KB).  fp8 (up
  // to 16 rows, MMA rows 0..15): slabs of 16 rows packed 2 KB apart, their
  // unused rows reading into the stages, then the rope rows (1 KB).
  __host__ __device__ static constexpr int qslab_off(int a) {
    return kFp8 ? a * 2048 : (a >> 1) * 16384 + (a & 1) * 2048;
  }
  __host__ __device__ static constexpr int qrope_off() { return kFp8 ? 4 * 2048 : 2 * 16384; }
  __host__ __device__ static constexpr int qbytes() { return kFp8 ? 4 * 2048 + 1024 : 2 * 16384 + 8192; }
  static constexpr int max_rows = kFp8 ? 16 : 64;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_STAGE = (qbytes() + 1023) / 1024 * 1024;  // 40 KB bf16, 9 KB fp8
  static constexpr int OFF_RAW = OFF_STAGE + NS * STAGE;
  static constexpr int OFF_RECV = OFF_RAW + (kFp8 ? NR * RAW_PART : 0);
  static constexpr int RECV = (max_rows / 16) * 2 * RECV_W;  // two softmax warps a quarter
  static constexpr int OFF_XFREE = OFF_RECV + RECV;
  // the key-split exchange: [quarter][3 slots][2 warps][32 lanes] x 16 B
  static constexpr int OFF_XMAX = OFF_XFREE + 128;
  static constexpr int OFF_BAR = OFF_XMAX + (max_rows / 16) * 3 * 2 * 32 * 16;
  static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;
};
static_assert(Layout<false>::SMEM_BYTES <= 232448, "bf16 smem");
static_assert(Layout<true>::SMEM_BYTES <= 232448, "fp8 smem");
static_assert(Layout<false>::OFF_STAGE % 1024 == 0 && Layout<true>::OFF_STAGE % 1024 == 0 &&
                  STAGE % 1024 == 0 && RATOM % 512 == 0,
              "swizzle atoms stay aligned");

// TMEM columns
constexpr uint32_t TM_O = 0;    // 256 fp32 columns: this CTA's value half
constexpr uint32_t TM_S = 256;  // two 128-column score buffers; P overwrites them
                                // (bf16: cols 0..63 weights, 64..127 low-order terms)
constexpr uint32_t TM_COLS = 512;

constexpr float kRescaleThreshold = 8.0f;
constexpr float kMaxSentinel = -1.0e30f;
constexpr uint64_t kDrainNs = 500000000ull;
constexpr uint32_t kSleepNs = 20000;

struct Bars {
  uint64_t kv_full[NS];   // every loader part of the stage landed (32 lanes a part)
  uint64_t kv_empty[NS][4];  // a loader part's rows of the stage are read for the last time
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t recv_full[8];  // per softmax warp
  uint64_t recv_free[8];
  uint64_t o_done;
  uint64_t o_final;
  uint64_t q_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort;
  uint64_t heavy[2];
  uint64_t xchg[4][3];  // per quarter: the two warps' maxima (per tile parity) and final sums
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

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two_codes));
  return r;
}

__device__ __forceinline__ uint32_t round_up_bits(float x) { return __float_as_uint(x) + 0x80u; }

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
__device__ __forceinline__ uint64_t kdesc128(uint32_t addr) { return ptx::smem_desc(addr, 16, 1024, 2); }
// K-major, 64B-swizzled operand (the rope halves): rows 64 B apart, 8-row groups 512 B apart.
__device__ __forceinline__ uint64_t kdesc64(uint32_t addr) { return ptx::smem_desc(addr, 16, 512, 4); }
// The stage read MN-major as V: N = 256 value dims over 4 slabs ATOM apart,
// K = keys in 8-row groups 1 KB apart.
__device__ __forceinline__ uint64_t vdesc(uint32_t addr) { return ptx::smem_desc(addr, ATOM, 1024, 2); }

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128B-swizzled slab,
// and of chunk `c` (0..3) of row `r` in a 64B-swizzled one.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return r * 128 + ((c ^ (r & 7)) * 16); }
__device__ __forceinline__ uint32_t sw64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) * 16); }

template <bool kFp8, bool kWide>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Warps<kWide>::count * 32, 1)
    fwd_small_kernel(mla::FwdParams p) {
  using L = Layout<kFp8>;
  constexpr uint32_t kAB = kFp8 ? 0u : 1u;
  constexpr int PART = LoadPart<kFp8>::keys;
  constexpr int UPT = T / PART;  // loader parts per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Bars& bars = *reinterpret_cast<Bars*>(smem + L::OFF_BAR);
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  // The work unit (as in the 128-row kernel; rows fit one block here).
  int b, ctx, k0, k1;
  bool single;
  size_t part;
  if (p.units != nullptr) {
    ptx::grid_dependency_wait();
    const int u = blockIdx.x >> 1;
    if (u >= *p.n_units) return;
    const int4 d = p.units[u];
    const int4 si = p.seq_info[d.x];
    b = d.x;
    k0 = d.z;
    k1 = d.w;
    ctx = si.x;
    single = si.z == 1;
    part = (size_t)si.y + (d.y >> 8);
  } else {
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
  const float s_kv = (p.kv_dtype == MLA_KV_FP8_E4M3 && p.kv_scale) ? *p.kv_scale : 1.f;

  if (n_tiles == 0) {
    ptx::grid_dependency_wait();
    for (int row = threadIdx.x; row < p.rows; row += blockDim.x) {
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
      ptx::mbar_init(ptx::smem_u32(&bars.kv_full[s]), 32 * UPT);
      for (int h = 0; h < 4; ++h) ptx::mbar_init(ptx::smem_u32(&bars.kv_empty[s][h]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(&bars.s_full[i]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.p_full[i]), 32 * Warps<kWide>::softmax);
    }
    for (int w = 0; w < 8; ++w) {
      ptx::mbar_init(ptx::smem_u32(&bars.recv_full[w]), 1);
      ptx::mbar_init(ptx::smem_u32(&bars.recv_free[w]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&bars.o_done), 1);
    ptx::mbar_init(ptx::smem_u32(&bars.o_final), 1);
    ptx::mbar_init(ptx::smem_u32(&bars.q_ready), 32 * Warps<kWide>::softmax);
    ptx::mbar_init(ptx::smem_u32(&bars.drain), 1);
    for (int q = 0; q < 4; ++q)
      for (int i = 0; i < 3; ++i) ptx::mbar_init(ptx::smem_u32(&bars.xchg[q][i]), 64);
    bars.heavy[0] = bars.heavy[1] = 0;  // bytes of absent warps stay zero
    bars.abort = 0;
    ptx::fence_mbar_init_cluster();
  }
  if (warp == Warps<kWide>::mma) {
    ptx::tmem_alloc(ptx::smem_u32(&bars.tmem_base), TM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync_all();
  ptx::tc_fence_after();
  ptx::grid_dependency_wait();
  const uint32_t tmem = bars.tmem_base;
  Ctx c{p.status, &bars.abort, p.wait_ns,
        (uint32_t)(p.wait_ns < (uint64_t)kSleepNs ? p.wait_ns : (uint64_t)kSleepNs)};

  if (warp == Warps<kWide>::mma) {
    // --------------------------------------------------------------- MMA ---
    if (lane == 0) {
      const uint32_t id_qk = ptx::idesc_f16(128, T, kAB, false, false);
      const uint32_t id_pv = ptx::idesc_f16(128, 256, kAB, false, true);
      bool ok = wait(c, ptx::smem_u32(&bars.q_ready), 0);
      ptx::tc_fence_after();
      const uint32_t qa = sbase + L::OFF_Q;
      auto issue_qk = [&](int u) {
        const uint32_t d = tmem + TM_S + (u & 1) * T;
        const uint32_t st = sbase + L::OFF_STAGE + (u % NS) * STAGE;
        for (int a = 0; a < 4; ++a)
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ss(d, kdesc128(qa + L::qslab_off(a) + kk * 32),
                        kdesc128(st + a * ATOM + kk * 32), id_qk, (a | kk) != 0);
        for (int kk = 0; kk < 2; ++kk)  // this CTA's 32 rope dims
          ptx::mma_ss(d, kdesc64(qa + L::qrope_off() + kk * 32), kdesc64(st + 4 * ATOM + kk * 32),
                      id_qk, 1);
        ptx::mma_commit(ptx::smem_u32(&bars.s_full[u & 1]));
      };
      // heavy: bit kk asks for the low-order weights of the tile's 16-key group kk
      auto issue_pv = [&](int t, uint32_t heavy) {
        const int s = t % NS;
        const uint32_t pa = tmem + TM_S + (t & 1) * T;
        const uint32_t st = sbase + L::OFF_STAGE + s * STAGE;
        const bool two = !kFp8 && heavy != 0;
        constexpr int MPP = PART / 16;  // value MMAs (16 keys each) per loader part
        for (int kk = 0; kk < T / 16; ++kk) {
          ptx::mma_ts(tmem + TM_O, pa + kk * 8, vdesc(st + kk * 2048), id_pv, (t | kk) != 0);
          // the part's rows are read for the last time (the score MMAs of
          // this tile are long done): its loader may refill them
          if (!two && kk % MPP == MPP - 1) ptx::mma_commit(ptx::smem_u32(&bars.kv_empty[s][kk / MPP]));
        }
        if (two) {
          for (int kk = 0; kk < T / 16; ++kk)
            if ((heavy >> kk) & 1u)
              ptx::mma_ts(tmem + TM_O, pa + T / 2 + kk * 8, vdesc(st + kk * 2048), id_pv, 1);
        }
        ptx::mma_commit(ptx::smem_u32(&bars.o_done));
        if (t == n_tiles - 1) ptx::mma_commit(ptx::smem_u32(&bars.o_final));
        if (two)
          for (int h = 0; h < UPT; ++h) ptx::mma_commit(ptx::smem_u32(&bars.kv_empty[s][h]));
      };
      int nq = 0, np = 0;
      uint64_t t_last = ptx::globaltimer_ns();
      uint32_t idle = 0;
      while (ok && np < n_tiles) {
        bool progress = false;
        if (nq < n_tiles && nq <= np + 1 &&
            ptx::mbar_test_wait(ptx::smem_u32(&bars.kv_full[nq % NS]), (nq / NS) & 1)) {
          ptx::tc_fence_after();
          issue_qk(nq++);
          progress = true;
        }
        if (np < nq && ptx::mbar_test_wait(ptx::smem_u32(&bars.p_full[np & 1]), (np >> 1) & 1)) {
          ptx::tc_fence_after();
          const uint64_t hv = *reinterpret_cast<volatile uint64_t*>(&bars.heavy[np & 1]);
          uint32_t heavy = 0;  // the OR of the softmax warps' bytes
          for (int i = 0; i < 8; ++i) heavy |= (uint32_t)(hv >> (8 * i)) & 0xFFu;
          issue_pv(np++, heavy);
          progress = true;
        }
        if (progress) {
          idle = 0;
          t_last = 0;
          continue;
        }
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
  } else if (is_loader_warp<kWide>(warp)) {
    // ------------------------------------------------------------ loader ---
    // The tile sequence of the split is cut into parts of PART keys (64 for
    // bf16, 32 for fp8); loader warp w fills parts u = w, w + 3, ... (tile
    // u / UPT, keys PART (u % UPT) .. of it) into stage (u / UPT) % 2.  A key's
    // piece of a 64-dim latent slab is 128 bytes (8 lanes x 16 B for bf16, 4
    // lanes x 16 codes for fp8) and its rope half 64 bytes (4 lanes of bf16,
    // 2 of fp8).  bf16 copies go straight into the stage once it is free.
    // fp8 codes go into one of the warp's two raw slots and are converted to
    // f16 by the same lanes; the copy of the warp's next part is issued before
    // the current one waits for its stage and converts, so a part is always in
    // flight.
    constexpr int LPI = kFp8 ? 4 : 8;  // lanes per 128-byte latent piece
    constexpr int IPI = 32 / LPI;      // keys per warp instruction
    constexpr int NK = PART / IPI;     // keys per lane and part: 16 (bf16) or 4 (fp8)
    const int g = lane / LPI, sub = lane % LPI;
    const int32_t* bt =
        p.bt + (p.bt_indptr ? (size_t)p.bt_indptr[b] : (size_t)b * p.bt_stride);
    const char* cache = static_cast<const char*>(p.cache);
    const int n_units = UPT * n_tiles;
    const int lw = loader_index<kWide>(warp);
    constexpr int kLoaders = Warps<kWide>::loaders;
    // i-th key of this lane in part u, clamped to the split's last key k1 - 1:
    // a partial part, or the empty parts of a split's last tile, repeat a real
    // row (its weights are masked to zero), so every key read lies in
    // [k0, k1) and no stage slot the value MMA reads holds anything but cache
    // rows.
    auto key_of = [&](int u, int i) -> int { return min(k0 + u * PART + i * IPI + g, k1 - 1); };
    const uint32_t pdiv = (uint32_t)p.page_size;
    const uint32_t plog = 32u - __clz(pdiv - 1u);
    const uint32_t pmul = (uint32_t)(((1ull << 32) * ((1ull << plog) - pdiv)) / pdiv) + 1u;
    const uint32_t pshift = plog > 0 ? plog - 1u : 0u;
    auto page_of = [&](uint32_t key) -> uint32_t {
      const uint32_t t = __umulhi(pmul, key);
      return pdiv == 1u ? key : (t + ((key - t) >> 1)) >> pshift;
    };
    int pg[NK];
    auto load_pages = [&](int u) {
      if (u >= n_units) return;
#pragma unroll
      for (int i = 0; i < NK; ++i) pg[i] = __ldg(&bt[page_of((uint32_t)key_of(u, i))]);
    };
    uint32_t rix[NK];  // cache row of each key of a part (num_pages * page_size < 2^31)
    auto rows_of = [&](int u) {  // from the block-table entries in pg
      bool bad = false;
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        int64_t page = pg[i];
        if (page < 0 || page >= p.num_pages) {
          bad = true;
          page = 0;
        }
        const uint32_t key = (uint32_t)key_of(u, i);
        rix[i] = (uint32_t)page * pdiv + (key - page_of(key) * pdiv);
      }
      if (bad) atomicOr(p.status, MLA_DEVFLAG_BAD_PAGE);
    };
    auto row = [&](int i) { return cache + (size_t)rix[i] * (kFp8 ? mla::kDQK : mla::kDQK * 2); };
    load_pages(lw);
    if constexpr (!kFp8) {
      for (int u = lw; u < n_units; u += kLoaders) {
        const int t = u / UPT, h = u % UPT, s = t % NS;
        rows_of(u);
        load_pages(u + kLoaders);
        const uint32_t stage = sbase + L::OFF_STAGE + s * STAGE;
        if (t >= NS && !wait_all(c, ptx::smem_u32(&bars.kv_empty[s][h]), ((t / NS) - 1) & 1)) break;
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int kk = h * PART + i * IPI + g;  // key within the tile
#pragma unroll
          for (int sl = 0; sl < 4; ++sl)
            ptx::cp_async_16(stage + sl * ATOM + sw128(kk, sub), row(i) + (vdim0 + sl * 64 + sub * 8) * 2);
          if (sub < 4)  // the CTA's rope half: dims 512 + 32 rank + 8 sub
            ptx::cp_async_16(stage + 4 * ATOM + sw64(kk, sub), row(i) + (512 + 32 * (int)rank + sub * 8) * 2);
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait<0>();
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(ptx::smem_u32(&bars.kv_full[s]));
      }
    } else {
      // raw slot j of this warp: [PART keys][288 codes]; loader 0 has one
      const int nslot = lw == 0 ? 1 : 2;
      auto raw_slot = [&](int j) { return sbase + L::OFF_RAW + (lw == 0 ? 0 : 2 * lw - 1 + j) * RAW_PART; };
      auto issue_raw = [&](int u, int j) {
        rows_of(u);
        const uint32_t raw = raw_slot(j);
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int kr = i * IPI + g;  // key within the part
#pragma unroll
          for (int sl = 0; sl < 4; ++sl)
            ptx::cp_async_16(raw + kr * 288 + sl * 64 + sub * 16, row(i) + vdim0 + sl * 64 + sub * 16);
          if (sub < 2)
            ptx::cp_async_16(raw + kr * 288 + 256 + sub * 16, row(i) + 512 + 32 * (int)rank + sub * 16);
        }
      };
      if (lw < n_units) issue_raw(lw, 0);
      ptx::cp_async_commit();
      load_pages(lw + kLoaders);
      int j = 0;
      for (int u = lw; u < n_units; u += kLoaders, j ^= nslot - 1) {
        const int un = u + kLoaders;
        if (nslot == 2 && un < n_units) {
          issue_raw(un, j ^ 1);
          load_pages(un + kLoaders);
        }
        ptx::cp_async_commit();
        ptx::cp_async_wait<1>();  // this lane's copies of part u have landed
        const int t = u / UPT, h = u % UPT, s = t % NS;
        if (t >= NS && !wait_all(c, ptx::smem_u32(&bars.kv_empty[s][h]), ((t / NS) - 1) & 1)) break;
        // e4m3 codes -> f16 operands (exact); the per-tensor scale goes to
        // the scores and the output instead.  A lane converts the codes it
        // copied.
        const uint32_t stage = sbase + L::OFF_STAGE + s * STAGE;
        const uint32_t raw = raw_slot(j);
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const int kr = i * IPI + g, kk = h * PART + kr;
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            const uint4 x = ld_shared_u4(raw + kr * 288 + sl * 64 + sub * 16);
            uint4 lo, hi;
            lo.x = e4m3x2_to_f16x2(x.x);
            lo.y = e4m3x2_to_f16x2(x.x >> 16);
            lo.z = e4m3x2_to_f16x2(x.y);
            lo.w = e4m3x2_to_f16x2(x.y >> 16);
            hi.x = e4m3x2_to_f16x2(x.z);
            hi.y = e4m3x2_to_f16x2(x.z >> 16);
            hi.z = e4m3x2_to_f16x2(x.w);
            hi.w = e4m3x2_to_f16x2(x.w >> 16);
            st_shared_u4(stage + sl * ATOM + sw128(kk, 2 * sub), lo);
            st_shared_u4(stage + sl * ATOM + sw128(kk, 2 * sub + 1), hi);
          }
          if (sub < 2) {
            const uint4 x = ld_shared_u4(raw + kr * 288 + 256 + sub * 16);
            uint4 lo, hi;
            lo.x = e4m3x2_to_f16x2(x.x);
            lo.y = e4m3x2_to_f16x2(x.x >> 16);
            lo.z = e4m3x2_to_f16x2(x.y);
            lo.w = e4m3x2_to_f16x2(x.y >> 16);
            hi.x = e4m3x2_to_f16x2(x.z);
            hi.y = e4m3x2_to_f16x2(x.z >> 16);
            hi.z = e4m3x2_to_f16x2(x.w);
            hi.w = e4m3x2_to_f16x2(x.w >> 16);
            st_shared_u4(stage + 4 * ATOM + sw64(kk, 2 * sub), lo);
            st_shared_u4(stage + 4 * ATOM + sw64(kk, 2 * sub + 1), hi);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive(ptx::smem_u32(&bars.kv_full[s]));
        if (nslot == 1 && un < n_units) {  // its one slot is free again
          issue_raw(un, 0);
          load_pages(un + kLoaders);
          ptx::cp_async_commit();
        }
      }
    }
    ptx::cp_async_wait<0>();
  } else if (!is_softmax_warp<kWide>(warp)) {
    // warp 5 of the narrow form: no work
  } else {
    // ----------------------------------------------------------- softmax ---
    // As in the 128-row kernel's 16x256b access: warp q owns TMEM lanes
    // 32 q .. 32 q + 15 (problem rows 16 q .. 16 q + 15); thread i holds
    // lanes 32 q + i/4 and + 8 (rows rA = 16 q + i/4, rB = rA + 8) and, of
    // every 8-key group j of its 64-key half kh, keys 64 kh + 8j + 2(i%4) and
    // + 1.  Only warps whose rows are real work; the others keep the barrier
    // phases moving.
    constexpr int NSW = Warps<kWide>::softmax;
    const int q4 = warp & 3;
    const int kh = warp >> 2;     // key half
    const int sw = 2 * q4 + kh;   // index among the softmax warps
    const int lbase = q4 * 32;
    const int cq = lane & 3;
    const int rA = 16 * q4 + (lane >> 2), rB = rA + 8;  // problem rows
    const uint32_t lanes16 = (uint32_t)lbase << 16;
    auto visible = [&](int r) {
      if (r >= p.rows) return 0;
      const int tok = r / p.heads;
      int nvis = p.causal ? ctx - p.sq + tok + 1 : ctx;
      nvis = max(0, min(nvis, ctx));
      return min(nvis, k1);
    };
    const int visA = visible(rA), visB = visible(rB);
    const bool live = 16 * q4 < p.rows;

    // Q -> shared memory: this CTA's 256 latent dims (4 slabs, 128B swizzle)
    // and its 32 rope dims (64B swizzle), problem row r at MMA row
    // mma_row(r).
    {
      bool q_range = false;
      const int n_pieces = p.rows * 36;  // per row: 4 slabs x 8 chunks + 4 rope chunks
      // Piece i of row r: its global source and its place in shared memory.
      auto piece = [&](int i, uint4& x, uint32_t& dst) {
        const int r = i / 36, pc = i % 36, ar = mma_row(r);
        const uint16_t* qrow = p.q + ((size_t)b * p.rows + r) * mla::kDQK;
        if (pc < 32) {
          const int sl = pc >> 3, ch = pc & 7;
          x = reinterpret_cast<const uint4*>(qrow + vdim0 + sl * 64)[ch];
          dst = sbase + L::OFF_Q + L::qslab_off(sl) + sw128(ar, ch);
        } else {
          const int ch = pc - 32;
          x = reinterpret_cast<const uint4*>(qrow + 512 + 32 * (int)rank)[ch];
          dst = sbase + L::OFF_Q + L::qrope_off() + sw64(ar, ch);
        }
      };
      // Up to kQPieces pieces a thread (every form's row limit keeps it
      // there): every load first, then the stores, which are ordered memory
      // operations that loads between them would each wait for.
      constexpr int kQPieces = 9;
      const int i0 = sw * 32 + lane, step = 32 * NSW;
      uint4 xs[kQPieces];
      uint32_t dsts[kQPieces];
#pragma unroll
      for (int k = 0; k < kQPieces; ++k)
        if (i0 + k * step < n_pieces) piece(i0 + k * step, xs[k], dsts[k]);
#pragma unroll
      for (int k = 0; k < kQPieces; ++k)
        if (i0 + k * step < n_pieces) {
          if (kFp8) xs[k] = bf16x8_to_f16x8(xs[k], q_range);
          st_shared_u4(dsts[k], xs[k]);
        }
      for (int i = i0 + kQPieces * step; i < n_pieces; i += step) {  // beyond the forms' limits
        uint4 x;
        uint32_t dst;
        piece(i, x, dst);
        if (kFp8) x = bf16x8_to_f16x8(x, q_range);
        st_shared_u4(dst, x);
      }
      if (kFp8 && q_range) atomicOr(p.status, MLA_DEVFLAG_Q_RANGE);
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(ptx::smem_u32(&bars.q_ready));
    }

    const float c2 = p.softmax_scale * s_kv * 1.4426950408889634f;
    float mA = kMaxSentinel, mB = kMaxSentinel;
    float lA = 0.f, lB = 0.f;
    const uint32_t my_recv = sbase + L::OFF_RECV + sw * RECV_W;  // this warp's receive slot
    const uint32_t peer_recv = ptx::mapa(my_recv, peer);
    const uint32_t peer_free = ptx::mapa(sbase + L::OFF_XFREE + sw * 4, peer);
    const uint32_t recv_full = ptx::smem_u32(&bars.recv_full[sw]);
    const uint32_t recv_free = ptx::smem_u32(&bars.recv_free[sw]);
    // slot i of warp w (key half) of this quarter in the exchange area
    auto xslot = [&](int i, int w) {
      return sbase + L::OFF_XMAX + ((q4 * 3 + i) * 2 + w) * 512 + lane * 16;
    };
    const uint32_t xchg0 = ptx::smem_u32(&bars.xchg[q4][0]);  // tile parity i at xchg0 + 8 i
    const uint32_t xchg_end = ptx::smem_u32(&bars.xchg[q4][2]);
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
      // s[4 j + e]: 8-key group j of the key half; e = 0, 1 -> row A keys
      // 64 kh + 8j + 2cq + e; e = 2, 3 -> row B
      float s[32];
      {
        uint32_t raw[32];
        ptx::tmem_ld16x256b_x8(scol + kh * 64, raw);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(raw[i]);
      }
      // Swap partial scores with the same warp of the partner CTA (single
      // receive buffer: tile t goes once the partner has read tile t - 1).
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
          for (int k = 0; k < 4; ++k)
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
            float uu[4];
            unpack24(w + 3 * k, uu);
#pragma unroll
            for (int e = 0; e < 4; ++e) s[16 * qd + 4 * k + e] += uu[e];
          }
        }
        const bool any = __any_sync(0xffffffffu, fold == 0x9E3779B9u);
        if (t + 1 < n_tiles && lane == 0)
          ptx::st_async_b32(peer_free, any ? 1u : 0u, ptx::mapa(recv_free, peer));
      }
      const int tile0 = k0 + t * T;
      const int limA = visA - tile0, limB = visB - tile0;
      const bool all_full = __all_sync(0xffffffffu, limA >= T && limB >= T);
      float mxA = -INFINITY, mxB = -INFINITY;
      if (all_full) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          mxA = fmaxf(mxA, fmaxf(s[4 * j], s[4 * j + 1]));
          mxB = fmaxf(mxB, fmaxf(s[4 * j + 2], s[4 * j + 3]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int k = 64 * kh + 8 * j + 2 * cq + e;
            if (k < limA) mxA = fmaxf(mxA, s[4 * j + e]);
            if (k < limB) mxB = fmaxf(mxB, s[4 * j + 2 + e]);
          }
      }
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
      // The two warps of the quarter trade their half-tile maxima and their
      // sums so far (the same lane holds the same rows in both), so that
      // both take the same rescale decisions and keep one running max.  Two
      // slots by tile parity: a warp writes slot t % 2 again only after the
      // other has passed tile t + 1's exchange, so after it read tile t's
      // values.
      float olA, olB;
      {
        st_shared_u4(xslot(buf, kh), make_uint4(__float_as_uint(mxA), __float_as_uint(mxB),
                                                __float_as_uint(lA), __float_as_uint(lB)));
        ptx::mbar_arrive(xchg0 + 8 * buf);
        if (!wait_all(c, xchg0 + 8 * buf, (t >> 1) & 1)) { ok = false; break; }
        const uint4 o = ld_shared_u4(xslot(buf, kh ^ 1));
        mxA = fmaxf(mxA, __uint_as_float(o.x));
        mxB = fmaxf(mxB, __uint_as_float(o.y));
        olA = __uint_as_float(o.z);
        olB = __uint_as_float(o.w);
      }
      const float mtA = limA > 0 ? mxA * c2 : -INFINITY;
      const float mtB = limB > 0 ? mxB * c2 : -INFINITY;
      const bool needA = mtA > mA + kRescaleThreshold, needB = mtB > mB + kRescaleThreshold;
      float alA = 1.f, alB = 1.f;
      if (__any_sync(0xffffffffu, needA || needB)) {
        const float nA = needA ? fmaxf(mA, mtA) : mA, nB = needB ? fmaxf(mB, mtB) : mB;
        alA = exp2f(mA - nA);
        alB = exp2f(mB - nB);
        if (t > 0) {
          // The PV of the previous tile must have finished: QK^T of this
          // tile was issued after PV of tile t - 2 and the pipe runs in
          // order, so o_done is at most one phase short.
          if (!wait_all(c, ptx::smem_u32(&bars.o_done), (t - 1) & 1)) { ok = false; break; }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int ch = 2 * kh; ch < 2 * kh + 2; ++ch) {
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
      // Weights p = 2^(s*c2 - m), 16-bit pairs to TMEM by key half: weights
      // in columns 0..63, for bf16 the low-order terms in 64..127.
      const float nmA = -mA, nmB = -mB;
      float sA = 0.f, sB = 0.f;
      const uint32_t pcol = tmem + lanes16 + TM_S + buf * T;
      float gA[4] = {0.f, 0.f, 0.f, 0.f}, gB[4] = {0.f, 0.f, 0.f, 0.f};  // per 16-key group
      {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = 64 * kh + 8 * j + 2 * cq;
          float a0 = fast_exp2(fmaf(s[4 * j], c2, nmA));
          float a1 = fast_exp2(fmaf(s[4 * j + 1], c2, nmA));
          float b0 = fast_exp2(fmaf(s[4 * j + 2], c2, nmB));
          float b1 = fast_exp2(fmaf(s[4 * j + 3], c2, nmB));
          if (!all_full) {
            a0 = k < limA ? a0 : 0.f;
            a1 = k + 1 < limA ? a1 : 0.f;
            b0 = k < limB ? b0 : 0.f;
            b1 = k + 1 < limB ? b1 : 0.f;
          }
          sA += a0 + a1;
          sB += b0 + b1;
          if (!kFp8) {
            gA[j >> 1] = fmaxf(gA[j >> 1], fmaxf(a0, a1));
            gB[j >> 1] = fmaxf(gB[j >> 1], fmaxf(b0, b1));
          }
          hi[2 * j] = kFp8 ? pack_f16(a0, a1) : pack_bf16(a0, a1);
          hi[2 * j + 1] = kFp8 ? pack_f16(b0, b1) : pack_bf16(b0, b1);
          if (!kFp8) {
            lo[2 * j] = pack_bf16(a0 - __uint_as_float(hi[2 * j] << 16),
                                   a1 - __uint_as_float(hi[2 * j] & 0xFFFF0000u));
            lo[2 * j + 1] = pack_bf16(b0 - __uint_as_float(hi[2 * j + 1] << 16),
                                       b1 - __uint_as_float(hi[2 * j + 1] & 0xFFFF0000u));
          }
        }
        ptx::tmem_st16x128b_x8(pcol + kh * 32, hi);
        if (!kFp8) ptx::tmem_st16x128b_x8(pcol + T / 2 + kh * 32, lo);
      }
      lA += sA;
      lB += sB;
      if constexpr (!kFp8) {
        // The low-order terms are written for every tile; the second PV runs
        // only over the 16-key groups where one key carries more than 1/16
        // of a row's weight.  The row's sum counts the other warp's keys up
        // to the previous tile only, which errs towards the second PV.  Bit
        // g of this warp's byte is group 4 kh + g of the tile.
        float rsA = lA + olA * alA, rsB = lB + olB * alB;
        rsA += __shfl_xor_sync(0xffffffffu, rsA, 1);
        rsB += __shfl_xor_sync(0xffffffffu, rsB, 1);
        rsA += __shfl_xor_sync(0xffffffffu, rsA, 2);
        rsB += __shfl_xor_sync(0xffffffffu, rsB, 2);
        uint32_t gm = 0;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          if (gA[g] * 16.f > rsA || gB[g] * 16.f > rsB) gm |= 1u << g;
        gm = __reduce_or_sync(0xffffffffu, gm);
        if (lane == 0) reinterpret_cast<volatile uint8_t*>(&bars.heavy[buf])[sw] = (uint8_t)(gm << (4 * kh));
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_u32(&bars.p_full[buf]));
    }

    // ---------------------------------------------------------- epilogue ---
    if (ok) {  // the other warp's share of the row sums
      st_shared_u4(xslot(2, kh), make_uint4(__float_as_uint(lA), __float_as_uint(lB), 0u, 0u));
      ptx::mbar_arrive(xchg_end);
      if (wait_all(c, xchg_end, 0)) {
        const uint4 o = ld_shared_u4(xslot(2, kh ^ 1));
        lA += __uint_as_float(o.x);
        lB += __uint_as_float(o.y);
      } else {
        ok = false;
      }
    }
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    if (ok && live && wait_all(c, ptx::smem_u32(&bars.o_final), 0)) {
      ptx::tc_fence_after();
      const float invA = lA > 0.f ? s_kv / lA : 0.f, invB = lB > 0.f ? s_kv / lB : 0.f;
      const bool okA = rA < p.rows, okB = rB < p.rows;
      const size_t pA = part * p.rows + rA;  // problem rows (TMEM lanes are spread)
      const size_t pB = part * p.rows + rB;
#pragma unroll 1
      for (int ch = 2 * kh; ch < 2 * kh + 2; ++ch) {
        uint32_t o[32];
        ptx::tmem_ld16x256b_x8(tmem + lanes16 + TM_O + ch * 64, o);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int dim = vdim0 + ch * 64 + 8 * j + 2 * cq;
          const float a0 = __uint_as_float(o[4 * j]) * invA, a1 = __uint_as_float(o[4 * j + 1]) * invA;
          const float b0 = __uint_as_float(o[4 * j + 2]) * invB, b1 = __uint_as_float(o[4 * j + 3]) * invB;
          if (single) {
            if (okA) *reinterpret_cast<uint32_t*>(p.out + ((size_t)b * p.rows + rA) * mla::kDV + dim) = pack_bf16(a0, a1);
            if (okB) *reinterpret_cast<uint32_t*>(p.out + ((size_t)b * p.rows + rB) * mla::kDV + dim) = pack_bf16(b0, b1);
          } else {
            if (okA) *reinterpret_cast<float2*>(p.part_o + pA * mla::kDV + dim) = make_float2(a0, a1);
            if (okB) *reinterpret_cast<float2*>(p.part_o + pB * mla::kDV + dim) = make_float2(b0, b1);
          }
        }
      }
      if (rank == 0 && cq == 0 && kh == 0) {
        const float lseA = lA > 0.f ? (mA + log2f(lA)) * 0.6931471805599453f : -INFINITY;
        const float lseB = lB > 0.f ? (mB + log2f(lB)) * 0.6931471805599453f : -INFINITY;
        if (single) {
          if (okA) p.lse[(size_t)b * p.rows + rA] = lseA;
          if (okB) p.lse[(size_t)b * p.rows + rB] = lseB;
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
  if (warp == Warps<kWide>::mma) {
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
  ptx::cluster_sync_all();
}

}  // namespace

bool mla_small_rows_fit(int rows, int kv_dtype) {
  return rows <= (kv_dtype == MLA_KV_FP8_E4M3 ? Layout<true>::max_rows : Layout<false>::max_rows);
}

int mla_launch_fwd_small_sm103(const mla::FwdParams& p, void* stream) {
  const bool fp8 = p.kv_dtype == MLA_KV_FP8_E4M3;
  const bool wide = p.rows > 16;  // more than lane quarter 0 holds rows (bf16 only)
  auto kernel = fp8 ? fwd_small_kernel<true, false>
                    : (wide ? fwd_small_kernel<false, true> : fwd_small_kernel<false, false>);
  const int smem = fp8 ? Layout<true>::SMEM_BYTES : Layout<false>::SMEM_BYTES;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  e = mla::opt_in_smem(reinterpret_cast<const void*>(kernel), smem, dev, fp8 ? 4 : (wide ? 5 : 3));
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.units != nullptr ? dim3(2 * p.unit_capacity, 1, 1)
                                  : dim3(2, p.batch, p.num_splits);
  cfg.blockDim = dim3(32 * (wide ? Warps<true>::count : Warps<false>::count), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, kernel, p);
}
