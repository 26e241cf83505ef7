// Batched fp32 GEMM on the tensor cores: C = alpha op(A) op(B) + beta C for every problem of a
// device table, in one persistent launch (the contractions of the second-order optimizers:
// Shampoo's statistics, coupled-Newton roots and preconditioning in fp32 precision, SOAP's
// statistics, Q^T L Q, Rayleigh quotients and its rotations into and out of the eigenbasis).
//
// Precision ("3xTF32" with k-block accumulation).  Each fp32 operand value x is cut into
// hi = x with its 13 low mantissa bits cleared (a TF32 value) and lo = x - hi (exact in fp32);
// tcgen05.mma kind::tf32 forms hi*hi + hi*lo + lo*hi.  The dropped lo*lo term and the TF32
// reading of lo are each below 2^-20 of |x y|.  The tensor core's fp32 accumulation is not
// rounded to nearest: measured on this GPU, accumulating a whole K = 768 product in tensor
// memory left a relative error of 6e-6, ten times an fp32 FFMA GEMM's, growing with K.  So
// each k-block of 32 (12 MMAs) goes into a fresh accumulator, and the epilogue warps add the
// k-block partials in fp32 registers (round to nearest), which keeps the result at an fp32
// GEMM's accuracy.
//
// Structure (one CTA per SM, 512 threads in four warpgroups, registers split by setmaxnreg):
//   warps 0-3    producers (104 registers): copy a 128 x 32 tile of op(A) and a 256 x 32
//                tile of op(B) from global memory with cp.async straight into the
//                128-byte-swizzled K-major layout the MMA reads (an MN-major operand, stored
//                transposed, value by value to its transposed place; zero outside the
//                problem), then split each value in place into hi and lo; two stages of
//                96 KB (A hi, B hi, A lo, B lo), full / empty mbarriers.  A k-block is split
//                as soon as its copies land and the next one's copies go out as soon as its
//                stage is free, so they fly while the MMA works on the other stage.  (In the
//                TMA variant below the tiles arrive by TMA and these warps only split them.)
//   warp 4       lane 0 issues the MMAs (M = 128, N = 256, K = 8; 12 per k-block) into one of
//                two TMEM accumulators (2 x 256 columns), one k-block each, alternating;
//                warps 5-7 idle (32 registers; in the TMA variant warp 5 lane 0 issues the
//                operand loads);
//   warps 8-15   epilogue (176 registers): warp w reads TMEM lanes 32 (w % 4) .. + 31 and
//                columns 128 ((w - 8) / 4) .. + 127 of each k-block partial (tcgen05.ld),
//                adds them into a 128-value running sum per thread, releases the
//                accumulator, and at the end of the tile writes alpha * sum + beta * C (and
//                T = (5 I - C) / 4 where the problem asks for it) with fp32 stores.
// Tiles are visited in one order shared by all roles: problems longest contraction first, a
// problem's tiles row by row; CTA b takes tiles b, b + grid, ...
//
// Every mbarrier wait is bounded (globaltimer): when one runs out the kernel records
// MFSDP_ETIMEOUT in the status word, raises an abort flag that every role polls, waits
// (bounded) for its MMAs in flight, frees its tensor memory and returns.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <type_traits>
#include <vector>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

constexpr int kGM = 128, kGN = 256, kGK = 32;           // tile rows, tile columns, k-block
constexpr int kGStages = 2;
constexpr uint32_t kGATile = kGM * kGK * 4;             // 16 KB
constexpr uint32_t kGBTile = kGN * kGK * 4;             // 32 KB
constexpr uint32_t kGStageBytes = 2 * (kGATile + kGBTile);
constexpr uint32_t kGLoOffset = kGATile + kGBTile;      // stage: [A hi | B hi | A lo | B lo]
constexpr int kGProducers = 128;                        // warpgroup 0
constexpr int kGMmaWarp = 4;                            // warpgroup 1 (warps 5-7 idle)
constexpr int kGEpiWarp0 = 8, kGEpiWarps = 8;           // warpgroups 2 and 3
constexpr int kGThreads = 512;
constexpr uint32_t kGBarOffset = kGStages * kGStageBytes;
constexpr uint32_t kGSmem = 1024 + kGBarOffset + 256;
constexpr uint32_t kGTmemCols = 2 * kGN;
// Registers per thread after setmaxnreg: the four warpgroups together must stay within the
// 512 x 128 the block is launched with (launch_gemm checks the kernel's register count).
constexpr int kGRegsProd = 104, kGRegsMma = 32, kGRegsEpi = 176;
static_assert(128 * kGRegsProd + 128 * kGRegsMma + 256 * kGRegsEpi <= kGThreads * 128,
              "register split");
static_assert(kGRegsMma <= 128 && kGRegsEpi >= 128, "the MMA warpgroup frees, the epilogue takes");
static_assert(kGSmem <= 227 * 1024, "shared memory");

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct GGuard {
  volatile int* abort;
  uint64_t limit_ns;
  int* status;
};

// Wait for the phase of `parity` (bounded, inline: no calls inside setmaxnreg regions); false
// if the kernel is aborting or the wait ran out (which starts the abort).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, const GGuard& g,
                                         bool honor_abort = true) {
  if (bar_try_wait(bar, parity)) return true;
  const uint64_t t0 = timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (bar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (honor_abort && *g.abort) return false;
      if (timer_ns() - t0 > g.limit_ns) {
        atomicOr(g.status, kStatusTimeout);
        *g.abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (+)= A B^T for tf32 operands, A: M x K and B: N x K, both K-major in shared memory.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (waits for the load).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte-swizzled layout: rows
// of 32 fp32 (128 B), 8-row atoms 1024 B apart (stride-dimension offset); start >> 4 at bit
// 0, leading-dimension offset >> 4 at bit 16 (unused by this layout, 16 B), stride offset >> 4
// at bit 32, version 1 at bit 46, swizzle mode 2 (128 B) at bit 61.  The k-step j of 8 tf32
// starts 32 bytes further into the rows.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(16u >> 4) << 16) |
         ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::tf32: fp32 accumulator (dtype 1 at bit 4), TF32 A and B
// (format 2 at bits 7 and 10), both K-major (bits 15, 16 clear), N >> 3 at bit 17, M >> 4 at
// bit 24.
constexpr uint32_t kGIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kGN >> 3) << 17) |
                             ((uint32_t)(kGM >> 4) << 24);

__device__ __forceinline__ void sts128f(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// x = hi + lo: hi = x with its 13 low mantissa bits cleared (a TF32 value), lo = x - hi (exact
// in fp32, below 2^-10 |x|); the MMA reads lo as TF32, losing below 2^-20 |x|.  Two
// instructions per value: the producers' issue slots, not the split's accuracy, are what the
// tile rate needs (non-finite inputs give non-finite results).
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  lo = x - hi;
}

// Byte offset of element (row r, k) of a K-major 32-wide tile in the 128-byte-swizzled
// layout: 16-byte chunk k / 4 of row r stored at chunk (k / 4) ^ (r % 8).
__device__ __forceinline__ uint32_t tile_off(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 2) ^ (r & 7)) & 7) << 4) +
                    (k & 3) * 4);
}


// Split four values and store them as one 16-byte chunk (hi and lo halves) at byte `off`.
__device__ __forceinline__ void store_split4(uint32_t s_hi, uint32_t off, float4 x) {
  float4 h, lo;
  split_tf32(x.x, h.x, lo.x);
  split_tf32(x.y, h.y, lo.y);
  split_tf32(x.z, h.z, lo.z);
  split_tf32(x.w, h.w, lo.w);
  sts128f(s_hi + off, h);
  sts128f(s_hi + kGLoOffset + off, lo);
}

// ---------------------------------------------------------------- asynchronous operand copies
__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src, int bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// ---------------------------------------------------------------- TMA (the TMA variant)
__device__ __forceinline__ void tma_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// Box at (x, y) of a 2D tensor map (x = the innermost coordinate, a multiple of 32 fp32 here)
// into shared memory; completion is counted on the mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128u(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  const uint4 v = lds128u(a);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                     __uint_as_float(v.w));
}
// Copy four consecutive fp32 (`avail` of them inside the operand, the rest zero-filled) from
// global to shared memory with cp.async: one 16-byte copy when the source is 16-byte aligned,
// else four 4-byte copies.
__device__ __forceinline__ void copy4(uint32_t dst, const float* src, int avail,
                                      const float* base) {
  const int bytes = avail >= 4 ? 16 : (avail > 0 ? 4 * avail : 0);
  if (bytes == 0) {
    cp_async16(dst, base, 0);  // nothing read: zero fill
  } else if (aligned16(src)) {
    cp_async16(dst, src, bytes);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) cp_async4(dst + 4 * e, e < avail ? src + e : base, e < avail ? 4 : 0);
  }
}

// One operand tile (R rows x 32 k) of a k-block, moved by the 128 producer threads (p = thread
// index) in two steps.  issue() starts asynchronous copies of the fp32 values straight to their
// places in the stage's lo half (K-major, 128-byte-swizzled; zero outside the problem), so that
// a k-block's loads are in flight while the previous one is converted; convert(), once this
// thread's copies have landed, splits every 16-byte chunk it copied into hi (written to the hi
// half) and lo (written over the raw chunk).  A thread converts exactly the chunks it copied,
// so no other thread's copies are involved.
// K-major source (element (r, k) at src[(row0 + r) * ld + k0 + k]): chunk idx holds row idx / 8,
// k 4 (idx % 8) .. + 3, one 16-byte copy; a quarter warp covers one row (conflict-free).
// MN-major source (element (r, k) at src[(k0 + k) * ld + row0 + r]): a thread takes the 4 x 4
// block of rows 4 rq .. + 3 at k 4 kq .. + 3 (lane l: kq = l % 8, row quad 4 g + l / 8): four
// 16-byte copies, one per k, each landing in one of the block's four final chunk places (k
// 4 kq + i in the place of row 4 rq + i), so that the block occupies exactly the places its
// four rows' chunks end up in; convert() transposes it in registers.  Each quarter warp
// touches 8 distinct bank groups.
template <int R, bool MN>
struct Operand {
  static constexpr int kChunks = R / 16;  // 16-byte chunks per thread per k-block
  static_assert(R * 8 == kChunks * kGProducers, "chunks per thread");

  __device__ __forceinline__ static void issue(const float* src, int64_t ld, int row0, int rows,
                                               int k0, int K, uint32_t s_lo, int p) {
    if (!MN) {
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        const int idx = j * kGProducers + p;
        const int row = row0 + (idx >> 3), kk = k0 + 4 * (idx & 7);
        const uint32_t dst = s_lo + tile_off(idx >> 3, 4 * (idx & 7));
        if (row < rows)
          copy4(dst, src + (int64_t)row * ld + kk, K - kk, src);
        else
          copy4(dst, src, 0, src);
      }
    } else {
#pragma unroll
      for (int b = 0; b < kChunks / 4; ++b) {
        const int bi = b * kGProducers + p, l = bi & 31;
        const int kq = l & 7, rq = 4 * (bi >> 5) + (l >> 3);
        const int row = row0 + 4 * rq;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int kk = k0 + 4 * kq + i;
          const uint32_t dst = s_lo + tile_off(4 * rq + i, 4 * kq);
          if (kk < K)
            copy4(dst, src + (int64_t)kk * ld + row, rows - row, src);
          else
            copy4(dst, src, 0, src);
        }
      }
    }
  }

  __device__ __forceinline__ static void convert(uint32_t s_hi, uint32_t s_lo, int p) {
    if (!MN) {
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        const int idx = j * kGProducers + p;
        const uint32_t off = tile_off(idx >> 3, 4 * (idx & 7));
        store_split4(s_hi, off, lds128f(s_lo + off));  // lo goes over the raw chunk
      }
    } else {
#pragma unroll
      for (int b = 0; b < kChunks / 4; ++b) {
        const int bi = b * kGProducers + p, l = bi & 31;
        const int kq = l & 7, rq = 4 * (bi >> 5) + (l >> 3);
        float4 y[4];  // y[i]: rows 4 rq .. + 3 at k 4 kq + i
#pragma unroll
        for (int i = 0; i < 4; ++i) y[i] = lds128f(s_lo + tile_off(4 * rq + i, 4 * kq));
        store_split4(s_hi, tile_off(4 * rq, 4 * kq), make_float4(y[0].x, y[1].x, y[2].x, y[3].x));
        store_split4(s_hi, tile_off(4 * rq + 1, 4 * kq), make_float4(y[0].y, y[1].y, y[2].y, y[3].y));
        store_split4(s_hi, tile_off(4 * rq + 2, 4 * kq), make_float4(y[0].z, y[1].z, y[2].z, y[3].z));
        store_split4(s_hi, tile_off(4 * rq + 3, 4 * kq), make_float4(y[0].w, y[1].w, y[2].w, y[3].w));
      }
    }
  }
};

// One launch covers up to kGMaxProbs problems.  The host lists them longest contraction first
// (order[]) with the first tile index of each (tile_start[], 128 x 256 tiles numbered row by
// row within a problem); CTA b runs tiles b, b + grid, ... of that sequence, so every CTA takes
// its share of the longest tiles first.
constexpr int kGMaxProbs = 480;
struct GemmLaunch {
  const GemmDesc* descs;
  int32_t nprob, total_tiles;
  uint64_t wait_limit_ns;
  int* status;
  int16_t order[kGMaxProbs];
  int32_t tile_start[kGMaxProbs + 1];
};
static_assert(sizeof(GemmLaunch) <= 4096, "kernel parameter space");

// The TMA variant (both operands K-major, pitches TMA can address): the launch also carries
// each problem's tensor maps, in launch order, for at most kGTmaProbs problems (the kernel
// parameter space holds 32 KB).
constexpr int kGTmaProbs = 64;
struct GemmLaunchTma : GemmLaunch {
  alignas(64) CUtensorMap amap[kGTmaProbs];  // A, m x k: boxes of 32 k x 128 rows
  alignas(64) CUtensorMap bmap[kGTmaProbs];  // B stored n x k: boxes of 32 k x 256 rows
};
static_assert(sizeof(GemmLaunchTma) <= 32000, "kernel parameter space");

// Walks the tiles of one CTA in the launch order: next() moves to tile t (increasing) and
// yields its problem and origin.
struct TileCursor {
  int pos = 0;
  __device__ __forceinline__ void at(const GemmLaunch& P, int t, GemmDesc& d, int& m0,
                                     int& n0) {
    while (P.tile_start[pos + 1] <= t) ++pos;
    d = P.descs[P.order[pos]];
    const int local = t - P.tile_start[pos];
    const int tiles_n = (d.n + kGN - 1) / kGN;
    m0 = (local / tiles_n) * kGM;
    n0 = (local % tiles_n) * kGN;
  }
};

// op(A) is m x k: A stored m x k (TA = 0, K-major) or k x m (TA = 1, MN-major).  op(B) is
// k x n: B stored k x n (TB = 0, MN-major for the MMA's N x K operand) or n x k (TB = 1).
//
// TMA = true (TA = 0, TB = 1 only): one thread of the MMA warpgroup (warp 5) loads each
// k-block's raw fp32 tiles by TMA straight into the lo halves (the same 128-byte-swizzled
// K-major layout) and the producer warps only split them: they wait for the tiles to land,
// split in place and hand the stage to the MMA.  The cp.async producers spend most of their
// issue slots on copy addresses; here that work is the TMA unit's.
template <int TA, int TB, bool TMA>
__global__ void __launch_bounds__(kGThreads, 1)
    tf32x3_gemm_kernel(const __grid_constant__ std::conditional_t<TMA, GemmLaunchTma, GemmLaunch> P) {
  static_assert(!TMA || (TA == 0 && TB == 1), "the TMA variant reads both operands K-major");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGBarOffset);
  // bars: full[2] | empty[2] | tfull[2] | tempty[2] | drain | landed[2] (TMA tiles arrived)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_addr(bars + i); };
  constexpr int full0 = 0, empty0 = 2, tfull0 = 4, tempty0 = 6, drain = 8, landed0 = 9;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      bar_init(bar(full0 + s), kGProducers / 32);
      bar_init(bar(empty0 + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      bar_init(bar(tfull0 + a), 1);
      bar_init(bar(tempty0 + a), kGEpiWarps);
    }
    bar_init(bar(drain), 1);
    bar_init(bar(landed0), 1);
    bar_init(bar(landed0 + 1), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kGMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kGTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const GGuard g{abort_flag, P.wait_limit_ns, P.status};

  if (warp < 4) {
    // ------------------------------------------------------------ producers (warpgroup 0)
    // .dec may only lower the count and .inc only raise it (an illegal instruction otherwise)
    if constexpr (kGRegsProd > 128)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGRegsProd));
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGRegsProd));
    const int p = threadIdx.x;
    // k-block j - 1 is split as soon as its copies land (its stage was free when they were
    // issued), which can be while the MMA still works on k-block j - 2; then the producers
    // wait for the stage of k-block j (freed by k-block j - 2) and issue its copies, which fly
    // while the MMA works on k-block j - 1
    uint32_t j = 0;            // k-blocks issued so far (sequence over this CTA's tiles)
    TileCursor cur;
    bool ok = true;
    if constexpr (TMA) {
      // the tiles of k-block j arrive by TMA (landed[j % 2]); split them and hand them on
      for (int t = blockIdx.x; t < P.total_tiles && ok; t += gridDim.x) {
        GemmDesc d;
        int m0, n0;
        cur.at(P, t, d, m0, n0);
        const int nk = (d.k + kGK - 1) / kGK;
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int stage = (int)(j & 1u);
          if (!bar_wait(bar(landed0 + stage), (j >> 1) & 1u, g)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + (uint32_t)stage * kGStageBytes;
          Operand<kGM, false>::convert(sa, sa + kGLoOffset, p);
          Operand<kGN, false>::convert(sa + kGATile, sa + kGATile + kGLoOffset, p);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
          __syncwarp();
          if (lane == 0) bar_arrive(bar(full0 + stage));
        }
      }
    } else {
      auto finish = [&](uint32_t jj) {  // convert k-block jj and hand its stage to the MMA
        const uint32_t sa = sbase + (jj & 1u) * kGStageBytes;
        Operand<kGM, TA == 1>::convert(sa, sa + kGLoOffset, p);
        Operand<kGN, TB == 0>::convert(sa + kGATile, sa + kGATile + kGLoOffset, p);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
        __syncwarp();
        if (lane == 0) bar_arrive(bar(full0 + (int)(jj & 1u)));
      };
      for (int t = blockIdx.x; t < P.total_tiles && ok; t += gridDim.x) {
        GemmDesc d;
        int m0, n0;
        cur.at(P, t, d, m0, n0);
        const int nk = (d.k + kGK - 1) / kGK;
        for (int kb = 0; kb < nk; ++kb, ++j) {
          const int stage = (int)(j & 1u);
          if (j > 0) {
            cp_async_wait<0>();  // this thread's copies of k-block j - 1 have landed
            finish(j - 1);
          }
          if (*abort_flag || !bar_wait(bar(empty0 + stage), ((j >> 1) & 1u) ^ 1u, g)) {
            ok = false;
            break;
          }
          const uint32_t sa = sbase + (uint32_t)stage * kGStageBytes;
          Operand<kGM, TA == 1>::issue(d.a, d.lda, m0, d.m, kb * kGK, d.k, sa + kGLoOffset, p);
          Operand<kGN, TB == 0>::issue(d.b, d.ldb, n0, d.n, kb * kGK, d.k,
                                       sa + kGATile + kGLoOffset, p);
          cp_async_commit();
        }
      }
      cp_async_wait<0>();
      if (ok && j > 0) finish(j - 1);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ MMA issuer (warpgroup 1)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kGRegsMma));
    if (warp == kGMmaWarp && lane == 0) {
      uint32_t q = 0, c = 0;  // k-block (stage) and accumulator sequence numbers
      bool ok = true;
      TileCursor cur;
      for (int t = blockIdx.x; t < P.total_tiles && ok; t += gridDim.x) {
        GemmDesc d;
        int m0, n0;
        cur.at(P, t, d, m0, n0);
        const int nk = (d.k + kGK - 1) / kGK;
        for (int kb = 0; kb < nk; ++kb, ++q, ++c) {
          const int acc = (int)(c & 1u), stage = (int)(q & 1u);
          if (!bar_wait(bar(tempty0 + acc), ((c >> 1) & 1u) ^ 1u, g) ||
              !bar_wait(bar(full0 + stage), (q >> 1) & 1u, g)) {
            ok = false;
            break;
          }
          fence_after();
          const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kGN);
          const uint32_t sa = sbase + (uint32_t)stage * kGStageBytes, sb = sa + kGATile;
#pragma unroll
          for (int j = 0; j < kGK / 8; ++j) {
            const uint64_t ah = kmajor_desc(sa + 32u * j), bh = kmajor_desc(sb + 32u * j);
            const uint64_t al = kmajor_desc(sa + kGLoOffset + 32u * j);
            const uint64_t bl = kmajor_desc(sb + kGLoOffset + 32u * j);
            mma_tf32(d_tmem, ah, bh, kGIdesc, j != 0);
            mma_tf32(d_tmem, ah, bl, kGIdesc, 1u);
            mma_tf32(d_tmem, al, bh, kGIdesc, 1u);
          }
          mma_commit(bar(empty0 + stage));
          mma_commit(bar(tfull0 + acc));
        }
      }
      mma_commit(bar(drain));
      bar_wait(bar(drain), 0u, g, false);  // every MMA of this CTA has completed
    }
    if constexpr (TMA) {
      if (warp == kGMmaWarp + 1 && lane == 0) {
        // ---------------------------------------------------------- TMA loads (warp 5)
        uint32_t j = 0, armed = 0, last_par = 0;
        bool ok = true;
        TileCursor cur;
        for (int t = blockIdx.x; t < P.total_tiles && ok; t += gridDim.x) {
          GemmDesc d;
          int m0, n0;
          cur.at(P, t, d, m0, n0);
          const CUtensorMap* am = &P.amap[cur.pos];
          const CUtensorMap* bm = &P.bmap[cur.pos];
          const int nk = (d.k + kGK - 1) / kGK;
          for (int kb = 0; kb < nk; ++kb, ++j) {
            const int stage = (int)(j & 1u);
            if (!bar_wait(bar(empty0 + stage), ((j >> 1) & 1u) ^ 1u, g)) {
              ok = false;
              break;
            }
            const uint32_t sa = sbase + (uint32_t)stage * kGStageBytes;
            const uint32_t lb = bar(landed0 + stage);
            tma_expect_tx(lb, kGATile + kGBTile);
            tma_load_2d(sa + kGLoOffset, am, kb * kGK, m0, lb);
            tma_load_2d(sa + kGATile + kGLoOffset, bm, kb * kGK, n0, lb);
            armed |= 1u << stage;
            last_par = (last_par & ~(1u << stage)) | (((j >> 1) & 1u) << stage);
          }
        }
        // loads in flight when the kernel gives up must land before the CTA leaves
        if (!ok)
          for (int st = 0; st < 2; ++st)
            if (armed & (1u << st)) bar_wait(bar(landed0 + st), (last_par >> st) & 1u, g, false);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warpgroups 2, 3)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kGRegsEpi));
    const int quarter = warp & 3;              // TMEM lanes 32 * quarter .. + 31
    const int half = (warp - kGEpiWarp0) >> 2;  // columns 128 * half .. + 127
    uint32_t c = 0;
    bool ok = true;
    TileCursor cur;
    for (int t = blockIdx.x; t < P.total_tiles && ok; t += gridDim.x) {
      GemmDesc d;
      int m0, n0;
      cur.at(P, t, d, m0, n0);
      const int nk = (d.k + kGK - 1) / kGK;
      float s[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) s[j] = 0.f;
      for (int kb = 0; kb < nk; ++kb, ++c) {
        const int acc = (int)(c & 1u);
        if (!bar_wait(bar(tfull0 + acc), (c >> 1) & 1u, g)) {
          ok = false;
          break;
        }
        fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) +
                               (uint32_t)(acc * kGN + 128 * half);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float a[16];
          tmem_ld16(taddr + (uint32_t)(16 * cc), a);
#pragma unroll
          for (int j = 0; j < 16; ++j) s[16 * cc + j] += a[j];
        }
        fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(bar(tempty0 + acc));
      }
      if (!ok) break;
      const int r = m0 + 32 * quarter + lane;
      const int c0 = n0 + 128 * half;
      if (r >= d.m || c0 >= d.n) continue;
      float* cp = d.c + (int64_t)r * d.ldc + c0;
      float* tp = d.t_out ? d.t_out + (int64_t)r * d.ldc + c0 : nullptr;
      if (c0 + 128 <= d.n && aligned16(cp) && (!tp || aligned16(tp))) {
#pragma unroll
        for (int q4 = 0; q4 < 32; ++q4) {
          float4 o = make_float4(d.alpha * s[4 * q4], d.alpha * s[4 * q4 + 1],
                                 d.alpha * s[4 * q4 + 2], d.alpha * s[4 * q4 + 3]);
          if (d.beta != 0.f) {
            const float4 cv = *reinterpret_cast<const float4*>(cp + 4 * q4);
            o.x = fmaf(d.beta, cv.x, o.x);
            o.y = fmaf(d.beta, cv.y, o.y);
            o.z = fmaf(d.beta, cv.z, o.z);
            o.w = fmaf(d.beta, cv.w, o.w);
          }
          *reinterpret_cast<float4*>(cp + 4 * q4) = o;
          if (tp) {
            const int cl = c0 + 4 * q4;
            *reinterpret_cast<float4*>(tp + 4 * q4) =
                make_float4(((r == cl ? 5.f : 0.f) - o.x) * 0.25f,
                            ((r == cl + 1 ? 5.f : 0.f) - o.y) * 0.25f,
                            ((r == cl + 2 ? 5.f : 0.f) - o.z) * 0.25f,
                            ((r == cl + 3 ? 5.f : 0.f) - o.w) * 0.25f);
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 128; ++j) {
          const int cl = c0 + j;
          if (cl < d.n) {
            float o = d.alpha * s[j];
            if (d.beta != 0.f) o = fmaf(d.beta, cp[j], o);
            cp[j] = o;
            if (tp) tp[j] = ((r == cl ? 5.f : 0.f) - o) * 0.25f;
          }
        }
      }
    }
  }

  fence_before();
  __syncthreads();
  if (warp == kGMmaWarp) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kGTmemCols)
                 : "memory");
  }
}

template <int TA, int TB, bool TMA>
cudaError_t launch_one(const std::conditional_t<TMA, GemmLaunchTma, GemmLaunch>& p, int grid,
                       cudaStream_t st) {
  static int attr_set[64] = {};  // per device: the dynamic shared-memory limit was raised
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    // setmaxnreg.inc draws on the registers the block was launched with: a kernel built with
    // fewer than the split needs would wait forever in it, so it is refused here instead
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, tf32x3_gemm_kernel<TA, TB, TMA>);
    if (e != cudaSuccess) return e;
    if ((int64_t)fa.numRegs * kGThreads < 128 * kGRegsProd + 128 * kGRegsMma + 256 * kGRegsEpi)
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(tf32x3_gemm_kernel<TA, TB, TMA>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = 1;
  }
  tf32x3_gemm_kernel<TA, TB, TMA><<<(unsigned)grid, kGThreads, kGSmem, st>>>(p);
  return cudaGetLastError();
}

// Whether the TMA variant can read this problem: both operands K-major (A m x k, B n x k),
// 16-byte aligned bases and pitches that are multiples of 4 floats.
bool tma_ok(const GemmDesc& d) {
  auto al = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  return d.k > 0 && al(d.a) && al(d.b) && d.lda % 4 == 0 && d.ldb % 4 == 0 && d.lda >= d.k &&
         d.ldb >= d.k;
}

}  // namespace

int launch_gemm(const GemmDesc* dev_descs, const GemmDesc* host_descs, int nprob, int ta,
                int tb, cudaStream_t st) {
  if (nprob <= 0) return MFSDP_OK;
  if (!dev_descs || !host_descs || nprob > 32767) return MFSDP_EINVAL;
  int* status = status_word_address();
  if (!status) return MFSDP_ECUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MFSDP_ECUDA;
  // problems with work, longest contraction first (ties: table order)
  std::vector<int> order;
  for (int z = 0; z < nprob; ++z)
    if (host_descs[z].m > 0 && host_descs[z].n > 0) order.push_back(z);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return host_descs[a].k > host_descs[b].k; });
  bool tma = ta == 0 && tb == 1;
  for (int z : order) tma = tma && tma_ok(host_descs[z]);
  const size_t per_launch = tma ? (size_t)kGTmaProbs : (size_t)kGMaxProbs;
  for (size_t first = 0; first < order.size(); first += per_launch) {
    const size_t cnt = std::min(order.size() - first, per_launch);
    GemmLaunchTma p{};
    p.descs = dev_descs;
    p.nprob = (int32_t)cnt;
    p.wait_limit_ns = wait_limit_ns();
    p.status = status;
    int64_t tiles = 0;
    for (size_t j = 0; j < cnt; ++j) {
      const GemmDesc& d = host_descs[order[first + j]];
      p.order[j] = (int16_t)order[first + j];
      p.tile_start[j] = (int32_t)tiles;
      tiles += (int64_t)((d.m + kGM - 1) / kGM) * ((d.n + kGN - 1) / kGN);
    }
    if (tiles > INT32_MAX) return MFSDP_ESHAPE;
    p.tile_start[cnt] = (int32_t)tiles;
    for (size_t j = cnt; j < (size_t)kGMaxProbs; ++j) p.tile_start[j + 1] = (int32_t)tiles;
    p.total_tiles = (int32_t)tiles;
    const int grid = (int)std::min<int64_t>(tiles, sms);
    cudaError_t e;
    if (tma) {
      for (size_t j = 0; j < cnt; ++j) {
        const GemmDesc& d = host_descs[order[first + j]];
        if (!encode_map_f32(&p.amap[j], d.a, d.m, d.k, d.lda, kGM) ||
            !encode_map_f32(&p.bmap[j], d.b, d.n, d.k, d.ldb, kGN))
          return MFSDP_ECUDA;
      }
      e = launch_one<0, 1, true>(p, grid, st);
    } else {
      const GemmLaunch& q = p;
      if (ta == 0 && tb == 0) e = launch_one<0, 0, false>(q, grid, st);
      else if (ta == 0 && tb == 1) e = launch_one<0, 1, false>(q, grid, st);
      else if (ta == 1 && tb == 0) e = launch_one<1, 0, false>(q, grid, st);
      else e = launch_one<1, 1, false>(q, grid, st);
    }
    if (e != cudaSuccess) return MFSDP_ECUDA;
  }
  return MFSDP_OK;
}

}  // namespace mfsdp

using namespace mfsdp;

extern "C" size_t mfsdp_gemm_f32_workspace_bytes(int32_t n_probs) {
  return n_probs > 0 ? (size_t)n_probs * sizeof(GemmDesc) : 0;
}

extern "C" int mfsdp_gemm_f32_batched(const mfsdp_gemm_problem* probs, int32_t n_probs,
                                      int32_t trans_a, int32_t trans_b, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (n_probs < 0 || (n_probs > 0 && !probs)) return MFSDP_EINVAL;
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return MFSDP_EINVAL;
  std::vector<GemmDesc> descs;
  for (int32_t i = 0; i < n_probs; ++i) {
    const mfsdp_gemm_problem& q = probs[i];
    if (q.m < 0 || q.n < 0 || q.k < 0) return MFSDP_EINVAL;
    if (q.m == 0 || q.n == 0) continue;
    if (!q.c || q.ldc < q.n) return MFSDP_EINVAL;
    if (q.k > 0) {
      if (!q.a || !q.b) return MFSDP_EINVAL;
      if (q.lda < (trans_a ? q.m : q.k) || q.ldb < (trans_b ? q.k : q.n)) return MFSDP_EINVAL;
    }
    GemmDesc d{};
    d.a = q.a;
    d.b = q.b;
    d.c = q.c;
    d.t_out = nullptr;
    d.m = q.m;
    d.n = q.n;
    d.k = q.k;
    d.lda = q.lda;
    d.ldb = q.ldb;
    d.ldc = q.ldc;
    d.alpha = q.alpha;
    d.beta = q.beta;
    descs.push_back(d);
  }
  if (descs.empty()) return MFSDP_OK;
  if (!workspace || workspace_bytes < mfsdp_gemm_f32_workspace_bytes(n_probs) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the table is staged out of pageable host memory before cudaMemcpyAsync returns
  if (cudaMemcpyAsync(workspace, descs.data(), descs.size() * sizeof(GemmDesc),
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MFSDP_ECUDA;
  return launch_gemm(static_cast<const GemmDesc*>(workspace), descs.data(), (int)descs.size(),
                     trans_a, trans_b, st);
}
