// Newton–Schulz phases as one persistent, grouped tcgen05 GEMM launch per phase.
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §2: Muon
// orthogonalises each whole 2D matrix with Newton–Schulz steps whose products include X X^T.
// One quintic iteration, X of shape m x n with m <= n, is X' = a X + B X with A = X X^T and
// B = b A + c A A.  It runs as three products; with bf16 operands the a X term is folded into
// the second one (a X + B X = (a I + B) X):
//     gram  A  = X X^T                  (m x m, K = n, symmetric: upper-triangle tiles only)
//     poly  B' = a*I + b*A + c*A A      (m x m, K = m, symmetric: upper-triangle tiles only)
//     apply X' = B' X                   (m x n, K = m, no addend)
// so that only the polynomial phase reads an addend (A, m x m) and the apply phase, the
// largest small-K product, streams nothing but its operands.  Split (hi + lo) operands keep
// poly B = b*A + c*A A and apply X' = a*X + B X: there B is held to ~2^-17 of its own size,
// which for directions with small singular values is much finer than 2^-17 of a I + B.
// A launch runs one phase for every owned matrix: a static list of 128 x 256 output tiles,
// taken round-robin by a persistent grid of one CTA per SM.
//
// CTA roles (320 threads):
//   warp 0             TMA producers, one lane per pipeline stage: 64-wide, 128-byte-swizzled
//                      bf16 boxes into a ring of stages guarded by full/empty mbarriers;
//   warp 1 (one lane)  MMA issuer: tcgen05.mma kind::f16 (M=128, N=256, K=16) from shared-
//                      memory descriptors into one of two TMEM accumulators (2 x 256 columns);
//   warps 2-9          epilogue: tcgen05.ld rows of the accumulator, out = alpha*acc + beta*D
//                      (+ a on the diagonal in a folded polynomial phase), round to bf16 (and the
//                      low half in split mode), store; symmetric tiles store the upper triangle
//                      and its mirror.
// Operands come from row-major bf16 buffers.  A "K-major" operand has the contraction index
// contiguous (rows of X for X X^T); an "MN-major" operand has the output index contiguous
// (X as the right factor of B X).  Both map to the canonical 128-byte-swizzled UMMA layouts.
//
// Every mbarrier wait is bounded (globaltimer): when a wait runs out the kernel records the
// timeout in the status word, raises an abort flag every role polls, waits (bounded) for its
// own TMA loads and MMAs in flight, frees its tensor memory and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

constexpr uint32_t kBoxBytes = 64 * 64 * 2;               // one 64 x 64 bf16 TMA box
constexpr uint32_t kABytes = kBM * kBK * 2;               // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;               // 32 KB
constexpr uint32_t kTmemCols = 2 * kBN;                   // two fp32 accumulators
constexpr int kEpiWarps = (kNsThreads / 32) - 2;          // epilogue warps: 2 per lane quarter
constexpr int kEpiChunks = (kBN / 32) / (kEpiWarps / 4);  // 32-column chunks per epilogue warp
static_assert(kEpiWarps == 8 && kEpiChunks == 4, "epilogue layout");

template <bool SPLIT>
struct Cfg {
  static constexpr int kOps = SPLIT ? 2 : 1;              // hi (+ lo) operand copies
  static constexpr int kStages = SPLIT ? 2 : 4;
  static constexpr uint32_t kStageBytes = kOps * (kABytes + kBBytes);
  static constexpr uint32_t kBarOffset = kStages * kStageBytes;
  static constexpr uint32_t kSmem = 1024 + kBarOffset + 256;
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

struct Guard {                 // shared abort flag + the launch's wait limit
  volatile int* abort;
  uint64_t limit_ns;
  int* status;
};

__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const Guard& g,
                                            bool honor_abort) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (honor_abort && *g.abort) return false;
      if (globaltimer() - t0 > g.limit_ns) {
        atomicOr(g.status, kStatusTimeout);
        *g.abort = 1;
        return false;
      }
    }
  }
}

// Wait for the phase of `parity` to complete (CTA-scope acquire): inline fast path, bounded slow
// path.  Returns false if the kernel is aborting or the wait ran out (which starts the abort).
// `honor_abort` = false is used during teardown.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Guard& g,
                                          bool honor_abort = true) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, g, honor_abort);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane; waits for the load to land.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 layout: start >> 4 at bit 0,
// leading-dimension byte offset >> 4 at bit 16, stride-dimension byte offset >> 4 at bit 32,
// version 1 at bit 46, swizzle mode 2 = 128B at bit 61).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// K-major operand: rows of 64 k-values (128 B), 8-row swizzle atoms 1024 B apart; the k-step
// j of 16 elements starts 32 bytes further.  MN-major operand: 64-wide output-index chunks
// (one box each, 8 KB apart), 8 k-rows of 128 B per atom; k-step j starts 16 rows further.
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int mn_major, int j) {
  return mn_major ? smem_desc(base + (uint32_t)j * 2048u, kBoxBytes, 1024u)
                  : smem_desc(base + (uint32_t)j * 32u, 16u, 1024u);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bit 4), bf16 A (bits 7-9) and B
// (bits 10-12), A / B major-ness (bits 15 / 16), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__device__ __forceinline__ uint32_t make_idesc(int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}


__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t f2bf(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
// Two floats rounded to nearest-even bf16 in one conversion: lo in bits 0-15, hi in 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 consecutive bf16 of row r starting at column c0 (c0 % 8 == 0, pitch % 8 == 0) as fp32.
__device__ __forceinline__ void load_row32(const uint16_t* p, int64_t ld, int r, int c0, int N,
                                           float (&d)[32]) {
  const uint16_t* row = p + (int64_t)r * ld + c0;
  if (c0 + 32 <= N) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + 8 * q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        d[8 * q + 2 * k] = bf_lo(w[k]);
        d[8 * q + 2 * k + 1] = bf_hi(w[k]);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) d[j] = (c0 + j < N) ? bf2f(row[j]) : 0.f;
  }
}

__device__ __forceinline__ void store_row32(uint16_t* p, int64_t ld, int r, int c0, int cmin,
                                            int N, const uint16_t (&h)[32]) {
  uint16_t* row = p + (int64_t)r * ld + c0;
  if (cmin <= c0 && c0 + 32 <= N) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 v;
      v.x = (uint32_t)h[8 * q + 0] | ((uint32_t)h[8 * q + 1] << 16);
      v.y = (uint32_t)h[8 * q + 2] | ((uint32_t)h[8 * q + 3] << 16);
      v.z = (uint32_t)h[8 * q + 4] | ((uint32_t)h[8 * q + 5] << 16);
      v.w = (uint32_t)h[8 * q + 6] | ((uint32_t)h[8 * q + 7] << 16);
      *reinterpret_cast<uint4*>(row + 8 * q) = v;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (c0 + j >= cmin && c0 + j < N) row[j] = h[j];
  }
}


// ---------------------------------------------------------------- multi-lane TMA producers
// A thread's TMA loads run one after another (a 64 x 128 box costs a thread ~600-750 cycles,
// whatever the pipeline depth), so one issuing thread cannot feed the tensor cores.  The
// producer warp therefore runs one issuer per pipeline stage: lane l owns stage l, and the
// lanes step through the k-block sequence in lockstep, each round issuing a fixed sequence of
// predicated TMA instructions (operand major-ness only changes which predicates are on).

// The table fields of one tile that the pair kernel's producer and MMA roles use, copied into
// registers.  The roles read them a tile ahead (from a tile row read two tiles ahead) and
// only use them a tile later, so no instruction waits for these loads inside the k-block loop.
struct TileFields {
  int K, a_mn, b_mn, sym, map_a, map_b, mn3d, tm, tn;
  __device__ __forceinline__ int nk() const { return (K + kBK - 1) / kBK; }
  // A tile (256-row blocks) on the diagonal of a symmetric product whose two operands are the
  // same rows of the same buffer (Gram: X X^T; polynomial: A A): each CTA's B half then holds
  // exactly its A half, so only A is loaded and the MMA reads it twice.
  __device__ __forceinline__ bool self() const {
    return sym && tm * 256 == tn * kBN && map_a == map_b && a_mn == b_mn;
  }
};
__device__ __forceinline__ NsTile tile_row(const NsLaunchParams& P, int t) {
  return t < P.ntiles ? P.tiles[t] : NsTile{0, 0, 0, 0};
}
__device__ __forceinline__ TileFields tile_fields(const NsLaunchParams& P, int t,
                                                  const NsTile& row) {
  TileFields f{0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (t >= P.ntiles) return f;
  const NsProblem& pr = P.probs[row.prob];
  f.K = pr.K;
  f.a_mn = pr.a_mn;
  f.b_mn = pr.b_mn;
  f.sym = pr.sym;
  f.map_a = pr.map_a;
  f.map_b = pr.map_b;
  f.mn3d = pr.mn3d;
  f.tm = row.tm;
  f.tn = row.tn;
  return f;
}

// Position in the k-block sequence of the tiles t0, t0 + step, ...
struct KCursor {
  int t, kb;
  __device__ __forceinline__ void norm(const NsLaunchParams& P, int step) {
    while (t < P.ntiles) {
      const int nk = (P.probs[P.tiles[t].prob].K + kBK - 1) / kBK;
      if (kb < nk) break;
      kb -= nk;
      t += step;
    }
  }
};

__device__ __forceinline__ void tma_load_p(bool p, uint32_t dst, const CUtensorMap* map, int x,
                                           int y, uint32_t bar) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %5, 0;\n"
      " @p cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n}\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "r"((uint32_t)p)
      : "memory");
}

__device__ __forceinline__ void expect_tx_p(bool p, uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n"
      " @p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}\n" ::"r"(bar),
      "r"(bytes), "r"((uint32_t)p)
      : "memory");
}

// `rows` rows (128 or 256) of one operand tile: MN-major as 64-wide boxes (map), K-major as
// 128-row boxes (map + 1); the same predicated instructions run in every lane.
template <int ROWS>
__device__ __forceinline__ void issue_operand_p(bool p, uint32_t dst, const CUtensorMap* map,
                                                int mn, int r0, int k0, uint32_t bar) {
#pragma unroll
  for (int c = 0; c < ROWS / 64; ++c) {
    tma_load_p(p && mn, dst + (uint32_t)c * kBoxBytes, map, r0 + 64 * c, k0, bar);
    if (c < ROWS / 128)
      tma_load_p(p && !mn, dst + (uint32_t)c * 2 * kBoxBytes, map + 1, k0, r0 + 128 * c, bar);
  }
}

// ---------------------------------------------------------------- the kernel
template <bool SPLIT>
__global__ void __launch_bounds__(kNsThreads, 1) ns_gemm_kernel(const __grid_constant__ NsLaunchParams P) {
  using C = Cfg<SPLIT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  // the next phase may launch now: its CTAs take SMs as ours leave and stop in
  // griddepcontrol.wait until this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  // bars: full[S] | empty[S] | tfull[2] | tempty[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int full0 = 0, empty0 = S, tfull0 = 2 * S, tempty0 = 2 * S + 2, drain = 2 * S + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(full0 + s), 1);
      mbar_init(bar(empty0 + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(tfull0 + a), 1);
      mbar_init(bar(tempty0 + a), kEpiWarps);
    }
    mbar_init(bar(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // everything above touched only this CTA's shared and tensor memory; from here on the
  // previous phase's outputs are read
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t tmem_base = *tmem_slot;
  const Guard g{abort_flag, P.wait_limit_ns, P.status};

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers (lane = stage)
    if (lane < S) {
      const unsigned pmask = (1u << S) - 1u;
      KCursor cur{(int)blockIdx.x, lane};
      cur.norm(P, gridDim.x);
      uint32_t q = (uint32_t)lane;  // position in the k-block sequence; stage = q % S = lane
      bool armed = false;
      uint32_t last_par = 0;
      const uint32_t sb = sbase + (uint32_t)lane * C::kStageBytes;
      const uint32_t fb = bar(full0 + lane);
      for (;;) {
        bool act = cur.t < P.ntiles && !*abort_flag;
        if (!__any_sync(pmask, act)) break;
        const uint32_t ph = (q / S) & 1u;
        if (act && !mbar_wait(bar(empty0 + lane), ph ^ 1u, g)) act = false;
        const CUtensorMap* ma = P.maps;
        const CUtensorMap* mb = P.maps;
        int a_mn = 0, b_mn = 0, m0 = 0, n0 = 0, k0 = 0;
        if (act) {
          const NsTile tile = P.tiles[cur.t];
          const NsProblem& pr = P.probs[tile.prob];
          ma = P.maps + pr.map_a;
          mb = P.maps + pr.map_b;
          a_mn = pr.a_mn;
          b_mn = pr.b_mn;
          m0 = tile.tm * kBM;
          n0 = tile.tn * kBN;
          k0 = cur.kb * kBK;
          if (cur.kb == 0) {
            prefetch_map(ma + (a_mn ? 0 : 1));
            prefetch_map(mb + (b_mn ? 0 : 1));
          }
        }
        expect_tx_p(act, fb, C::kStageBytes);
        issue_operand_p<kBM>(act, sb, ma, a_mn, m0, k0, fb);
        issue_operand_p<kBN>(act, sb + kABytes, mb, b_mn, n0, k0, fb);
        if (SPLIT) {
          issue_operand_p<kBM>(act, sb + kABytes + kBBytes, ma + kMapsPerHalf, a_mn, m0, k0, fb);
          issue_operand_p<kBN>(act, sb + 2 * kABytes + kBBytes, mb + kMapsPerHalf, b_mn, n0, k0, fb);
        }
        if (act) {
          armed = true;
          last_par = ph;
        }
        q += S;
        cur.kb += S;
        cur.norm(P, gridDim.x);
      }
      // teardown: every load this lane issued has landed before the CTA may exit
      if (armed) mbar_wait(bar(full0 + lane), last_par, g, false);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
      const NsTile tile = P.tiles[t];
      const NsProblem& pr = P.probs[tile.prob];
      const int nk = (pr.K + kBK - 1) / kBK;
      const int a_mn = pr.a_mn, b_mn = pr.b_mn;
      const uint32_t idesc = make_idesc(a_mn, b_mn);
      if (!mbar_wait(bar(tempty0 + acc), acc_phase ^ 1u, g)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(bar(full0 + stage), phase, g)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = sbase + (uint32_t)stage * C::kStageBytes;
        const uint32_t sbb = sa + kABytes;
#pragma unroll
        for (int j = 0; j < kBK / 16; ++j) {
          const uint64_t ad = operand_desc(sa, a_mn, j);
          const uint64_t bd = operand_desc(sbb, b_mn, j);
          tc_mma(d_tmem, ad, bd, idesc, (kb | j) != 0);
          if (SPLIT) {
            const uint64_t adl = operand_desc(sa + kABytes + kBBytes, a_mn, j);
            const uint64_t bdl = operand_desc(sbb + kABytes + kBBytes, b_mn, j);
            tc_mma(d_tmem, ad, bdl, idesc, 1u);   // hi * lo
            tc_mma(d_tmem, adl, bd, idesc, 1u);   // lo * hi
          }
        }
        tc_commit(bar(empty0 + stage));  // frees the stage once these MMAs have read it
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit(bar(tfull0 + acc));      // accumulator ready for the epilogue
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    // teardown: all MMAs issued by this thread have completed
    tc_commit(bar(drain));
    mbar_wait(bar(drain), 0u, g, false);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // Two warps per TMEM lane quarter: warps 2-5 take columns 0-127 of the tile, warps 6-9
    // columns 128-255.  The addend rows D of a tile are loaded into registers before the wait
    // for its accumulator, so their latency overlaps the tile's main loop.
    const int quarter = warp & 3;             // TMEM lanes 32*quarter .. +31 are this warp's rows
    const int c_first = ((warp - 2) >> 2) * kEpiChunks;  // first 32-column chunk of this warp
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < P.ntiles; t += gridDim.x) {
      const NsTile tile = P.tiles[t];
      const NsProblem& pr = P.probs[tile.prob];
      const int M = pr.M, N = pr.N, kind = pr.kind, sym = pr.sym;
      const int m0 = tile.tm * kBM, n0 = tile.tn * kBN;
      const int rw = m0 + quarter * 32;  // first row of this warp
      const int r = rw + lane;
      const bool rvalid = r < M;
      const float s = 1.f / (P.norm[pr.mat] + P.eps);
      uint4 dpre[kEpiChunks][4];
      if (!SPLIT && (kind == kPoly || (kind == kApply && !pr.fold_a)) && rvalid) {
#pragma unroll
        for (int q = 0; q < kEpiChunks; ++q) {
          const int c0 = n0 + (c_first + q) * 32;
          if (c0 + 32 <= N && !(sym && c0 + 31 < rw)) {
            const uint4* src = reinterpret_cast<const uint4*>(pr.d_hi + (int64_t)r * pr.ldd + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k) dpre[q][k] = src[k];
          }
        }
      }
      if (!mbar_wait(bar(tfull0 + acc), acc_phase, g)) break;
      tc_fence_after();
      float alpha = 1.f, beta = 0.f;
      if (kind == kGram) {
        alpha = pr.first ? s * s : 1.f;
      } else if (kind == kPoly) {
        alpha = P.c;
        beta = P.b;
      } else {
        alpha = pr.first ? s : 1.f;
        if (!pr.fold_a) beta = P.a * alpha;
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll
      for (int q = 0; q < kEpiChunks; ++q) {
        const int cc = c_first + q;
        const int c0 = n0 + cc * 32;
        if (c0 >= N || rw >= M) break;                 // warp-uniform
        if (sym && c0 + 31 < rw) continue;             // chunk entirely below the diagonal
        float v[32];
        tc_ld32(taddr + (uint32_t)(cc * 32), v);
        if (!rvalid) continue;
        if (beta != 0.f) {
          float d[32];
          if (!SPLIT && c0 + 32 <= N) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t w[4] = {dpre[q][k].x, dpre[q][k].y, dpre[q][k].z, dpre[q][k].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                d[8 * k + 2 * e] = bf_lo(w[e]);
                d[8 * k + 2 * e + 1] = bf_hi(w[e]);
              }
            }
          } else {
            load_row32(pr.d_hi, pr.ldd, r, c0, N, d);
            if (SPLIT) {
              float dl[32];
              load_row32(pr.d_lo, pr.ldd, r, c0, N, dl);
#pragma unroll
              for (int j = 0; j < 32; ++j) d[j] += dl[j];
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = fmaf(alpha, v[j], beta * d[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
        }
        if (kind == kPoly && pr.fold_a && c0 == rw) {  // a on the diagonal: column `lane`
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == lane) v[j] += P.a;
        }
        uint16_t h[32], l[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          h[j] = f2bf(v[j]);
          if (SPLIT) l[j] = f2bf(v[j] - bf2f(h[j]));
        }
        const int cmin = sym ? r : 0;  // symmetric: this row stores columns >= r ...
        store_row32(pr.o_hi, pr.ldo, r, c0, cmin, N, h);
        if (SPLIT) store_row32(pr.o_lo, pr.ldo, r, c0, cmin, N, l);
        if (sym && c0 + 31 > r) {      // ... and mirrors columns > r into row c, column r
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j;
            if (c > r && c < N) {
              pr.o_hi[(int64_t)c * pr.ldo + r] = h[j];
              if (SPLIT) pr.o_lo[(int64_t)c * pr.ldo + r] = l[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(tempty0 + acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(kTmemCols)
                 : "memory");
  }
}


// ================================================================ CTA-pair kernel
// The same three phases on 256 x 256 output tiles computed by a pair of CTAs (a cluster of
// two) with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16): CTA rank r holds rows
// 128r..128r+127 of the A tile and rows 128r..128r+127 of the 256-row B tile in its own
// shared memory, and receives rows 128r..128r+127 of the accumulator in its own tensor
// memory.  Per k-block each CTA stages 32 KB instead of 48 KB, so six stages fit, and the
// pair reads each B panel once instead of twice.
//   both CTAs  warp 0, four issuing lanes: TMA loads of the CTA's own halves; completion is
//              counted on the leader's (rank 0) full barrier;
//   leader     warp 1 lane 0: waits the full barrier, issues the pair MMAs, and commits to
//              the empty barrier and accumulator-full barrier of both CTAs (multicast);
//   both CTAs  warps 2-9: epilogue of the CTA's 128 rows; release the accumulator by arriving
//              on the leader's accumulator-empty barrier (16 arrivals).
// Tensor memory is allocated by one warp of each CTA (cta_group::2) and both CTAs check that
// they received the same base column before any work; on a mismatch the kernel records an
// error and does nothing.
// SPLIT: split-precision operands (hi and lo bf16 copies of both tiles in every stage, three
// MMAs per k-step) and an epilogue that writes hi and lo rows directly, no staging.
template <bool SPLIT>
struct PairCfgT {
  static constexpr int kOps = SPLIT ? 2 : 1;              // hi (+ lo) operand copies
  static constexpr int kStages = SPLIT ? 3 : 6;
  static constexpr uint32_t kHalfA = 128 * kBK * 2;       // 16 KB: this CTA's A rows
  static constexpr uint32_t kHalfB = 128 * kBK * 2;       // 16 KB: this CTA's B rows
  static constexpr uint32_t kLoOffset = kHalfA + kHalfB;  // the lo copies follow the hi ones
  static constexpr uint32_t kStageBytes = kOps * (kHalfA + kHalfB);
  static constexpr uint32_t kStagingOffset = kStages * kStageBytes;
  static constexpr uint32_t kStagingPerWarp = SPLIT ? 0 : 2 * 32 * 32 * 2;  // block + transpose
  static constexpr uint32_t kBarOffset = kStagingOffset + kEpiWarps * kStagingPerWarp;
  static constexpr uint32_t kSmem = 1024 + kBarOffset + 256;
  static constexpr uint32_t kTmemCols = 512;              // two 128 x 256 fp32 accumulators
  static constexpr int kAccs = kTmemCols / kBN;
};
using PairCfg = PairCfgT<false>;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at shared::cta address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t map_rank(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __noinline__ bool mbar_wait_cl_slow(uint32_t bar, uint32_t parity, const Guard& g,
                                               bool honor_abort) {
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (honor_abort && *g.abort) return false;
      if (globaltimer() - t0 > g.limit_ns) {
        atomicOr(g.status, kStatusTimeout);
        *g.abort = 1;
        return false;
      }
    }
  }
}

// The same with cluster-scope acquire, for barriers that receive arrivals from the peer CTA's
// threads (the accumulator-empty barrier).
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, const Guard& g,
                                             bool honor_abort = true) {
  return mbar_try_wait_cl(bar, parity) || mbar_wait_cl_slow(bar, parity, g, honor_abort);
}

// Arrival on a barrier of either CTA of the pair (the accumulator-empty barrier, in the
// leader).  What it publishes is that this warp's tensor-memory reads have completed
// (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync); the MMA issuer reads no memory
// this thread wrote, so the release is CTA-scoped.  A cluster-scoped release made every
// epilogue warp wait at each tile's end for its outstanding memory operations (3 % of the
// GPT-2-small Newton-Schulz time).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}


__device__ __forceinline__ void tma_load3d_pair_p(bool p, uint32_t dst, const CUtensorMap* map,
                                                  int x, int y, int z, uint32_t leader_bar) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " @p cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n}\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(leader_bar),
      "r"((uint32_t)p)
      : "memory");
}

__device__ __forceinline__ void tma_load_pair_p(bool p, uint32_t dst, const CUtensorMap* map,
                                                int x, int y, uint32_t leader_bar) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %5, 0;\n"
      " @p cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n}\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(leader_bar), "r"((uint32_t)p)
      : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---------------------------------------------------------------- pair-kernel epilogue helpers
// Staging block of one epilogue warp: 32 rows x 32 bf16, 64 B per row, the four 16-byte
// chunks of row r stored in the order k ^ ((r >> 1) & 3).  With that permutation a warp
// access of one chunk of each of 32 rows (one row per lane) and a warp access of 8 whole rows
// (four lanes per row) both spread over all eight 16-byte bank groups: 4 wavefronts for
// 512 B, the minimum.
__device__ __forceinline__ uint32_t stg_off(int r, int k) {
  return (uint32_t)(r * 64 + ((k ^ ((r >> 1) & 3)) << 4));
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t a, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Eight bf16 at (r, c) of a row-major buffer (c % 8 == 0, ld % 8 == 0), zero outside M x N.
__device__ __forceinline__ uint4 load_granule(const uint16_t* p, int64_t ld, int r, int c, int M,
                                              int N) {
  if (r >= M || c >= N) return make_uint4(0u, 0u, 0u, 0u);
  const uint16_t* src = p + (int64_t)r * ld + c;
  if (c + 8 <= N) return *reinterpret_cast<const uint4*>(src);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  for (int e = 0; e < 8; ++e)
    if (c + e < N) w[e >> 1] |= (uint32_t)src[e] << (16 * (e & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// tcgen05.ld of 32 consecutive fp32 columns of this thread's TMEM lane, split in issue and
// wait so that other work overlaps the load; the registers are read-write operands of the
// wait, so no use of them can move above it.
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void tma_store_block(const CUtensorMap* map, uint32_t src, int x,
                                                int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
}

__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

template <bool SPLIT>
__global__ void __launch_bounds__(kNsThreads, 1) ns_gemm_pair_kernel(const __grid_constant__ NsLaunchParams P) {
  using C = PairCfgT<SPLIT>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // as in ns_gemm_kernel
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  // bars: full[S] | empty[S] | tfull[2] | tempty[2] | drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int full0 = 0, empty0 = S, tfull0 = 2 * S, tempty0 = 2 * S + 2, drain = 2 * S + 4;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar(full0 + s), 1);
      mbar_init(bar(empty0 + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(tfull0 + a), 1);
      mbar_init(bar(tempty0 + a), 2 * kEpiWarps);
    }
    mbar_init(bar(drain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(C::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous phase has completed
  const uint32_t tmem_base = *tmem_slot;
  uint32_t peer_base;
  asm volatile("ld.shared::cluster.u32 %0, [%1];"
               : "=r"(peer_base)
               : "r"(map_rank(smem_u32(tmem_slot), rank ^ 1u))
               : "memory");
  const bool usable = peer_base == tmem_base;
  if (!usable && threadIdx.x == 0) atomicOr(P.status, kStatusTmemMismatch);
  const Guard g{abort_flag, P.wait_limit_ns, P.status};
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (!usable) {
    // nothing runs: fall through to the teardown
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // Four lanes in lockstep, one round per two k-blocks: lane bit 1 picks the k-block of the
    // round (even / odd), lane bit 0 the operand (A / B half).  Each lane issues one 16 KB
    // load per round (or two 8 KB loads for an MN-major operand without the 3D view); the
    // leader's A lane arms the stage's full barrier for the bytes of both CTAs.
    if (lane < 4) {
      const int par = lane >> 1, opnd = lane & 1;
      // This lane's tile and k-block; the tile's table fields come a tile ahead (TileFields).
      int t = pair, kb = par;
      TileFields cur = tile_fields(P, t, tile_row(P, t));
      TileFields nxt = tile_fields(P, t + npairs, tile_row(P, t + npairs));
      NsTile row2 = tile_row(P, t + 2 * npairs);
      auto advance = [&]() {       // past the tiles whose k-blocks this lane has left
        while (t < P.ntiles && kb >= cur.nk()) {
          kb -= cur.nk();
          t += npairs;
          cur = nxt;
          nxt = tile_fields(P, t + npairs, row2);
          row2 = tile_row(P, t + 2 * npairs);
        }
      };
      advance();
      uint32_t q = (uint32_t)par;  // position in the k-block sequence
      uint32_t armed = 0, last_par = 0;
      int last_q = -1;             // the last k-block this lane issued
      for (;;) {
        bool act = t < P.ntiles && !*abort_flag;
        if (!__any_sync(0xFu, act)) break;
        const int stage = (int)(q % S);
        const uint32_t ph = (q / S) & 1u;
        if (act && !mbar_wait(bar(empty0 + stage), ph ^ 1u, g)) act = false;
        const CUtensorMap* mp = P.maps + (opnd ? cur.map_b : cur.map_a);
        const int mn = opnd ? cur.b_mn : cur.a_mn;
        const int view3 = SPLIT ? 0 : (cur.mn3d >> opnd) & 1;
        const int r0 = opnd ? cur.tn * kBN + 128 * (int)rank : cur.tm * 256 + 128 * (int)rank;
        const int k0 = kb * kBK;
        const bool self = cur.self();
        if (act && kb == 0) prefetch_map(mp + (mn ? (view3 ? 2 : 0) : 1));
        const uint32_t fb_local = bar(full0 + stage);
        const uint32_t fb = map_rank(fb_local, 0);
        const uint32_t dst = sbase + (uint32_t)stage * C::kStageBytes + (opnd ? C::kHalfA : 0u);
        // a self-operand tile loads the A halves only (both CTAs' bytes on the leader's barrier)
        expect_tx_p(act && leader && opnd == 0, fb_local,
                    self ? 2u * C::kOps * C::kHalfA : 2u * C::kStageBytes);
        const bool ld = act && !(self && opnd == 1);
        tma_load3d_pair_p(ld && mn && view3, dst, mp + 2, 0, k0, r0 / 64, fb);
        tma_load_pair_p(ld && mn && !view3, dst, mp, r0, k0, fb);
        tma_load_pair_p(ld && mn && !view3, dst + kBoxBytes, mp, r0 + 64, k0, fb);
        tma_load_pair_p(ld && !mn, dst, mp + 1, k0, r0, fb);
        if constexpr (SPLIT) {  // the lo copy of the same box, from the lo half's maps
          const CUtensorMap* ml = mp + kMapsPerHalf;
          const uint32_t dl = dst + C::kLoOffset;
          tma_load_pair_p(ld && mn, dl, ml, r0, k0, fb);
          tma_load_pair_p(ld && mn, dl + kBoxBytes, ml, r0 + 64, k0, fb);
          tma_load_pair_p(ld && !mn, dl, ml + 1, k0, r0, fb);
        }
        if (act && opnd == 0) {
          armed |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
          last_q = (int)q;
        }
        q += 2;
        kb += 2;
        advance();
      }
      // teardown: the leader's full barriers count both CTAs' bytes
      if constexpr (S % 2 == 0) {
        // an even stage count gives each parity lane its own stages
        if (leader)
          for (int st = 0; st < S; ++st)
            if (armed & (1u << st)) mbar_wait(bar(full0 + st), (last_par >> st) & 1u, g, false);
      } else {
        // an odd stage count makes the two parity lanes share stages, so a lane's own record
        // can be a phase behind: every k-block q < n was issued (even ones by lane 0, odd
        // ones by lane 2), and stage st last held k-block st + S floor((n - 1 - st) / S)
        const int l0 = __shfl_sync(0xFu, last_q, 0), l2 = __shfl_sync(0xFu, last_q, 2);
        const int n = max(l0, l2) + 1;
        if (leader && lane == 0)
          for (int st = 0; st < S && st < n; ++st) {
            const int ql = st + S * ((n - 1 - st) / S);
            mbar_wait(bar(full0 + st), (uint32_t)((ql / S) & 1), g, false);
          }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    // the tile's table fields come a tile ahead (TileFields)
    TileFields nxt = tile_fields(P, pair, tile_row(P, pair));
    NsTile row1 = tile_row(P, pair + npairs);
    for (int t = pair; t < P.ntiles; t += npairs) {
      const TileFields cur = nxt;
      nxt = tile_fields(P, t + npairs, row1);
      row1 = tile_row(P, t + 2 * npairs);
      const int nk = cur.nk(), a_mn = cur.a_mn, b_mn = cur.b_mn;
      const uint32_t b_off = cur.self() ? 0u : C::kHalfA;  // B = A on the diagonal
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) |
                             ((uint32_t)b_mn << 16) | ((uint32_t)(kBN >> 3) << 17) |
                             ((uint32_t)(256 >> 4) << 24);
      if (!mbar_wait_cl(bar(tempty0 + acc), acc_phase ^ 1u, g)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(bar(full0 + stage), phase, g)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = sbase + (uint32_t)stage * C::kStageBytes;
        const uint32_t sbb = sa + b_off;
#pragma unroll
        for (int j = 0; j < kBK / 16; ++j) {
          const uint64_t ad = operand_desc(sa, a_mn, j), bd = operand_desc(sbb, b_mn, j);
          tc_mma_pair(d_tmem, ad, bd, idesc, (kb | j) != 0);
          if constexpr (SPLIT) {
            tc_mma_pair(d_tmem, ad, operand_desc(sbb + C::kLoOffset, b_mn, j), idesc, 1u);
            tc_mma_pair(d_tmem, operand_desc(sa + C::kLoOffset, a_mn, j), bd, idesc, 1u);
          }
        }
        tc_commit_pair(bar(empty0 + stage), 0x3);
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit_pair(bar(tfull0 + acc), 0x3);
      if (++acc == C::kAccs) { acc = 0; acc_phase ^= 1u; }
    }
    tc_commit_pair(bar(drain), 0x1);
    mbar_wait(bar(drain), 0u, g, false);
  } else if (warp >= 2 && SPLIT) {
    // ------------------------------------------------------------ epilogue, split outputs
    // One row per lane: the fp32 accumulator, combined with the addend (its hi + lo rows),
    // is rounded to a hi and a lo bf16 part and both are stored directly; a symmetric output
    // stores the columns >= r of row r and mirrors the columns > r.
    const int quarter = warp & 3;
    const int c_first = ((warp - 2) >> 2) * kEpiChunks;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < P.ntiles; t += npairs) {
      const NsTile tile = P.tiles[t];
      const NsProblem& pr = P.probs[tile.prob];
      const int M = pr.M, N = pr.N, kind = pr.kind, sym = pr.sym;
      const int m0 = tile.tm * 256 + 128 * (int)rank, n0 = tile.tn * kBN;
      const int rw = m0 + quarter * 32, r = rw + lane;
      const bool rvalid = r < M;
      const float s = 1.f / (P.norm[pr.mat] + P.eps);
      if (!mbar_wait(bar(tfull0 + acc), acc_phase, g)) break;
      tc_fence_after();
      float alpha = 1.f, beta = 0.f;
      if (kind == kGram) {
        alpha = pr.first ? s * s : 1.f;
      } else if (kind == kPoly) {
        alpha = P.c;
        beta = P.b;
      } else {
        alpha = pr.first ? s : 1.f;
        if (!pr.fold_a) beta = P.a * alpha;
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll 1
      for (int q = 0; q < kEpiChunks; ++q) {
        const int cc = c_first + q, c0 = n0 + cc * 32;
        if (c0 >= N || rw >= M) break;                 // warp-uniform
        if (sym && c0 + 31 < rw) continue;             // chunk entirely below the diagonal
        uint32_t a32[32];
        tc_ld32_issue(taddr + (uint32_t)(cc * 32), a32);
        tc_ld_wait(a32);
        if (!rvalid) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(a32[j]);
        if (beta != 0.f) {
          float d[32], dl[32];
          load_row32(pr.d_hi, pr.ldd, r, c0, N, d);
          load_row32(pr.d_lo, pr.ldd, r, c0, N, dl);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = fmaf(alpha, v[j], beta * (d[j] + dl[j]));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
        }
        if (kind == kPoly && pr.fold_a && c0 == rw) {  // a on the diagonal: column `lane`
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == lane) v[j] += P.a;
        }
        uint16_t h[32], l[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          h[j] = f2bf(v[j]);
          l[j] = f2bf(v[j] - bf2f(h[j]));
        }
        const int cmin = sym ? r : 0;
        store_row32(pr.o_hi, pr.ldo, r, c0, cmin, N, h);
        store_row32(pr.o_lo, pr.ldo, r, c0, cmin, N, l);
        if (sym && c0 + 31 > r) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j;
            if (c > r && c < N) {
              pr.o_hi[(int64_t)c * pr.ldo + r] = h[j];
              pr.o_lo[(int64_t)c * pr.ldo + r] = l[j];
            }
          }
        }
        if (pr.t_hi) {
          // T = (5 I - out) / 4 of the stored output (hi + lo), as a split pair
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float tv = ((r == c0 + j ? 5.f : 0.f) - (bf2f(h[j]) + bf2f(l[j]))) * 0.25f;
            h[j] = f2bf(tv);
            l[j] = f2bf(tv - bf2f(h[j]));
          }
          store_row32(pr.t_hi, pr.ldo, r, c0, cmin, N, h);
          store_row32(pr.t_lo, pr.ldo, r, c0, cmin, N, l);
          if (sym && c0 + 31 > r) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int c = c0 + j;
              if (c > r && c < N) {
                pr.t_hi[(int64_t)c * pr.ldo + r] = h[j];
                pr.t_lo[(int64_t)c * pr.ldo + r] = l[j];
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_rank(bar(tempty0 + acc), 0));
      if (++acc == C::kAccs) { acc = 0; acc_phase ^= 1u; }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Warp w covers TMEM lane quarter (w & 3), i.e. 32 rows of the CTA's 128, and four
    // 32-column chunks.  The addend D is read from global memory in coalesced form (a warp
    // access covers 8 rows x 64 B), two chunks ahead, and turned into one row per lane
    // through the warp's 4 KB staging area; each output block is written there (64-byte
    // swizzled, the layout of the store map) and leaves by TMA store.  A symmetric output uses
    // both 2 KB halves (block + transpose) and waits for the previous store group; any other
    // output alternates between the halves, so one store may still be reading the other half.
    // A launch runs one phase, so its outputs are all symmetric (Gram, polynomial) or all not
    // (apply).
    const int quarter = warp & 3;
    const int c_first = ((warp - 2) >> 2) * kEpiChunks;
    const uint32_t stg0 = sbase + C::kStagingOffset + (uint32_t)(warp - 2) * C::kStagingPerWarp;
    const uint32_t stg_t = stg0 + 2048u;  // the transposed block of a symmetric output
    uint32_t nstore = 0;
    const int crow = lane >> 2, cchunk = lane & 3;
    // A tile's table fields, read two tiles ahead (from a tile row read three tiles ahead), and
    // its norm, read one tile ahead: neither the tile setup nor the addend prefetch waits for a
    // table read.
    struct EpiFields {
      int M, N, kind, sym, first, fold_a, map_o, mat, tm, tn, ldd;
      const uint16_t* d_hi;
    };
    auto epi_fields = [&](int t, const NsTile& row) {
      EpiFields f{0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, nullptr};
      if (t >= P.ntiles) return f;
      const NsProblem& pp = P.probs[row.prob];
      f.M = pp.M;
      f.N = pp.N;
      f.kind = pp.kind;
      f.sym = pp.sym;
      f.first = pp.first;
      f.fold_a = pp.fold_a;
      f.map_o = pp.map_o;
      f.mat = pp.mat;
      f.tm = row.tm;
      f.tn = row.tn;
      f.ldd = (int)pp.ldd;
      f.d_hi = pp.d_hi;
      return f;
    };
    // Where this warp's D of a tile comes from: the addend at the warp's first row and first
    // column, its pitch, and packed in one word which of the four chunks have one (bits 0-3),
    // the rows left from there (bits 4-9, at most 32) and the columns left (bits 10-17, at
    // most 128).  A tile past the end (M = 0) has none.
    struct DSrc {
      const uint16_t* p;
      int ld;
      uint32_t bits;
    };
    auto dsrc_of = [&](const EpiFields& f) {
      DSrc d{nullptr, 0, 0u};
      const int rw_ = f.tm * 256 + 128 * (int)rank + quarter * 32;
      const int cb = f.tn * kBN + c_first * 32;
      const bool has_d = f.kind == kPoly || (f.kind == kApply && !f.fold_a);
      if (!has_d || rw_ >= f.M) return d;
      d.p = f.d_hi + (int64_t)rw_ * f.ldd + cb;
      d.ld = f.ldd;
      uint32_t live = 0u;
#pragma unroll
      for (int q = 0; q < kEpiChunks; ++q) {
        const int c0_ = cb + 32 * q;
        if (c0_ < f.N && !(f.sym && c0_ + 31 < rw_)) live |= 1u << q;
      }
      const uint32_t rows = (uint32_t)min(f.M - rw_, 32), cols = (uint32_t)min(f.N - cb, 128);
      d.bits = live | (rows << 4) | (cols << 10);
      return d;
    };
    auto load_d = [&](const DSrc& ds, int q, uint4 (&dst)[4]) {
      if (!((ds.bits >> q) & 1u)) return;
      const int rows = (int)((ds.bits >> 4) & 63u), cols = (int)(ds.bits >> 10);
      if (rows == 32 && cols == 128) {  // the warp's whole 32 x 128 region is inside
        const uint16_t* src = ds.p + (int64_t)crow * ds.ld + 32 * q + 8 * cchunk;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          dst[i] = __ldg(reinterpret_cast<const uint4*>(src + (int64_t)(8 * i) * ds.ld));
        return;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = load_granule(ds.p, ds.ld, 8 * i + crow, 32 * q + 8 * cchunk, rows, cols);
    };
    // D is prefetched two chunks ahead (chunk q + 2 of the tile, or chunk q - 2 of the next
    // one), in a ring of two register slots: slot q & 1 holds chunk q.
    uint4 dpre[2][4];
    EpiFields f0 = epi_fields(pair, tile_row(P, pair));
    EpiFields f1 = epi_fields(pair + npairs, tile_row(P, pair + npairs));
    NsTile row2 = tile_row(P, pair + 2 * npairs);
    float nrm0 = P.norm[f0.mat];
    DSrc cur = dsrc_of(f0);
    load_d(cur, 0, dpre[0]);
    load_d(cur, 1, dpre[1]);
    DSrc nxt = dsrc_of(f1);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < P.ntiles; t += npairs) {
      const EpiFields f = f0;
      const int M = f.M, N = f.N, kind = f.kind, sym = f.sym;
      const int m0 = f.tm * 256 + 128 * (int)rank, n0 = f.tn * kBN;
      const int rw = m0 + quarter * 32;
      const int r = rw + lane;
      const float s = 1.f / (nrm0 + P.eps);
      // read ahead: the fields of tile t + 2 npairs, the row of t + 3 npairs, the norm of t + npairs
      const EpiFields f2 = epi_fields(t + 2 * npairs, row2);
      row2 = tile_row(P, t + 3 * npairs);
      const float nrm1 = P.norm[f1.mat];
      // refill slot q & 1 once chunk q has taken its D
      auto refill = [&](int q) {
        if (q + 2 < kEpiChunks)
          load_d(cur, q + 2, dpre[q & 1]);
        else
          load_d(nxt, q + 2 - kEpiChunks, dpre[q & 1]);
      };
      if (!mbar_wait(bar(tfull0 + acc), acc_phase, g)) break;
      tc_fence_after();
      float alpha = 1.f, beta = 0.f;
      if (kind == kGram) {
        alpha = f.first ? s * s : 1.f;
      } else if (kind == kPoly) {
        alpha = P.c;
        beta = P.b;
      } else {
        alpha = f.first ? s : 1.f;
        if (!f.fold_a) beta = P.a * alpha;
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll
      for (int q = 0; q < kEpiChunks; ++q) {
        const int cc = c_first + q;
        const int c0 = n0 + cc * 32;
        // warp-uniform: the chunk has rows and columns, and is not below the diagonal
        if (c0 >= N || rw >= M || (sym && c0 + 31 < rw)) {
          refill(q);
          continue;
        }
        uint32_t a32[32];
        tc_ld32_issue(taddr + (uint32_t)(cc * 32), a32);
        const uint32_t half = sym ? 0u : (nstore & 1u);
        const uint32_t stg = stg0 + half * 2048u;
        if (lane == 0) {
          if (sym)
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
          else
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        }
        __syncwarp();
        uint32_t dw[16];  // D as bf16 pairs, one row per lane
        if (beta != 0.f) {
          // D from the coalesced layout to one row per lane
#pragma unroll
          for (int i = 0; i < 4; ++i) sts128(stg + stg_off(8 * i + crow, cchunk), dpre[q & 1][i]);
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 w4 = lds128(stg + stg_off(lane, k));
            dw[4 * k] = w4.x;
            dw[4 * k + 1] = w4.y;
            dw[4 * k + 2] = w4.z;
            dw[4 * k + 3] = w4.w;
          }
          __syncwarp();
        }
        refill(q);
        tc_ld_wait(a32);
        // the polynomial phase adds a on the diagonal: column `lane` of a chunk on it
        const float dg = (kind == kPoly && f.fold_a && c0 == rw) ? P.a : 0.f;
        uint32_t hw[16];  // bf16 pairs (column 2k in the low half)
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          float v0 = __uint_as_float(a32[2 * k]), v1 = __uint_as_float(a32[2 * k + 1]);
          if (beta != 0.f) {
            v0 = fmaf(alpha, v0, beta * bf_lo(dw[k]));
            v1 = fmaf(alpha, v1, beta * bf_hi(dw[k]));
          } else {
            v0 *= alpha;
            v1 *= alpha;
          }
          if (dg != 0.f) {
            if (2 * k == lane) v0 += dg;
            if (2 * k + 1 == lane) v1 += dg;
          }
          hw[k] = pack_bf16x2(v0, v1);
        }
        // stage the block (and its transpose for a symmetric output), then TMA store
#pragma unroll
        for (int k = 0; k < 4; ++k)
          sts128(stg + stg_off(lane, k), make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2],
                                                    hw[4 * k + 3]));
        if (sym) {
          // the transpose, 8 x 8 sub-blocks at a time: ldmatrix.trans reads sub-blocks
          // (n, 0..3) of the staged block transposed into registers and stmatrix writes them as
          // sub-blocks (0..3, n) of the transposed block (both conflict-free in this layout)
          __syncwarp();
#pragma unroll
          for (int n = 0; n < 4; ++n) {
            uint32_t t0, t1, t2, t3;
            asm volatile(
                "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                : "=r"(t0), "=r"(t1), "=r"(t2), "=r"(t3)
                : "r"(stg + stg_off(8 * n + (lane & 7), lane >> 3))
                : "memory");
            asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(
                             stg_t + stg_off(lane, n)),
                         "r"(t0), "r"(t1), "r"(t2), "r"(t3)
                         : "memory");
          }
        }
        const bool diag = sym && c0 == rw;
        if (diag) {
          // block on the diagonal: the stored block is symmetric, row r keeping its own
          // columns >= r and taking, below the diagonal, column r of row c from the staged
          // transpose; it leaves in one store (rows and columns past M clipped by the map).
          // Word w of a staged row holds columns 2w (low half) and 2w + 1 (high half).
          __syncwarp();
#pragma unroll 1
          for (int w = 0; w < 16; ++w) {
            if (2 * w < lane) {
              const uint32_t off = stg_off(lane, w >> 2) + (uint32_t)((w & 3) * 4);
              const uint32_t tv = lds32(stg_t + off);
              if (2 * w + 1 < lane)
                sts32(stg + off, tv);
              else
                sts16(stg + off, (uint16_t)tv);
            }
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          const CUtensorMap* map_o = P.maps + f.map_o;
          tma_store_block(map_o, stg, c0, rw);
          if (sym && !diag) tma_store_block(map_o, stg_t, rw, c0);
          asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        ++nstore;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_rank(bar(tempty0 + acc), 0));
      if (++acc == C::kAccs) { acc = 0; acc_phase ^= 1u; }
      cur = nxt;
      nxt = dsrc_of(f2);
      f0 = f1;
      f1 = f2;
      nrm0 = nrm1;
    }
    if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");  // stores done
    __syncwarp();
  }

  tc_fence_before();
  __syncwarp();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while its peer may still use its memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(C::kTmemCols)
                 : "memory");
  }
}

}  // namespace


cudaError_t ns_prepare_kernels() {
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_pair_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PairCfg::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ns_gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)PairCfgT<true>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(ns_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)Cfg<true>::kSmem);
}

int ns_pair_max_clusters(int num_sms, bool split) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
  cfg.blockDim = dim3(kNsThreads, 1, 1);
  cfg.dynamicSmemBytes = split ? PairCfgT<true>::kSmem : PairCfg::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t e = split
      ? cudaOccupancyMaxActiveClusters(&n, ns_gemm_pair_kernel<true>, &cfg)
      : cudaOccupancyMaxActiveClusters(&n, ns_gemm_pair_kernel<false>, &cfg);
  return e == cudaSuccess ? n : -1;
}

cudaError_t launch_ns_phase(const NsLaunchParams& p, bool split, int grid, cudaStream_t s) {
  if (p.ntiles <= 0) return cudaSuccess;
  // Programmatic dependent launch: a phase's grid may start while the previous one drains
  // (its prologue overlaps that tail; the kernel waits for the previous grid before it reads).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kNsThreads, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  if (split) {
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.dynamicSmemBytes = Cfg<true>::kSmem;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ns_gemm_kernel<true>, p);
  }
  // bf16 operands: CTA pairs; `grid` is the number of co-resident pairs
  const int pairs = std::max(1, std::min(p.ntiles, grid));
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.dynamicSmemBytes = PairCfg::kSmem;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel<false>, p);
}

cudaError_t launch_ns_pair_split(const NsLaunchParams& p, int pairs, cudaStream_t s) {
  if (p.ntiles <= 0) return cudaSuccess;
  pairs = std::max(1, std::min(p.ntiles, pairs));
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kNsThreads, 1, 1);
  cfg.dynamicSmemBytes = PairCfgT<true>::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ns_gemm_pair_kernel<true>, p);
}

}  // namespace mfsdp
