// HBM-streaming kernels of the owner-local step: owner gradient deposit fused with Nesterov
// momentum and the Frobenius-norm partials, the fixed-order norm reduction, the scaled update
// with decoupled weight decay, AdamW on the packed tail, and small helpers.
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §3 and
// §4.2 (the reduced full gradient is written into the owner segment), §2 (Muon's input is the
// momentum-buffered gradient), §5.1 (torch.optim.Muon / AdamW semantics).
//
// Layout: every per-element buffer is flat over the owner's matrices (each matrix a
// contiguous row-major range).  A launch partitions each matrix into CTAs of kChunk
// consecutive elements, so a CTA never straddles two matrices and the per-CTA norm partials
// can be reduced per matrix in a fixed order.  Accesses are 16-byte vectors, coalesced across
// the warp; a matrix whose offset is not a multiple of 8 elements takes a scalar path.
#include <cuda_bf16.h>

#include "mfsdp_internal.h"

namespace mfsdp {

__device__ int g_status_word;

int* status_word_address() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

namespace {

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <typename T>
__device__ __forceinline__ float load1(const void* base, int64_t e);
template <>
__device__ __forceinline__ float load1<__nv_bfloat16>(const void* base, int64_t e) {
  return bf16_bits_to_float(static_cast<const uint16_t*>(base)[e]);
}
template <>
__device__ __forceinline__ float load1<float>(const void* base, int64_t e) {
  return static_cast<const float*>(base)[e];
}

// CTA -> matrix: the last matrix whose first CTA is <= b (binary search over cta_begin).
__device__ __forceinline__ int find_matrix(const DevMat* mats, int n, int b) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mats[mid].cta_begin <= b) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Fixed-order block sum of one float per thread (xor-shuffle tree, then warp 0 over warps).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  if (w == 0) {
    s = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  }
  return s;  // valid in thread 0
}

// Raw 16-byte-aligned load of 8 contribution elements (one or two 16-byte vectors).
template <typename T>
struct Raw8;
template <>
struct Raw8<__nv_bfloat16> {
  uint4 v;
  __device__ __forceinline__ void load(const void* base, int64_t e) {
    v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e));
  }
  __device__ __forceinline__ void add_to(float (&g)[8]) const {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      g[2 * i] += bf16_bits_to_float(w[i] & 0xFFFFu);
      g[2 * i + 1] += bf16_bits_to_float(w[i] >> 16);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const void* base, int64_t e) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
    a = __ldcs(p);
    b = __ldcs(p + 1);
  }
  __device__ __forceinline__ void add_to(float (&g)[8]) const {
    g[0] += a.x; g[1] += a.y; g[2] += a.z; g[3] += a.w;
    g[4] += b.x; g[5] += b.y; g[6] += b.z; g[7] += b.w;
  }
};

// Momentum update, Nesterov input and the bf16 outputs of 8 consecutive elements at e, given
// their deposited gradient g (before grad_scale) and old momentum m8; adds u^2 to ss.
__device__ __forceinline__ void finish8(const ReduceParams& P, bool lo_out, int64_t e,
                                        float (&g)[8], const float (&m8)[8], float& ss) {
  const float gs = P.grad_scale, mu = P.mu, omm = P.one_minus_mu;
  float bm[8], u[8];
  uint32_t hb[4], lb[4];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float gj = g[j] * gs;
    g[j] = gj;
    bm[j] = fmaf(mu, m8[j], omm * gj);
    u[j] = P.nesterov ? fmaf(omm, gj, mu * bm[j]) : bm[j];
    ss = fmaf(u[j], u[j], ss);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint16_t h0 = float_to_bf16_bits(u[2 * j]), h1 = float_to_bf16_bits(u[2 * j + 1]);
    hb[j] = (uint32_t)h0 | ((uint32_t)h1 << 16);
    const uint16_t l0 = float_to_bf16_bits(u[2 * j] - bf16_bits_to_float(h0));
    const uint16_t l1 = float_to_bf16_bits(u[2 * j + 1] - bf16_bits_to_float(h1));
    lb[j] = (uint32_t)l0 | ((uint32_t)l1 << 16);
  }
  float4* mp = reinterpret_cast<float4*>(P.momentum + e);
  mp[0] = make_float4(bm[0], bm[1], bm[2], bm[3]);
  mp[1] = make_float4(bm[4], bm[5], bm[6], bm[7]);
  *reinterpret_cast<uint4*>(P.uhat + e) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
  if (lo_out) *reinterpret_cast<uint4*>(P.uhat_lo + e) = make_uint4(lb[0], lb[1], lb[2], lb[3]);
  if (P.grad) {
    float4* gp = reinterpret_cast<float4*>(P.grad + e);
    gp[0] = make_float4(g[0], g[1], g[2], g[3]);
    gp[1] = make_float4(g[4], g[5], g[6], g[7]);
  }
}

// The same for one element (scalar tails and unaligned matrices).
template <typename T>
__device__ __forceinline__ void finish1(const ReduceParams& P, bool lo_out, int64_t e, float& ss) {
  float g = 0.f;
  for (int w = 0; w < P.W; ++w) g += load1<T>(P.contrib.p[w], e);
  g *= P.grad_scale;
  const float bm = fmaf(P.mu, P.momentum[e], P.one_minus_mu * g);
  P.momentum[e] = bm;
  const float u = P.nesterov ? fmaf(P.one_minus_mu, g, P.mu * bm) : bm;
  const uint16_t h = float_to_bf16_bits(u);
  P.uhat[e] = h;
  if (lo_out) P.uhat_lo[e] = float_to_bf16_bits(u - bf16_bits_to_float(h));
  if (P.grad) P.grad[e] = g;
  ss = fmaf(u, u, ss);
}

// ------------------------------------------------------------------------------------------
// Owner gradient deposit + Nesterov momentum + norm partials, register path (used when some
// matrix starts at an element offset that is not a multiple of 8).  One CTA per chunk of
// kChunk elements; passes of kPassVecs 8-element vectors per thread with the contribution loop
// unrolled by kUnrollW, so kPassVecs x kUnrollW independent 16-byte loads are in flight.
// Contributions are summed in index order w = 0, 1, ... for every element.
// ------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2)
reduce_momentum_kernel(const __grid_constant__ ReduceParams P) {
  constexpr int kPassVecs = 2;
  constexpr int kUnrollW = sizeof(T) == 2 ? 4 : 2;
  __shared__ float red[kStreamThreads / 32];
  const int b = blockIdx.x;
  const int mi = find_matrix(P.mats, P.n_mats, b);
  const DevMat dm = P.mats[mi];
  const int64_t start = (int64_t)(b - dm.cta_begin) * kChunk;
  const int64_t cnt = min((int64_t)kChunk, dm.numel - start);
  const int64_t base = dm.offset + start;
  const bool lo_out = dm.split && P.uhat_lo != nullptr;
  const int W = P.W;
  float ss = 0.f;
  int64_t done = 0;
  if ((base & 7) == 0) {
    const int64_t nvec = cnt / kVec;
    for (int64_t v0 = 0; v0 < nvec; v0 += (int64_t)kStreamThreads * kPassVecs) {
      int64_t ev[kPassVecs];
      bool ok[kPassVecs];
#pragma unroll
      for (int i = 0; i < kPassVecs; ++i) {
        const int64_t v = v0 + (int64_t)i * kStreamThreads + threadIdx.x;
        ok[i] = v < nvec;
        ev[i] = base + (ok[i] ? v : 0) * kVec;
      }
      float g[kPassVecs][8];
#pragma unroll
      for (int i = 0; i < kPassVecs; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) g[i][j] = 0.f;
      int w = 0;
      for (; w + kUnrollW <= W; w += kUnrollW) {
        Raw8<T> raw[kUnrollW][kPassVecs];
#pragma unroll
        for (int u = 0; u < kUnrollW; ++u)
#pragma unroll
          for (int i = 0; i < kPassVecs; ++i)
            if (ok[i]) raw[u][i].load(P.contrib.p[w + u], ev[i]);
#pragma unroll
        for (int u = 0; u < kUnrollW; ++u)
#pragma unroll
          for (int i = 0; i < kPassVecs; ++i)
            if (ok[i]) raw[u][i].add_to(g[i]);
      }
      for (; w < W; ++w) {
#pragma unroll
        for (int i = 0; i < kPassVecs; ++i)
          if (ok[i]) {
            Raw8<T> raw;
            raw.load(P.contrib.p[w], ev[i]);
            raw.add_to(g[i]);
          }
      }
#pragma unroll
      for (int i = 0; i < kPassVecs; ++i) {
        if (!ok[i]) continue;
        const float4* mp = reinterpret_cast<const float4*>(P.momentum + ev[i]);
        const float4 m0 = mp[0], m1 = mp[1];
        const float m8[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        finish8(P, lo_out, ev[i], g[i], m8, ss);
      }
    }
    done = nvec * kVec;
  }
  for (int64_t k = done + threadIdx.x; k < cnt; k += kStreamThreads)  // scalar remainder
    finish1<T>(P, lo_out, base + k, ss);
  const float tot = block_sum(ss, red);
  if (threadIdx.x == 0) P.partials[b] = tot;
}

// ------------------------------------------------------------------------------------------
// Owner gradient deposit + Nesterov momentum + norm partials, bulk-copy path.
// A persistent grid walks the same per-matrix chunk partition (chunk c = CTA c of the
// partition; CTA b takes chunks b, b + grid, ...).  Each chunk is split into sub-chunks of
// E elements that flow through a ring of S shared-memory stages:
//   warp 8 (producer)  for each sub-chunk, once all consumer warps have released the stage
//                      (its empty mbarrier), copies the W contribution slices and the momentum
//                      slice in with cp.async.bulk, one slice per lane (a thread's bulk copies
//                      run one after another), completion counted on the stage's full
//                      mbarrier;
//   warps 0-7          wait for the stage, form G, the new momentum and the bf16 NS input for
//                      their 8-element vectors, write them to global memory, add u^2 to a
//                      per-thread sum, and release the stage (one arrival per warp).
// Warps are only coupled through the ring, never by a CTA-wide barrier.  At the end of a chunk
// each warp reduces its sum (xor-shuffle tree) into a per-chunk slot; the last warp to finish
// the chunk adds the eight warp sums in warp order and writes the chunk's partial, so the
// partial is the same for any grid size and any warp timing.  Waits are bounded; on expiry
// the kernel records a timeout, stops, waits for its copies in flight and exits.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ bool bulk_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ bool bulk_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, int* status,
                          volatile int* abort_flag, bool honor_abort) {
  if (bulk_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  for (uint32_t i = 1;; ++i) {
    if (bulk_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (honor_abort && *abort_flag) return false;
      if (gtimer() - t0 > limit_ns) {
        atomicOr(status, kStatusTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

constexpr int kConsumerWarps = kStreamThreads / 32;
constexpr int kBulkThreads = kStreamThreads + 32;  // consumers + the producer warp
constexpr int kChunkSlots = 16;                     // > stages: a warp runs at most S ahead

template <typename T>
__global__ void __launch_bounds__(kBulkThreads, 1)
reduce_momentum_bulk_kernel(const __grid_constant__ ReduceParams P,
                            const __grid_constant__ BulkCfg C) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ __align__(8) uint64_t full[kMaxBulkStages];
  __shared__ __align__(8) uint64_t empty[kMaxBulkStages];
  __shared__ float wsum[kChunkSlots][kConsumerWarps];
  __shared__ int wdone[kChunkSlots];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int W = P.W, E = C.sub_elems, S = C.stages;
  const uint32_t cbytes = (uint32_t)sizeof(T);
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(sm);
  auto fbar = [&](int st) { return (uint32_t)__cvta_generic_to_shared(&full[st]); };
  auto ebar = [&](int st) { return (uint32_t)__cvta_generic_to_shared(&empty[st]); };
  if (tid == 0) {
    for (int st = 0; st < S; ++st) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(fbar(st)), "r"(1u));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(ebar(st)),
                   "r"((uint32_t)kConsumerWarps));
    }
    for (int k = 0; k < kChunkSlots; ++k) wdone[k] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------------ producer warp
    uint32_t armed = 0, last_parity = 0;
    uint32_t q = 0;
    bool ok = true;
    for (int pc = blockIdx.x; pc < P.total_ctas && ok; pc += gridDim.x) {
      const int mi = find_matrix(P.mats, P.n_mats, pc);
      const DevMat dm = P.mats[mi];
      const int64_t rel0 = (int64_t)(pc - dm.cta_begin) * kChunk;
      const int64_t ccnt = min((int64_t)kChunk, dm.numel - rel0);
      for (int64_t sub0 = 0; sub0 < ccnt; sub0 += E, ++q) {
        const int st = (int)(q % (uint32_t)S);
        const uint32_t round = q / (uint32_t)S;
        // the stage's previous contents (round - 1) have been released by every consumer
        if (round > 0) {
          if (lane == 0)
            ok = bulk_wait(ebar(st), (round - 1) & 1u, C.wait_limit_ns, P.status, &abort_flag,
                           true);
          ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
          if (!ok) break;
        }
        const int64_t e0 = dm.offset + rel0 + sub0;
        const int n = (int)min((int64_t)E, ccnt - sub0);
        const int n8 = n & ~7;
        const uint32_t bar = fbar(st);
        const uint32_t dst = sbase + (uint32_t)st * C.stage_bytes;
        if (lane == 0)
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                       "r"((uint32_t)n8 * (cbytes * W + 4u))
                       : "memory");
        if (n8 > 0) {
          for (int w = lane; w <= W; w += 32) {
            if (w < W)
              bulk_copy(dst + (uint32_t)(w * E) * cbytes,
                        static_cast<const uint8_t*>(P.contrib.p[w]) + e0 * cbytes,
                        (uint32_t)n8 * cbytes, bar);
            else
              bulk_copy(dst + (uint32_t)(W * E) * cbytes, P.momentum + e0, (uint32_t)n8 * 4u,
                        bar);
          }
        }
        armed |= 1u << st;
        last_parity = (last_parity & ~(1u << st)) | ((round & 1u) << st);
      }
    }
    // every copy this CTA issued has landed before it exits
    if (lane == 0)
      for (int st = 0; st < S; ++st)
        if (armed & (1u << st))
          bulk_wait(fbar(st), (last_parity >> st) & 1u, C.wait_limit_ns, P.status, &abort_flag,
                    false);
  } else {
    // ------------------------------------------------------------------ consumer warps
    uint32_t q = 0, slot = 0;
    bool ok = true;
    for (int c = blockIdx.x; c < P.total_ctas && ok; c += gridDim.x, slot = (slot + 1) % kChunkSlots) {
      const int mi = find_matrix(P.mats, P.n_mats, c);
      const DevMat dm = P.mats[mi];
      const int64_t rel0 = (int64_t)(c - dm.cta_begin) * kChunk;
      const int64_t ccnt = min((int64_t)kChunk, dm.numel - rel0);
      const int64_t cbase = dm.offset + rel0;
      const bool lo_out = dm.split && P.uhat_lo != nullptr;
      float ss = 0.f;
      for (int64_t sub0 = 0; sub0 < ccnt; sub0 += E, ++q) {
        const int st = (int)(q % (uint32_t)S);
        ok = bulk_wait(fbar(st), (q / (uint32_t)S) & 1u, C.wait_limit_ns, P.status, &abort_flag,
                       true);
        if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
        const int n = (int)min((int64_t)E, ccnt - sub0);
        const int n8 = n & ~7;
        const int64_t e0 = cbase + sub0;
        const uint8_t* stage = sm + (size_t)st * C.stage_bytes;
        const float4* mo = reinterpret_cast<const float4*>(stage + (size_t)(W * E) * cbytes);
        for (int v = tid; v < (n8 >> 3); v += kStreamThreads) {
          float g[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int w = 0; w < W; ++w) {
            const uint8_t* cw = stage + (size_t)(w * E) * cbytes;
            Raw8<T> r;
            if (sizeof(T) == 2) {
              reinterpret_cast<uint4*>(&r)[0] = reinterpret_cast<const uint4*>(cw)[v];
            } else {
              reinterpret_cast<float4*>(&r)[0] = reinterpret_cast<const float4*>(cw)[2 * v];
              reinterpret_cast<float4*>(&r)[1] = reinterpret_cast<const float4*>(cw)[2 * v + 1];
            }
            r.add_to(g);
          }
          const float4 m0 = mo[2 * v], m1 = mo[2 * v + 1];
          const float m8[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          finish8(P, lo_out, e0 + (int64_t)v * 8, g, m8, ss);
        }
        if (tid < n - n8) finish1<T>(P, lo_out, e0 + n8 + tid, ss);  // last < 8 elements
        __syncwarp();
        if (lane == 0)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(ebar(st)) : "memory");
      }
      if (!ok) break;
      // chunk partial: warp sums in a slot, the last warp adds them in warp order
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      if (lane == 0) {
        wsum[slot][warp] = ss;
        __threadfence_block();
        if (atomicAdd(&wdone[slot], 1) == kConsumerWarps - 1) {
          __threadfence_block();
          float tot = 0.f;
          for (int k = 0; k < kConsumerWarps; ++k) tot += wsum[slot][k];
          P.partials[c] = tot;
          atomicExch(&wdone[slot], 0);
        }
      }
    }
  }
}

// One CTA per matrix: nu = sqrt(sum of its CTA partials), summed in fp64 in index order.
__global__ void __launch_bounds__(256) norm_finalize_kernel(const __grid_constant__ NormParams P) {
  __shared__ double red[256];
  const int i = blockIdx.x;
  const DevMat dm = P.mats[i];
  const int nparts = (int)((dm.numel + kChunk - 1) / kChunk);
  double s = 0.0;
  for (int k = threadIdx.x; k < nparts; k += blockDim.x) s += (double)P.partials[dm.cta_begin + k];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double nu = sqrt(red[0]);
    P.norm[i] = (float)nu;
    if (!isfinite(nu)) atomicOr(P.status, kStatusNonFinite);
  }
}

// ------------------------------------------------------------------------------------------
// Scaled update with decoupled weight decay: W = W*(1 - lr*wd) - lr*s*(O + O_lo).
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kStreamThreads)
apply_update_kernel(const __grid_constant__ UpdateParams P) {
  const int b = blockIdx.x;
  const int mi = find_matrix(P.mats, P.n_mats, b);
  const DevMat dm = P.mats[mi];
  const int64_t start = (int64_t)(b - dm.cta_begin) * kChunk;
  const int64_t cnt = min((int64_t)kChunk, dm.numel - start);
  const int64_t base = dm.offset + start;
  const float coef = P.lr * (P.lr_adjust ? dm.scale_rms : dm.scale_original);
  const float decay = P.decay;
  const bool use_lo = dm.split && P.ortho_lo != nullptr;
  int64_t done = 0;
  if ((base & 7) == 0) {
    const int64_t nvec = cnt / kVec;
#pragma unroll 4
    for (int64_t v = threadIdx.x; v < nvec; v += kStreamThreads) {
      const int64_t e = base + v * kVec;
      const uint4 o = __ldcs(reinterpret_cast<const uint4*>(P.ortho + e));
      const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
      float of[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        of[2 * j] = bf16_bits_to_float(ow[j] & 0xFFFFu);
        of[2 * j + 1] = bf16_bits_to_float(ow[j] >> 16);
      }
      if (use_lo) {
        const uint4 l = *reinterpret_cast<const uint4*>(P.ortho_lo + e);
        const uint32_t lw[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          of[2 * j] += bf16_bits_to_float(lw[j] & 0xFFFFu);
          of[2 * j + 1] += bf16_bits_to_float(lw[j] >> 16);
        }
      }
      float4* wp = reinterpret_cast<float4*>(P.weights + e);
      float4 w0 = wp[0], w1 = wp[1];
      w0.x = fmaf(-coef, of[0], w0.x * decay); w0.y = fmaf(-coef, of[1], w0.y * decay);
      w0.z = fmaf(-coef, of[2], w0.z * decay); w0.w = fmaf(-coef, of[3], w0.w * decay);
      w1.x = fmaf(-coef, of[4], w1.x * decay); w1.y = fmaf(-coef, of[5], w1.y * decay);
      w1.z = fmaf(-coef, of[6], w1.z * decay); w1.w = fmaf(-coef, of[7], w1.w * decay);
      wp[0] = w0;
      wp[1] = w1;
    }
    done = nvec * kVec;
  }
  for (int64_t k = done + threadIdx.x; k < cnt; k += kStreamThreads) {
    const int64_t e = base + k;
    float o = bf16_bits_to_float(P.ortho[e]);
    if (use_lo) o += bf16_bits_to_float(P.ortho_lo[e]);
    P.weights[e] = fmaf(-coef, o, P.weights[e] * decay);
  }
}

// ------------------------------------------------------------------------------------------
// AdamW on the packed tail (4 elements per thread per step).
// ------------------------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float tail_grad(const AdamParams& P, int64_t e) {
  float g = 0.f;
  for (int w = 0; w < P.W; ++w) g += load1<T>(P.contrib.p[w], e);
  return g * P.grad_scale;
}

__device__ __forceinline__ void adam_one(const AdamParams& P, int64_t e, float g) {
  float p = P.p[e] * P.decay;
  const float m = fmaf(P.b1, P.m[e], P.one_minus_b1 * g);
  const float v = fmaf(P.b2, P.v[e], P.one_minus_b2 * g * g);
  const float denom = fmaf(sqrtf(v), P.inv_sqrt_bc2, P.eps);
  p -= P.step_size * (m / denom);
  P.p[e] = p;
  P.m[e] = m;
  P.v[e] = v;
}

template <typename T>
__global__ void __launch_bounds__(256) adamw_kernel(const __grid_constant__ AdamParams P) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < P.n; e += stride)
    adam_one(P, e, tail_grad<T>(P, e));
}

__global__ void copy2d_kernel(const __grid_constant__ CopyParams P) {
  const int64_t total = P.rows * P.cols;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += stride) {
    const int64_t r = k / P.cols, c = k - r * P.cols;
    P.dst[r * P.ld_dst + c] = P.src[r * P.ld_src + c];
  }
}

// A bounded wait on an mbarrier that nothing arrives at: the wait must run out and report.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(1u));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
      uint32_t ok;
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(ok) : "r"(a), "r"(0u) : "memory");
      if (ok) break;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > limit_ns) {
        atomicOr(status, kStatusTimeout);
        break;
      }
    }
  }
}

int grid_for(int64_t n, int threads, int cap) {
  int64_t g = (n + threads - 1) / threads;
  if (g < 1) g = 1;
  return (int)(g < cap ? g : cap);
}

}  // namespace

cudaError_t launch_reduce_momentum(const ReduceParams& p, int contrib_dtype, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  if (!p.offsets_aligned) {
    if (contrib_dtype == 1)
      reduce_momentum_kernel<__nv_bfloat16><<<p.total_ctas, kStreamThreads, 0, s>>>(p);
    else
      reduce_momentum_kernel<float><<<p.total_ctas, kStreamThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // Sub-chunk of E elements: the W contribution slices plus the momentum slice of one stage
  // fit in kBulkStageBudget bytes (fewer contributions, longer copies: each bulk copy has a
  // fixed issue cost); as many stages as fit in kBulkSmemBudget (2 to 8).
  const int esz = contrib_dtype == 1 ? 2 : 4;
  const int per_elem = p.W * esz + 4;
  // E is a power of two from 256 up: it divides the chunk, and for E >= 2048 every thread of
  // the CTA gets the same number of 8-element vectors per stage.
  // (one or two contributions: 64 KB stages, three of them, so each copy is longer)
  const size_t budget = p.W <= 2 ? (size_t)64 * 1024 : kBulkStageBudget;
  int E = 256;
  while (2 * E <= kChunk && (size_t)(2 * E) * per_elem <= budget) E *= 2;
  BulkCfg c{};
  c.sub_elems = E;
  c.stage_bytes = E * per_elem;
  const int stages = (int)(kBulkSmemBudget / c.stage_bytes);
  c.stages = stages < 2 ? 2 : (stages > kMaxBulkStages ? kMaxBulkStages : stages);
  c.wait_limit_ns = p.wait_limit_ns;
  const size_t smem = (size_t)c.stages * c.stage_bytes;
  const int grid = p.total_ctas < sms ? p.total_ctas : sms;
  if (contrib_dtype == 1) {
    e = cudaFuncSetAttribute(reduce_momentum_bulk_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      reduce_momentum_bulk_kernel<__nv_bfloat16><<<grid, kBulkThreads, smem, s>>>(p, c);
  } else {
    e = cudaFuncSetAttribute(reduce_momentum_bulk_kernel<float>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) reduce_momentum_bulk_kernel<float><<<grid, kBulkThreads, smem, s>>>(p, c);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_norm_finalize(const NormParams& p, cudaStream_t s) {
  if (p.n_mats <= 0) return cudaSuccess;
  norm_finalize_kernel<<<p.n_mats, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_apply_update(const UpdateParams& p, cudaStream_t s) {
  if (p.total_ctas <= 0) return cudaSuccess;
  apply_update_kernel<<<p.total_ctas, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_adamw(const AdamParams& p, int contrib_dtype, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  const int grid = grid_for(p.n, 256, 152 * 16);
  if (contrib_dtype == 1)
    adamw_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(p);
  else
    adamw_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_copy2d(const CopyParams& p, cudaStream_t s) {
  if (p.rows <= 0 || p.cols <= 0) return cudaSuccess;
  copy2d_kernel<<<grid_for(p.rows * p.cols, 256, 152 * 8), 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* status, cudaStream_t s) {
  wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace mfsdp
