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

// Load 8 consecutive contribution elements as fp32.
template <typename T>
__device__ __forceinline__ void load8(const void* base, int64_t e, float (&x)[8]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const void* base, int64_t e, float (&x)[8]) {
  const uint4 v = __ldcs(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + e));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = bf16_bits_to_float(w[i] & 0xFFFFu);
    x[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

template <>
__device__ __forceinline__ void load8<float>(const void* base, int64_t e, float (&x)[8]) {
  const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + e);
  const float4 a = __ldcs(p), b = __ldcs(p + 1);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
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

// ------------------------------------------------------------------------------------------
// Owner gradient deposit + Nesterov momentum + norm partials.
// ------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kStreamThreads)
reduce_momentum_kernel(const __grid_constant__ ReduceParams P) {
  __shared__ float red[kStreamThreads / 32];
  const int b = blockIdx.x;
  const int mi = find_matrix(P.mats, P.n_mats, b);
  const DevMat dm = P.mats[mi];
  const int64_t start = (int64_t)(b - dm.cta_begin) * kChunk;
  const int64_t cnt = min((int64_t)kChunk, dm.numel - start);
  const int64_t base = dm.offset + start;
  const float gs = P.grad_scale, mu = P.mu, omm = P.one_minus_mu;
  const bool lo_out = dm.split && P.uhat_lo != nullptr;
  float ss = 0.f;

  auto one = [&](float g, int64_t e) {
    g *= gs;
    const float bm = fmaf(mu, P.momentum[e], omm * g);
    P.momentum[e] = bm;
    const float u = P.nesterov ? fmaf(omm, g, mu * bm) : bm;
    const uint16_t h = float_to_bf16_bits(u);
    P.uhat[e] = h;
    if (lo_out) P.uhat_lo[e] = float_to_bf16_bits(u - bf16_bits_to_float(h));
    if (P.grad) P.grad[e] = g;
    ss = fmaf(u, u, ss);
  };

  int64_t done = 0;
  if ((base & 7) == 0) {
    const int64_t nvec = cnt / kVec;
    for (int64_t v0 = 0; v0 < nvec; v0 += (int64_t)kStreamThreads * kVecsPerThread) {
      float g[kVecsPerThread][8];
#pragma unroll
      for (int i = 0; i < kVecsPerThread; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) g[i][j] = 0.f;
      for (int w = 0; w < P.W; ++w) {
        const void* cw = P.contrib.p[w];
#pragma unroll
        for (int i = 0; i < kVecsPerThread; ++i) {
          const int64_t v = v0 + (int64_t)i * kStreamThreads + threadIdx.x;
          if (v < nvec) {
            float x[8];
            load8<T>(cw, base + v * kVec, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) g[i][j] += x[j];
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kVecsPerThread; ++i) {
        const int64_t v = v0 + (int64_t)i * kStreamThreads + threadIdx.x;
        if (v >= nvec) continue;
        const int64_t e = base + v * kVec;
        float4* mp = reinterpret_cast<float4*>(P.momentum + e);
        const float4 m0 = mp[0], m1 = mp[1];
        const float mo[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float bm[8], u[8];
        uint32_t hb[4], lb[4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float gj = g[i][j] * gs;
          g[i][j] = gj;
          bm[j] = fmaf(mu, mo[j], omm * gj);
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
        mp[0] = make_float4(bm[0], bm[1], bm[2], bm[3]);
        mp[1] = make_float4(bm[4], bm[5], bm[6], bm[7]);
        *reinterpret_cast<uint4*>(P.uhat + e) = make_uint4(hb[0], hb[1], hb[2], hb[3]);
        if (lo_out) *reinterpret_cast<uint4*>(P.uhat_lo + e) = make_uint4(lb[0], lb[1], lb[2], lb[3]);
        if (P.grad) {
          float4* gp = reinterpret_cast<float4*>(P.grad + e);
          gp[0] = make_float4(g[i][0], g[i][1], g[i][2], g[i][3]);
          gp[1] = make_float4(g[i][4], g[i][5], g[i][6], g[i][7]);
        }
      }
    }
    done = nvec * kVec;
  }
  for (int64_t k = done + threadIdx.x; k < cnt; k += kStreamThreads) {  // scalar remainder
    const int64_t e = base + k;
    float g = 0.f;
    for (int w = 0; w < P.W; ++w) g += load1<T>(P.contrib.p[w], e);
    one(g, e);
  }
  const float tot = block_sum(ss, red);
  if (threadIdx.x == 0) P.partials[b] = tot;
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
  if (contrib_dtype == 1)
    reduce_momentum_kernel<__nv_bfloat16><<<p.total_ctas, kStreamThreads, 0, s>>>(p);
  else
    reduce_momentum_kernel<float><<<p.total_ctas, kStreamThreads, 0, s>>>(p);
  return cudaGetLastError();
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
