// Owner SOAP: Adam in the eigenbasis of the Shampoo statistics, on the owner's whole matrices
// (fp32).
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §5.7:
// with every 2D matrix whole on its owner, the owner can run SOAP (Adam in the Shampoo
// eigenbasis) in place of Muon.  Per owned matrix G (rows x cols) and step t >= 1, the SOAP
// update of Vyas et al. (2024) with the eigenbasis taken exactly at every step:
//     L = bs L + (1 - bs) G G^T,   R = bs R + (1 - bs) G^T G
//     Q_L, Q_R = eigenvectors of L, R (columns, descending eigenvalue)
//     M = b1 M + (1 - b1) G;   G' = Q_L^T G Q_R;   M' = Q_L^T M Q_R
//     V = b2 V + (1 - b2) G'^2                   (V in eigenbasis coordinates)
//     N = Q_L [ (M' / (1 - b1^t)) / (sqrt(V / (1 - b2^t)) + eps) ] Q_R^T
//     W = W (1 - lr wd) - lr N
//
// Eigenbases: cyclic two-sided block Jacobi, warm-started from the previous step's basis Q:
// A = Q^T L Q (nearly diagonal once the statistics move slowly), Z = Q, then sweeps over all
// pairs of 32-index blocks in round-robin order.  In one round every pair (P, Q) of blocks
// forms a 64 x 64 subproblem [A_PP A_PQ; A_QP A_QQ], reduced by a CTA in shared memory (one
// cyclic sweep of plane rotations, Golub & Van Loan §8.5, then one polar step), giving a
// 64 x 64 orthogonal J; a second launch applies all of the round's J to A (A <- J^T A J, block
// by block) and a third, beside the next round, to Z, kept transposed (Z^T <- J^T Z^T:
// eigenvectors as rows).  A sweep in
// which no subproblem rotated ends the solve for that matrix.  The eigenvalues are the
// Rayleigh quotients of the final basis, sorted (descending, ties by index), and Z's columns
// are scattered into Q in that order.  Plane rotations are skipped where the coupling is at
// rounding level, |a_pq| <= tol max_i |a_ii| (tol = 1e-6, about 16u, by default): the rotations
// of a block are 64-term fp32 sums, whose rounding leaves couplings of a few u ||L|| between
// nearly equal eigenvalues, and eigenvectors are accurate to about tol ||L|| / gap.
//
// Every product (statistics, A = Q^T L Q, the rotations into and out of the eigenbasis, the
// basis' final polar step Z^T <- (3I - Z^T Z) Z^T / 2) is the batched fp32 GEMM on the tensor
// cores (3xTF32 with k-block accumulation in fp32 registers, an fp32 GEMM's accuracy), and so
// are the Jacobi rotations of Z^T (jacobi_zrot_tc_kernel, the same split, on a stream of their
// own).  The rotations of A stay fp32 FFMA: there their rounding is a backward error of the
// eigenproblem that the eigenvectors amplify by 1 / gap (a 3xTF32 form, measured, missed the
// eigenvector tolerance on tight spectra).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

constexpr int kJB = 32;           // Jacobi block (indices)
constexpr int kJP = 2 * kJB;      // a pair of blocks: one 64 x 64 subproblem
constexpr int kJLd = kJP + 1;     // shared-memory pitch (conflict-free column access)
constexpr int kJThreads = 128;      // apply kernel (4 x 8 outputs per thread)
constexpr int kSolveThreads = 544;  // solve kernel: one S block per thread (528), 17 warps
// Sweeps of one 64 x 64 subproblem per round.  One suffices: the subproblem need not be
// diagonalised exactly for the outer iteration to converge (an emulation of the solve on
// rank-deficient statistics takes the same number of outer sweeps with 1, 2, 3 or 12), and
// near convergence a single sweep does diagonalise it.
constexpr int kSubSweeps = 1;
constexpr float kDefaultJacobiTol = 1e-6f;  // couplings below tol * max_i a_ii are not rotated

struct SideDev {           // one statistics matrix of the Jacobi solve ("side")
  float* stat;             // L or R, d x d (pitch d)
  float* q;                // basis state, d x d (pitch d): previous basis in, sorted basis out
  float* eig;              // eigenvalue state, d (descending)
  float* a;                // dp x dp working matrix (pitch dp)
  float* zt;               // dp x dp accumulated eigenvectors, one per ROW (pitch dp)
  float* t;                // d x d scratch (pitch d)
  float* j;                // two buffers (by round parity) of the dp / 64 rotations of a
                           // round, 64 x 64 row-major each
  int32_t* rot;            // two buffers of, per pair of a round: 1 unless its rotation is
                           // the identity
  int32_t* rank;           // d: position of eigenvalue i in descending order
  float* diag_max;         // max_i |a_ii| of the working matrix (refreshed every sweep)
  float tol;               // relative rotation threshold
  int32_t orig;            // index of the side in table order (L of every matrix, then R)
  int32_t d, dp;
};

struct JacobiCtl {
  int32_t converged, rotated, sweeps, pad_;
};

struct MatDev {            // one owned matrix in the flat owner buffers
  int64_t offset, numel;
};

// Pair i of round r of the round-robin ("circle") schedule over n (even) indices: every index
// once per round, every pair once in n - 1 rounds.
__device__ __forceinline__ void circle_pair(int n, int r, int i, int& x, int& y) {
  if (i == 0) {
    x = n - 1;
    y = r;
  } else {
    x = (r + i) % (n - 1);
    y = (r - i + (n - 1)) % (n - 1);
  }
}

// Global index of local index c (0..63) of pair-block p in round r.
__device__ __forceinline__ int pair_index(int nb, int r, int p, int c) {
  int b0, b1;
  circle_pair(nb, r, p, b0, b1);
  return (c < kJB ? b0 : b1) * kJB + (c & (kJB - 1));
}

// The pair of round r that holds block x, and x's partner in it (inverse of circle_pair).
__device__ __forceinline__ int pair_of(int nb, int r, int x) {
  const int m = nb - 1, half = nb / 2;
  if (x == nb - 1 || x == r) return 0;
  int d = x - r;
  if (d < 0) d += m;
  return d <= half - 1 ? d : m - d;
}
__device__ __forceinline__ int partner_of(int nb, int r, int x) {
  int a, b;
  circle_pair(nb, r, pair_of(nb, r, x), a, b);
  return a == x ? b : a;
}

// The side whose range [begin[k], begin[k + 1]) of a compact grid holds block `bid`.
__device__ __forceinline__ int side_of(const int32_t* begin, int nsides, int bid) {
  int lo = 0, hi = nsides - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (begin[mid] <= bid) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Z^T = Q^T padded with the identity, A's padding = 0, the solve's control words reset.
__global__ void jacobi_setup_kernel(const SideDev* sides, JacobiCtl* ctl) {
  const SideDev s = sides[blockIdx.y];
  const int64_t n = (int64_t)s.dp * s.dp;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(e / s.dp), c = (int)(e % s.dp);
    const bool in = r < s.d && c < s.d;
    s.zt[e] = in ? s.q[(int64_t)c * s.d + r] : (r == c ? 1.f : 0.f);
    if (!in) s.a[e] = 0.f;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) ctl[blockIdx.y] = JacobiCtl{0, 0, 0, 0};
}

// max_i |a_ii|: a lower bound of ||L||_2 that is tight once A is nearly diagonal, so it is
// refreshed after every sweep (converged sides keep theirs).
__global__ void __launch_bounds__(1024) diag_max_kernel(const SideDev* sides,
                                                        const JacobiCtl* ctl) {
  __shared__ float red[1024];
  const SideDev s = sides[blockIdx.x];
  if (ctl && ctl[blockIdx.x].converged) return;
  float m = 0.f;
  for (int i = threadIdx.x; i < s.d; i += blockDim.x)
    m = fmaxf(m, fabsf(s.a[(int64_t)i * s.dp + i]));
  red[threadIdx.x] = m;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] = fmaxf(red[threadIdx.x], red[threadIdx.x + o]);
    __syncthreads();
  }
  if (threadIdx.x == 0) *s.diag_max = red[0];
}

// out (64 x 64, registers: rows ty + 16 ii, columns tx + 16 jj) = op(X) Y with
// op(X)[i][k] = X[k][i] (XT) or X[i][k].
template <bool XT>
__device__ __forceinline__ void mm64(const float (*X)[kJLd], const float (*Y)[kJLd], int ty,
                                     int tx, float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < kJP; ++kk) {
    float xv[4], yv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) xv[i] = XT ? X[kk][ty + 16 * i] : X[ty + 16 * i][kk];
#pragma unroll
    for (int j = 0; j < 4; ++j) yv[j] = Y[kk][tx + 16 * j];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xv[i], yv[j], acc[i][j]);
  }
}

constexpr int kTri = (kJP / 2) * (kJP / 2 + 1) / 2;                // 528 blocks (a, b), a <= b
static_assert(kTri <= kSolveThreads, "one S block per solve thread");
constexpr int kVPer = (kJP * (kJP / 2) + kSolveThreads - 33) / (kSolveThreads - 32);  // V units

// One round's subproblems: CTA (pair, side) diagonalises the 64 x 64 block of its pair.
// Compact grid: blocks [begin[k], begin[k + 1]) are the dp_k / 64 pairs of side k.  Each
// inner round has two phases between block barriers: warp 0 forms the round's 32 rotations
// while warps 1-16 apply the previous round's rotations to V; then every thread rotates one
// 2 x 2 block of S (528 blocks on 17 warps).  V takes each round's rotations in round order,
// so its result does not depend on the overlap.
__global__ void __launch_bounds__(kSolveThreads, 1)
    jacobi_solve_kernel(const SideDev* sides, const int32_t* begin, int nsides, JacobiCtl* ctl,
                        int round, int buf) {
  const int k = side_of(begin, nsides, blockIdx.x);
  const SideDev s = sides[k];
  const int nb = s.dp / kJB;
  if (ctl[k].converged || round >= nb - 1) return;
  __shared__ float S[kJP][kJLd];
  __shared__ float V[kJP][kJLd];
  __shared__ float cs[2][kJP / 2], sn[2][kJP / 2];  // rotations of two rounds
  __shared__ int sweep_rot, any_rot;
  __shared__ int gi[kJP];
  __shared__ uint16_t ptab[(kJP - 1) * (kJP / 2)];  // round r, pair a: p | q << 8, p < q
  __shared__ uint16_t ttab[(kJP / 2) * (kJP / 2 + 1) / 2];  // upper-triangle block: a | b << 8
  const int tid = threadIdx.x, pb = blockIdx.x - begin[k];
  if (tid < kJP) gi[tid] = pair_index(nb, round, pb, tid);
  for (int e = tid; e < (kJP - 1) * (kJP / 2); e += kSolveThreads) {
    int p, q;
    circle_pair(kJP, e / (kJP / 2), e % (kJP / 2), p, q);
    ptab[e] = (uint16_t)(min(p, q) | (max(p, q) << 8));
  }
  for (int e = tid; e < (kJP / 2) * (kJP / 2 + 1) / 2; e += kSolveThreads) {
    int a = 0, rem = e;  // e-th (a, b), a <= b, row by row
    while (rem >= kJP / 2 - a) { rem -= kJP / 2 - a; ++a; }
    ttab[e] = (uint16_t)(a | ((a + rem) << 8));
  }
  __syncthreads();
  for (int e = tid; e < kJP * kJP; e += kSolveThreads) {
    const int r = e / kJP, c = e % kJP;
    S[r][c] = s.a[(int64_t)gi[r] * s.dp + gi[c]];
    V[r][c] = r == c ? 1.f : 0.f;
  }
  const float tol = s.tol * *s.diag_max;
  // this thread's block of S: pair ta rows, pair tb columns (ta <= tb)
  const int tt = tid < kTri ? ttab[tid] : 0, ta = tt & 0xff, tb = tt >> 8;
  if (tid == 0) any_rot = 0;
  for (int sw = 0; sw < kSubSweeps; ++sw) {
    __syncthreads();  // every thread has read the previous sweep's flag
    if (tid == 0) sweep_rot = 0;
    __syncthreads();
    // V <- V J of the round `vr` (its rotations in buffer vr & 1) by warps 1-16, 2048 units
    // (row i, pair a) over the other 512 threads: the update of V runs beside the next round's
    // rotations (warp 0) instead of on the path between the two barriers of a round
    auto rotate_v = [&](int vr) {
      const uint16_t* pr = ptab + vr * (kJP / 2);
      const float* c_ = cs[vr & 1];
      const float* s_ = sn[vr & 1];
      const int kx = tid - 32;
      float vv[kVPer][2], vc[kVPer][2];
      int vidx[kVPer][2];
      bool va[kVPer];
#pragma unroll
      for (int u = 0; u < kVPer; ++u) {
        const int e = kx + u * (kSolveThreads - 32);
        va[u] = e < kJP * (kJP / 2);
        if (!va[u]) continue;
        const int i = e % kJP, a = e / kJP;
        const int pa = pr[a], p = pa & 0xff, p2 = pa >> 8;
        vc[u][0] = c_[a]; vc[u][1] = s_[a];
        vidx[u][0] = i * kJLd + p; vidx[u][1] = i * kJLd + p2;
        vv[u][0] = (&V[0][0])[vidx[u][0]];
        vv[u][1] = (&V[0][0])[vidx[u][1]];
      }
#pragma unroll
      for (int u = 0; u < kVPer; ++u) {
        if (!va[u]) continue;
        const float ca = vc[u][0], sa = vc[u][1];
        if (sa == 0.f) continue;
        (&V[0][0])[vidx[u][0]] = ca * vv[u][0] - sa * vv[u][1];
        (&V[0][0])[vidx[u][1]] = sa * vv[u][0] + ca * vv[u][1];
      }
    };
    int vpend = -1;  // the round whose rotations V has still to take
    for (int r = 0; r < kJP - 1; ++r) {
      int rotate = 0;
      if (tid < kJP / 2) {
        const int pq = ptab[r * (kJP / 2) + tid], p = pq & 0xff, q = pq >> 8;
        const float app = S[p][p], aqq = S[q][q], apq = S[p][q];
        float c = 1.f, sv = 0.f;
        if (fabsf(apq) > tol) {
          // the rotation that zeroes a_pq (symmetric Schur decomposition of the 2 x 2 block)
          const float tau = (aqq - app) / (2.f * apq);
          const float t = (tau >= 0.f ? 1.f : -1.f) / (fabsf(tau) + sqrtf(1.f + tau * tau));
          c = 1.f / sqrtf(1.f + t * t);
          sv = t * c;
          sweep_rot = 1;
        }
        cs[r & 1][tid] = c;
        sn[r & 1][tid] = sv;
        rotate = sv != 0.f;
      } else if (vpend >= 0) {
        rotate_v(vpend);
      }
      vpend = -1;
      // an inner round that rotates no pair leaves S and V as they are: skip its update (and
      // its second barrier); common once the subproblem is nearly diagonal
      if (!__syncthreads_or(rotate)) continue;
      // S <- J^T S J over the 2 x 2 blocks (pair a rows, pair b columns), a <= b, mirrored
      // (S stays symmetric): all disjoint, one per thread.
      if (tid < kTri) {
        const uint16_t* pr = ptab + r * (kJP / 2);
        const int pa = pr[ta], pb = pr[tb];
        const int p = pa & 0xff, p2 = pa >> 8, q = pb & 0xff, q2 = pb >> 8;
        const float ca = cs[r & 1][ta], sa = sn[r & 1][ta];
        const float cb = cs[r & 1][tb], sb = sn[r & 1][tb];
        const float x11 = S[p][q], x12 = S[p][q2], x21 = S[p2][q], x22 = S[p2][q2];
        if (sa != 0.f || sb != 0.f) {
          const float y11 = ca * x11 - sa * x21, y12 = ca * x12 - sa * x22;
          const float y21 = sa * x11 + ca * x21, y22 = sa * x12 + ca * x22;
          const float z11 = cb * y11 - sb * y12, z12 = sb * y11 + cb * y12;
          const float z21 = cb * y21 - sb * y22, z22 = sb * y21 + cb * y22;
          if (ta == tb) {
            S[p][q] = z11;
            S[p][q2] = 0.f;  // the coupling this rotation removes
            S[p2][q] = 0.f;
            S[p2][q2] = z22;
          } else {
            // block (a, b) and its mirror (b, a)
            S[p][q] = z11; S[p][q2] = z12; S[p2][q] = z21; S[p2][q2] = z22;
            S[q][p] = z11; S[q2][p] = z12; S[q][p2] = z21; S[q2][p2] = z22;
          }
        }
      }
      vpend = r;
      __syncthreads();
    }
    if (vpend >= 0) {
      if (tid >= 32) rotate_v(vpend);
      __syncthreads();
    }
    const bool more = sweep_rot != 0;
    if (tid == 0 && more) any_rot = 1;
    if (!more) break;
  }
  __syncthreads();
  if (any_rot) {
    // one polar (Newton–Schulz) step, V <- V (3I - V^T V) / 2: the rotations' rounding leaves
    // V^T V = I + E with |E| ~ 1e-5 (a bias of ~1e-8 per rotation in c^2 + s^2), the step
    // leaves O(E^2)
    // (the first 256 threads compute, 4 x 4 outputs each)
    const int ty = (tid >> 4) & 15, tx = tid & 15;
    const bool worker = tid < 256;
    float acc[4][4];
    if (worker) {
      mm64<true>(V, V, ty, tx, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = ty + 16 * i, c = tx + 16 * j;
          S[r][c] = ((r == c ? 3.f : 0.f) - acc[i][j]) * 0.5f;
        }
    }
    __syncthreads();
    if (worker) mm64<false>(V, S, ty, tx, acc);
    __syncthreads();
    if (worker) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) V[ty + 16 * i][tx + 16 * j] = acc[i][j];
    }
    __syncthreads();
  }
  const int nbp = s.dp / kJP;  // pairs of a round
  float* jout = s.j + ((int64_t)buf * nbp + pb) * kJP * kJP;
  for (int e = tid; e < kJP * kJP; e += kSolveThreads) jout[e] = V[e / kJP][e % kJP];
  if (tid == 0) {
    s.rot[buf * nbp + pb] = any_rot;
    if (any_rot) ctl[k].rotated = 1;
  }
}

constexpr int kALd = kJP + 4;  // apply kernel's shared-memory pitch: rows 16-byte aligned
constexpr size_t kApplySmem = 3 * sizeof(float) * kJP * kALd;  // 4 CTAs per SM

// acc = P^T Q over a 64 x 64 tile, acc[i][j] = sum_k P[k][4ty + i] Q[k][col_j] with one fmaf
// per k in increasing k; thread (ty, tx), ty in [0, 16), tx in [0, 8), owns rows 4ty .. + 3
// and columns col_j = 4tx + j (j < 4) and 32 + 4tx + j - 4 (j >= 4).  Each k reads three
// 128-bit words per thread for 32 FMAs: per warp one 64-byte P row segment (four ty) and two
// 128-byte Q row segments.
__device__ __forceinline__ int col8(int tx, int j) { return (j < 4 ? 4 * tx : 28 + 4 * tx) + j; }
__device__ __forceinline__ void mm64_tn(const float (*P)[kALd], const float (*Q)[kALd], int ty,
                                        int tx, float (&acc)[4][8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < kJP; ++kk) {
    const float4 pv = *reinterpret_cast<const float4*>(&P[kk][4 * ty]);
    const float4 q0 = *reinterpret_cast<const float4*>(&Q[kk][4 * tx]);
    const float4 q1 = *reinterpret_cast<const float4*>(&Q[kk][32 + 4 * tx]);
    const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
    const float qa[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(pa[i], qa[j], acc[i][j]);
  }
}

constexpr int kZCols = 512;  // columns of Z^T one rotation CTA updates with the same J_p

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 64 x 64 block of a row-major global matrix (pitch ld) into shared memory: rows rowi(r),
// columns coli(c), 4 consecutive columns at a time (they never straddle a 32-block).  The
// copies are asynchronous (16-byte cp.async): the caller commits and waits for them.
template <typename RowF, typename ColF>
__device__ __forceinline__ void load_block(float (*dst)[kALd], const float* src, int64_t ld,
                                           RowF rowi, ColF coli) {
  for (int e = threadIdx.x; e < kJP * kJP / 4; e += kJThreads) {
    const int r = e / (kJP / 4), c = (e % (kJP / 4)) * 4;
    cp_async16(&dst[r][c], src + (int64_t)rowi(r) * ld + coli(c));
  }
}

// The round's rotations applied to A, one CTA per block pair (p, q), p <= q: Y = Jp^T (A_pq
// Jq), with A_pq Jq formed from the mirrored block (A is symmetric), Y written to (p, q) and
// Y^T to (q, p).  A CTA loads A_pq and Jq as one copy group and Jp as a second, which lands
// while W = A_pq Jq is formed.  (Z^T's rows take the same rotations in jacobi_zrot_tc_kernel.)
// The next round's subproblems read only the block pairs of `critical` CTAs: (p, p) for
// every p, and for every pair of the next round (blocks x, y) the CTA of this round's pairs
// of x and y.  Part 1 (compact grid of 2P blocks per side) runs those; part 2 (the triangle of
// P(P + 1) / 2 per side) runs the others, beside the next round's subproblems.
__device__ __forceinline__ bool critical_pair(int nb, int round, int p, int q) {
  if (p == q) return true;
  const int rn = round + 1 == nb - 1 ? 0 : round + 1;
  int b0, b1;
  circle_pair(nb, round, p, b0, b1);
  return pair_of(nb, round, partner_of(nb, rn, b0)) == q ||
         pair_of(nb, round, partner_of(nb, rn, b1)) == q;
}
__global__ void __launch_bounds__(kJThreads) jacobi_apply_kernel(const SideDev* sides,
                                                                 const int32_t* begin,
                                                                 int nsides,
                                                                 const JacobiCtl* ctl,
                                                                 int round, int buf, int part) {
  const int k = side_of(begin, nsides, blockIdx.x);
  const SideDev s = sides[k];
  const int nb = s.dp / kJB, P = nb / 2;
  if (ctl[k].converged || round >= nb - 1) return;
  const int bid = blockIdx.x - begin[k];
  const float* jb = s.j + (int64_t)buf * P * kJP * kJP;
  const int32_t* rb = s.rot + buf * P;
  extern __shared__ __align__(16) float smem[];
  float (*B0)[kALd] = reinterpret_cast<float (*)[kALd]>(smem);
  float (*B1)[kALd] = B0 + kJP;
  float (*B2)[kALd] = B1 + kJP;
  __shared__ int ip[kJP], iq[kJP];  // global indices of the two pair-blocks
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  float acc[4][8];
  int p = 0, q = 0;
  if (part == 1) {
    if (bid < P) {
      p = q = bid;
    } else {
      // the CTA of next-round pair pp (blocks x, y); of two next-round pairs that meet the
      // same two pairs of this round, the lower one runs it
      const int pp = bid - P, rn = round + 1 == nb - 1 ? 0 : round + 1;
      int x, y;
      circle_pair(nb, rn, pp, x, y);
      const int px = pair_of(nb, round, x), py = pair_of(nb, round, y);
      if (px == py) return;
      const int x2 = partner_of(nb, round, x), p2 = pair_of(nb, rn, x2);
      if (p2 < pp && pair_of(nb, round, partner_of(nb, rn, x2)) == py) return;
      p = min(px, py);
      q = max(px, py);
    }
  } else {
    int rem = bid;
    while (rem >= P - p) { rem -= P - p; ++p; }
    q = p + rem;
    if (part == 2 && critical_pair(nb, round, p, q)) return;
  }
  if (!rb[p] && !rb[q]) return;
  if (tid < kJP) ip[tid] = pair_index(nb, round, p, tid);
  else if (tid < 2 * kJP) iq[tid - kJP] = pair_index(nb, round, q, tid - kJP);
  __syncthreads();
  auto idx = [&](int pb, int c) { return pb == p ? ip[c] : iq[c]; };
  const float* jp = jb + (int64_t)p * kJP * kJP;
  const float* jq = jb + (int64_t)q * kJP * kJP;
  // B0[k][i] = A[I_q(k)][I_p(i)] = A_pq[i][k]
  load_block(B0, s.a, s.dp, [&](int r) { return idx(q, r); }, [&](int c) { return idx(p, c); });
  load_block(B2, jq, kJP, [](int r) { return r; }, [](int c) { return c; });
  cp_async_commit();
  load_block(B1, jp, kJP, [](int r) { return r; }, [](int c) { return c; });
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();
  mm64_tn(B0, B2, ty, tx, acc);  // W = A_pq Jq
  __syncthreads();               // B0 is free: W goes there
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    *reinterpret_cast<float4*>(&B0[4 * ty + i][4 * tx]) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(&B0[4 * ty + i][32 + 4 * tx]) =
        make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
  cp_async_wait<0>();
  __syncthreads();
  mm64_tn(B1, B0, ty, tx, acc);  // Y = Jp^T W
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* row = s.a + (int64_t)idx(p, 4 * ty + i) * s.dp;
    *reinterpret_cast<float4*>(row + idx(q, 4 * tx)) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    *reinterpret_cast<float4*>(row + idx(q, 32 + 4 * tx)) =
        make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
  if (p != q) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int gr = idx(q, col8(tx, j)), gc = idx(p, 4 * ty);
      *reinterpret_cast<float4*>(s.a + (int64_t)gr * s.dp + gc) =
          make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
    }
  }
}

// ---------------------------------------------------------------- Z^T rotations, tensor cores
// Z^T <- J_p^T Z^T over the rows I_p of a pair, as D = A B^T on tcgen05 (kind::tf32) with
// A[c][k] = Z^T[I_p(k)][c0 + c] (128 columns of Z^T: the MMA's M) and B[i][k] = J_p[k][i]
// (N = 64), K = 64 in two 32-wide k-blocks (the two 32-row halves of I_p).  fp32 accuracy
// as in the batched GEMM: every operand value x is split into hi = x with its 13 low mantissa
// bits cleared and lo = x - hi, each k-block forms hi*hi + hi*lo + lo*hi (12 MMAs) in a TMEM
// accumulator of its own, and the two k-block partials are added in fp32 registers.  The
// operands are MN-major in memory; 128 threads copy 4 x 4 blocks into the 128-byte-swizzled
// K-major layout the MMA reads and transpose them in registers while splitting.
namespace ztc {

constexpr int kM = 128, kN = 64, kK = 32;           // MMA tile, k-block
constexpr int kGroups = kZCols / 128;               // 128-column groups per CTA
constexpr uint32_t kATile = kM * kK * 4;            // 16 KB per k-block
constexpr uint32_t kBTile = kN * kK * 4;            // 8 KB per k-block
constexpr uint32_t kAHi = 0, kALo = 2 * kATile;     // A: [hi kb0 | hi kb1 | lo kb0 | lo kb1]
constexpr uint32_t kBHi = 4 * kATile, kBLo = kBHi + 2 * kBTile;
constexpr uint32_t kBarOff = kBLo + 2 * kBTile;     // 96 KB
constexpr size_t kSmem = 1024 + kBarOff + 64;
constexpr uint32_t kTmemCols = 2 * kN;              // one accumulator per k-block
// kind::tf32: fp32 accumulator (bit 4), TF32 A and B (2 at bits 7 and 10), both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kM >> 4) << 24);
static_assert(kSmem <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `parity`; false when the limit ran out.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  for (uint32_t i = 1;; ++i) {
    if (try_wait(bar, parity)) return true;
    if ((i & 31) == 0 && now_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
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
// K-major operand in the 128-byte-swizzled layout: rows of 32 fp32 (128 B), 8-row atoms
// 1024 B apart (stride offset), leading offset unused (16 B), version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t kdesc(uint32_t s) {
  return (uint64_t)((s >> 4) & 0x3FFFu) | ((uint64_t)(16u >> 4) << 16) |
         ((uint64_t)(1024u >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Byte offset of (row r, k) in a K-major 32-wide tile: 16-byte chunk k / 4 of row r at chunk
// (k / 4) ^ (r % 8).
__device__ __forceinline__ uint32_t toff(int r, int k) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((((k >> 2) ^ (r & 7)) & 7) << 4) +
                    (k & 3) * 4);
}
__device__ __forceinline__ void cp16(uint32_t dst, const float* src, int bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ float4 lds4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts4(uint32_t a, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void split(float x, float& hi, float& lo) {
  hi = __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
  lo = x - hi;
}
// The 4 x 4 block of rows 4 rq .. + 3 and k 4 kq .. + 3 of an MN-major source (element
// (r, k) at src[k * ld + r]), `avail` rows of it inside (the rest zero), copied one k-row at a
// time into the places the block's four rows take in the K-major tile at s_lo.
__device__ __forceinline__ void issue_block(const float* src, int64_t ld, int rq, int kq,
                                            int avail, uint32_t s_lo) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float* g = src + (int64_t)(4 * kq + i) * ld + 4 * rq;
    cp16(s_lo + toff(4 * rq + i, 4 * kq), avail > 0 ? g : src, avail >= 4 ? 16 : 0);
  }
}
// Transpose the block in registers and split it: hi to s_hi, lo over the raw values.
__device__ __forceinline__ void convert_block(int rq, int kq, uint32_t s_hi, uint32_t s_lo) {
  float4 y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = lds4(s_lo + toff(4 * rq + i, 4 * kq));
  const float v[4][4] = {{y[0].x, y[1].x, y[2].x, y[3].x}, {y[0].y, y[1].y, y[2].y, y[3].y},
                         {y[0].z, y[1].z, y[2].z, y[3].z}, {y[0].w, y[1].w, y[2].w, y[3].w}};
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float4 h, l;
    split(v[r][0], h.x, l.x);
    split(v[r][1], h.y, l.y);
    split(v[r][2], h.z, l.z);
    split(v[r][3], h.w, l.w);
    const uint32_t off = toff(4 * rq + r, 4 * kq);
    sts4(s_hi + off, h);
    sts4(s_lo + off, l);
  }
}

}  // namespace ztc

// One CTA of 128 threads per (pair p of a side, 512 columns of Z^T): J_p is split once, then
// four 128-column groups go through copy, split, 24 MMAs and the epilogue, the next group's
// copies flying while the current one's results are stored.  Compact grid: blocks
// [begin[k], begin[k + 1]) of side k, block c P + p for pair p and columns 512 c .. + 511.
// Every wait is bounded: on a timeout the CTA records it in the status word, waits (bounded)
// for its MMAs, frees its tensor memory and returns.
__global__ void __launch_bounds__(128) jacobi_zrot_tc_kernel(const SideDev* sides,
                                                             const int32_t* begin, int nsides,
                                                             const JacobiCtl* ctl, int round,
                                                             int buf, uint64_t limit_ns,
                                                             int* status) {
  using namespace ztc;
  const int k = side_of(begin, nsides, blockIdx.x);
  const SideDev s = sides[k];
  const int nb = s.dp / kJB, P = nb / 2;
  if (ctl[k].converged || round >= nb - 1) return;
  const int bid = blockIdx.x - begin[k], cgrp = bid / P, p = bid % P;
  if (!s.rot[buf * P + p]) return;
  int b0, b1;
  circle_pair(nb, round, p, b0, b1);
  const float* jp = s.j + ((int64_t)buf * P + p) * kJP * kJP;
  const int ngroups = (s.dp + kM - 1) / kM;
  const int g0 = cgrp * kGroups, g1 = min(ngroups, g0 + kGroups);
  if (g0 >= g1) return;

  extern __shared__ uint8_t zsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(zsm_raw) + 1023) &
                                           ~uintptr_t(1023));
  const uint32_t sb = saddr(sm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kBarOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  const uint32_t mbar = saddr(bar);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     saddr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // this thread's 4 x 4 blocks: B (64 rows i): one per k-block; A (128 rows c): two
  const int l = tid & 31, kq = l & 7;
  const int rq_b = 4 * (tid >> 5) + (l >> 3);                     // 0 .. 15
  auto rq_a = [&](int u) { return 4 * (4 * u + (tid >> 5)) + (l >> 3); };  // 0 .. 31
  // B[i][k] = J_p[k][i]: k-block kb holds J_p rows 32 kb .. + 31
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
    issue_block(jp + (int64_t)(kK * kb) * kJP, kJP, rq_b, kq, 4, sb + kBLo + kb * kBTile);
  // A[c][k] = Z^T[I_p(k)][c0 + c]: k-block kb holds the rows of block b_kb
  auto issue_a = [&](int grp) {
    const int c0 = grp * kM;
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      const float* src = s.zt + (int64_t)(kJB * (kb ? b1 : b0)) * s.dp + c0;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int rq = rq_a(u);
        issue_block(src, s.dp, rq, kq, s.dp - (c0 + 4 * rq), sb + kALo + kb * kATile);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  issue_a(g0);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  uint32_t phase = 0;
  for (int grp = g0; grp < g1; ++grp) {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    if (grp == g0) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
        convert_block(rq_b, kq, sb + kBHi + kb * kBTile, sb + kBLo + kb * kBTile);
    }
#pragma unroll
    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
      for (int u = 0; u < 2; ++u)
        convert_block(rq_a(u), kq, sb + kAHi + kb * kATile, sb + kALo + kb * kATile);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
    fence_before();
    __syncthreads();
    fence_after();
    if (tid == 0) {
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
        const uint32_t d = tmem + (uint32_t)(kb * kN);
        const uint32_t ah = sb + kAHi + kb * kATile, al = sb + kALo + kb * kATile;
        const uint32_t bh = sb + kBHi + kb * kBTile, bl = sb + kBLo + kb * kBTile;
#pragma unroll
        for (int j = 0; j < kK / 8; ++j) {
          mma(d, kdesc(ah + 32u * j), kdesc(bh + 32u * j), j != 0);
          mma(d, kdesc(ah + 32u * j), kdesc(bl + 32u * j), 1u);
          mma(d, kdesc(al + 32u * j), kdesc(bh + 32u * j), 1u);
        }
      }
      commit(mbar);
    }
    if (!wait_bar(mbar, phase, limit_ns)) {
      atomicOr(status, kStatusTimeout);
      ok = false;
    }
    phase ^= 1u;
    fence_after();
    // A's buffers are free once the MMAs completed: the next group's copies fly while this
    // group's results are stored
    if (ok && grp + 1 < g1) issue_a(grp + 1);
    if (ok) {
      const int c = grp * kM + 32 * warp + lane;  // this thread's TMEM lane = column of Z^T
      const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
      for (int q = 0; q < kN / 16; ++q) {
        float v0[16], v1[16];
        tmem_ld16(ta + (uint32_t)(16 * q), v0);
        tmem_ld16(ta + (uint32_t)(kN + 16 * q), v1);
        if (c < s.dp) {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = 16 * q + e;  // output row I_p(i)
            const int row = (i < kJB ? b0 : b1) * kJB + (i & (kJB - 1));
            s.zt[(int64_t)row * s.dp + c] = v0[e] + v1[e];
          }
        }
      }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (!__syncthreads_and(ok)) break;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (!ok && tid == 0) wait_bar(mbar, phase ^ 1u, limit_ns);  // MMAs still in flight
  fence_before();
  __syncthreads();
  if (warp == 0) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}


// End of a sweep: a side whose sweep rotated nothing is converged.
__global__ void jacobi_sweep_end_kernel(JacobiCtl* ctl, int nsides) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= nsides) return;
  JacobiCtl c = ctl[k];
  if (!c.converged) {
    ++c.sweeps;
    if (!c.rotated) c.converged = 1;
  }
  c.rotated = 0;
  ctl[k] = c;
}

// The condition of a group's sweep loop when the sweeps run as a CUDA graph: go on while a
// side is unconverged and under the sweep limit.
__global__ void jacobi_loop_kernel(const JacobiCtl* ctl, int nsides, int max_sweeps,
                                   cudaGraphConditionalHandle handle) {
  int more = 0;
  for (int k = threadIdx.x; k < nsides; k += blockDim.x)
    more |= (!ctl[k].converged && ctl[k].sweeps < max_sweeps) ? 1 : 0;
  more = __syncthreads_or(more);
  if (threadIdx.x == 0) cudaGraphSetConditional(handle, more ? 1u : 0u);
}

// Rayleigh quotients of the final basis: lambda_i = z_i^T L z_i / z_i^T z_i, with T = Z^T L
// (rows z_i^T L) formed by the SGEMM; one warp per eigenvector.  They replace diag(A), whose
// entries carry the rounding of every rotation applied to A.
__global__ void rayleigh_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.y];
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int i = warp; i < s.d; i += nw) {
    const float* z = s.zt + (int64_t)i * s.dp;
    const float* t = s.t + (int64_t)i * s.d;
    float nf = 0.f, df = 0.f;  // per lane: d / 32 terms in fp32, then the lanes in fp64
    for (int c = lane; c < s.d; c += 32) {
      nf = fmaf(t[c], z[c], nf);
      df = fmaf(z[c], z[c], df);
    }
    double num = nf, den = df;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      num += __shfl_xor_sync(0xffffffffu, num, o);
      den += __shfl_xor_sync(0xffffffffu, den, o);
    }
    if (lane == 0) s.a[(int64_t)i * s.dp + i] = (float)(num / den);
  }
}

// rank[i] = position of diag(A)_i in descending order (ties by index); eig[rank[i]] = diag_i.
__global__ void eig_rank_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.y];
  __shared__ float lam[256];
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if ((int)(blockIdx.x * blockDim.x) >= s.d) return;  // block-uniform
  const float li = i < s.d ? s.a[(int64_t)i * s.dp + i] : 0.f;
  int rank = 0;
  for (int j0 = 0; j0 < s.d; j0 += 256) {
    __syncthreads();
    const int jj = j0 + threadIdx.x;
    lam[threadIdx.x] = jj < s.d ? s.a[(int64_t)jj * s.dp + jj] : 0.f;
    __syncthreads();
    const int cnt = min(256, s.d - j0);
    for (int u = 0; u < cnt; ++u) {
      const float lj = lam[u];
      rank += (lj > li || (lj == li && j0 + u < i)) ? 1 : 0;
    }
  }
  if (i < s.d) {
    s.rank[i] = rank;
    s.eig[rank] = li;
  }
}

// Q[r][rank[i]] = Z^T[i][r], through 32 x 32 shared-memory tiles (reads along rows of Z^T,
// writes along rows of Q).
__global__ void eig_scatter_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.z];
  __shared__ float tile[32][33];
  const int i0 = blockIdx.y * 32, r0 = blockIdx.x * 32;
  if (i0 >= s.d || r0 >= s.d) return;  // block-uniform
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8 threads
  for (int u = ty; u < 32; u += 8) {
    const int i = i0 + u, r = r0 + tx;
    tile[u][tx] = (i < s.d && r < s.d) ? s.zt[(int64_t)i * s.dp + r] : 0.f;
  }
  __syncthreads();
  for (int u = ty; u < 32; u += 8) {
    const int r = r0 + u, i = i0 + tx;
    if (r < s.d && i < s.d) s.q[(int64_t)r * s.d + s.rank[i]] = tile[tx][u];
  }
}

// Per-side solve report: sweeps used, negative when the sweep limit was reached first.
__global__ void jacobi_info_kernel(const SideDev* sides, const JacobiCtl* ctl, int nsides,
                                   int32_t* info) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k < nsides) info[sides[k].orig] = ctl[k].converged ? ctl[k].sweeps : -ctl[k].sweeps;
}

// M = b1 M + (1 - b1) G.
__global__ void soap_moment_kernel(const MatDev* mats, float* m, const float* g, float beta1) {
  const MatDev d = mats[blockIdx.y];
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < d.numel;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t o = d.offset + e;
    m[o] = fmaf(beta1, m[o], (1.f - beta1) * g[o]);
  }
}

// In the eigenbasis: V = b2 V + (1 - b2) G'^2; N' = (M' / bc1) / (sqrt(V / bc2) + eps) -> mrot.
__global__ void soap_adam_kernel(const MatDev* mats, const float* grot, float* mrot, float* v,
                                 float beta2, float bc1, float bc2, float eps) {
  const MatDev d = mats[blockIdx.y];
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < d.numel;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t o = d.offset + e;
    const float gr = grot[o];
    const float vn = fmaf(beta2, v[o], (1.f - beta2) * gr * gr);
    v[o] = vn;
    mrot[o] = (mrot[o] / bc1) / (sqrtf(vn / bc2) + eps);
  }
}

// W = W (1 - lr wd) - lr N; a non-finite N sets the device status word (one atomic per warp).
__global__ void soap_update_kernel(const MatDev* mats, float* w, const float* nbuf, float decay,
                                   float lr, int* status) {
  const MatDev d = mats[blockIdx.y];
  bool bad = false;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < d.numel;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t o = d.offset + e;
    bad |= !isfinite(nbuf[o]);
    w[o] = fmaf(w[o], decay, -lr * nbuf[o]);
  }
  if (__any_sync(__activemask(), bad) && (threadIdx.x & 31) == 0)
    atomicOr(status, kStatusNonFinite);
}

// Final polar step of the solve, Z^T <- (3I - Z^T Z) Z^T / 2 on the leading d x d block (the
// padding rows and columns stay the identity): T = 1.5 I here, T = -Z^T Z / 2 + T and
// A = T Z^T by the batched GEMM, then Z^T = A.  Hundreds of rounds of fp32 rotations leave
// Z^T a few 1e-6 from orthogonal; the next step starts from this basis (A = Q^T L Q), where
// that is a perturbation of the eigenproblem.  One step leaves about the square of it.
__global__ void polar_prep_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.y];
  const int64_t n = (int64_t)s.d * s.d;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x)
    s.t[e] = (e / s.d) == (e % s.d) ? 1.5f : 0.f;
}
__global__ void polar_copy_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.y];
  const int64_t n = (int64_t)s.d * s.d;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t at = (e / s.d) * s.dp + e % s.d;
    s.zt[at] = s.a[at];
  }
}

// L = R = 0, Q = I, eigenvalues 0 for every side; M = V = 0 over every matrix.
__global__ void soap_init_side_kernel(const SideDev* sides) {
  const SideDev s = sides[blockIdx.y];
  const int64_t n = (int64_t)s.d * s.d;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    s.stat[e] = 0.f;
    s.q[e] = (e / s.d) == (e % s.d) ? 1.f : 0.f;
    if (e < s.d) s.eig[e] = 0.f;
  }
}

__global__ void soap_zero_kernel(const MatDev* mats, float* m, float* v) {
  const MatDev d = mats[blockIdx.y];
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < d.numel;
       e += (int64_t)gridDim.x * blockDim.x) {
    m[d.offset + e] = 0.f;
    v[d.offset + e] = 0.f;
  }
}

}  // namespace
}  // namespace mfsdp

using namespace mfsdp;

// ------------------------------------------------------------------------------------------
// The owned-matrix set of the SOAP step and its workspace layout.
// ------------------------------------------------------------------------------------------
struct mfsdp_soap_set {
  struct Mat {
    int64_t rows, cols, offset;  // in the flat owner buffers (weights, gradient, M, V)
    int64_t l_off, r_off;        // in the flat L / R (and Q_L / Q_R) state buffers
    int64_t el_off, er_off;      // in the flat eigenvalue state buffers
  };
  struct Side {
    int32_t d, dp;
    size_t a, z, t, j, rot, rank;  // workspace byte offsets
  };
  std::vector<Mat> mats;
  std::vector<Side> sides;         // L of every matrix, then R of every matrix
  int64_t numel = 0, l_numel = 0, r_numel = 0, el_numel = 0, er_numel = 0;
  int32_t dp_max = 0, d_max = 0;
  size_t off_tmp_g = 0, off_tmp_m = 0, off_g_rot = 0, off_m_rot = 0;
  size_t off_dmax = 0, off_ctl = 0, off_tables = 0, table_bytes = 0, ws_bytes = 0;
  // The Jacobi solves run as two independent groups of sides, the second on an internal
  // stream, so that one group's (latency-bound) subproblem launches overlap the other's
  // (throughput-bound) rotation launches.  `order` lists the sides group by group.
  std::vector<int32_t> order;
  int32_t split = 0;             // sides in group 0
  int32_t nb_max_group[2] = {0, 0};
  mutable cudaStream_t aux = nullptr;
  mutable cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // Each group's Z^T rotations run on a stream of their own, a round or two behind its A
  // rotations: ev_j[g][b] marks round rotations written to buffer b, ev_z[g][b] the Z^T
  // rotations that read buffer b done, ev_zjoin[g] the group's last Z^T rotation.
  mutable cudaStream_t zst[2] = {nullptr, nullptr};
  mutable cudaEvent_t ev_j[2][2] = {}, ev_z[2][2] = {}, ev_zjoin[2] = {};
  // A's non-critical block pairs run on a third stream per group, beside the next round's
  // subproblems; ev_rest[g] marks the last of them.
  mutable cudaStream_t rst[2] = {nullptr, nullptr};
  mutable cudaEvent_t ev_rest[2] = {};
  // The sweeps as a CUDA graph: per group a while node whose body is one sweep, so that the
  // sweeps stop on the device once every side of the group has converged (no launches of
  // sweeps that would find every side converged).  Built for one workspace and sweep limit
  // (the kernels' arguments point into the workspace).
  mutable cudaGraphExec_t jgraph = nullptr;
  mutable const void* jgraph_ws = nullptr;
  mutable int jgraph_sweeps = 0;
  mutable bool jgraph_off = false;  // the graph could not be built: issue the sweeps one by one
  ~mfsdp_soap_set() {
    if (jgraph) cudaGraphExecDestroy(jgraph);
    if (aux) cudaStreamDestroy(aux);
    if (ev_fork) cudaEventDestroy(ev_fork);
    if (ev_join) cudaEventDestroy(ev_join);
    for (int g = 0; g < 2; ++g) {
      if (rst[g]) cudaStreamDestroy(rst[g]);
      if (ev_rest[g]) cudaEventDestroy(ev_rest[g]);
      if (zst[g]) cudaStreamDestroy(zst[g]);
      if (ev_zjoin[g]) cudaEventDestroy(ev_zjoin[g]);
      for (int b = 0; b < 2; ++b) {
        if (ev_j[g][b]) cudaEventDestroy(ev_j[g][b]);
        if (ev_z[g][b]) cudaEventDestroy(ev_z[g][b]);
      }
    }
  }
};

namespace {

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

constexpr int kGemmsPerMat = 18;  // stats 2, T 2, A 2, polar 4, Rayleigh 2, into the basis 4,
                                  // back 2

// Device tables of one step, in upload order.
struct SoapTables {
  std::vector<SideDev> sides;
  // compact grids of the two groups: subproblems, A block pairs (all; the critical ones),
  // Z^T row groups
  std::vector<int32_t> solve_begin[2], apply_begin[2], crit_begin[2], zrot_begin[2];
  std::vector<MatDev> mats;
  std::vector<GemmDesc> stats_l, stats_r, t, a, polar1, polar2, ray, rot1, rot2, back1, back2;
};

size_t soap_table_bytes(size_t n) {
  return al256(sizeof(SideDev) * 2 * n) + al256(sizeof(MatDev) * n) +
         8 * al256(sizeof(int32_t) * (2 * n + 1)) + al256(sizeof(GemmDesc) * kGemmsPerMat * n) +
         20 * 256;
}

}  // namespace

extern "C" int mfsdp_soap_set_create(const mfsdp_matrix* mats, int32_t n_mats,
                                     mfsdp_soap_set** out) {
  if (out == nullptr || n_mats < 0 || (n_mats > 0 && mats == nullptr)) return MFSDP_EINVAL;
  auto* s = new mfsdp_soap_set();
  int64_t lo = 0, ro = 0, elo = 0, ero = 0;
  for (int32_t i = 0; i < n_mats; ++i) {
    const mfsdp_matrix& m = mats[i];
    if (m.rows <= 0 || m.cols <= 0 || m.offset < 0 || m.rows > (1 << 16) || m.cols > (1 << 16)) {
      delete s;
      return MFSDP_ESHAPE;
    }
    s->mats.push_back({m.rows, m.cols, m.offset, lo, ro, elo, ero});
    lo += m.rows * m.rows;
    ro += m.cols * m.cols;
    elo += m.rows;
    ero += m.cols;
    s->numel = std::max(s->numel, m.offset + m.rows * m.cols);
  }
  s->l_numel = lo;
  s->r_numel = ro;
  s->el_numel = elo;
  s->er_numel = ero;
  size_t off = 0;
  for (int side = 0; side < 2; ++side)
    for (const auto& m : s->mats) {
      mfsdp_soap_set::Side sd{};
      sd.d = (int32_t)(side == 0 ? m.rows : m.cols);
      sd.dp = (sd.d + 63) / 64 * 64;
      const size_t dp2 = (size_t)sd.dp * sd.dp * sizeof(float);
      sd.a = off; off = al256(off + dp2);
      sd.z = off; off = al256(off + dp2);
      sd.t = off; off = al256(off + (size_t)sd.d * sd.d * sizeof(float));
      sd.j = off; off = al256(off + 2 * (size_t)(sd.dp / 64) * 64 * 64 * sizeof(float));
      sd.rot = off; off = al256(off + 2 * (size_t)(sd.dp / 64) * sizeof(int32_t));
      sd.rank = off; off = al256(off + (size_t)sd.d * sizeof(int32_t));
      s->dp_max = std::max(s->dp_max, sd.dp);
      s->d_max = std::max(s->d_max, sd.d);
      s->sides.push_back(sd);
    }
  {
    // two groups balanced by Jacobi work (~dp^3), largest first (the two largest sides land
    // in different groups)
    std::vector<int32_t> idx(s->sides.size());
    for (size_t k = 0; k < idx.size(); ++k) idx[k] = (int32_t)k;
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t x, int32_t y) {
      return s->sides[(size_t)x].dp > s->sides[(size_t)y].dp;
    });
    double load[2] = {0.0, 0.0};
    std::vector<int> grp(s->sides.size(), 0);
    for (int32_t k : idx) {
      const int g = load[1] < load[0] ? 1 : 0;
      const double dp = s->sides[(size_t)k].dp;
      load[g] += dp * dp * dp;
      grp[(size_t)k] = g;
    }
    for (int g = 0; g < 2; ++g)
      for (size_t k = 0; k < grp.size(); ++k)
        if (grp[k] == g) {
          s->order.push_back((int32_t)k);
          s->nb_max_group[g] = std::max(s->nb_max_group[g], s->sides[k].dp / kJB);
        }
    s->split = (int32_t)std::count(grp.begin(), grp.end(), 0);
  }
  const size_t flat = (size_t)s->numel * sizeof(float);
  s->off_tmp_g = off; off = al256(off + flat);
  s->off_tmp_m = off; off = al256(off + flat);
  s->off_g_rot = off; off = al256(off + flat);
  s->off_m_rot = off; off = al256(off + flat);
  const size_t n = std::max<size_t>(s->mats.size(), 1);
  s->off_dmax = off; off = al256(off + sizeof(float) * 2 * n);
  s->off_ctl = off; off = al256(off + sizeof(JacobiCtl) * 2 * n);
  s->off_tables = off;
  s->table_bytes = soap_table_bytes(n);
  s->ws_bytes = al256(off + s->table_bytes);
  *out = s;
  return MFSDP_OK;
}

extern "C" int mfsdp_soap_set_destroy(mfsdp_soap_set* set) {
  delete set;
  return MFSDP_OK;
}

extern "C" int mfsdp_soap_set_sizes(const mfsdp_soap_set* set, size_t* workspace_bytes,
                                    int64_t* l_numel, int64_t* r_numel, int64_t* eig_l_numel,
                                    int64_t* eig_r_numel) {
  if (set == nullptr) return MFSDP_EINVAL;
  if (workspace_bytes) *workspace_bytes = set->ws_bytes;
  if (l_numel) *l_numel = set->l_numel;
  if (r_numel) *r_numel = set->r_numel;
  if (eig_l_numel) *eig_l_numel = set->el_numel;
  if (eig_r_numel) *eig_r_numel = set->er_numel;
  return MFSDP_OK;
}

namespace {

bool state_ok(const mfsdp_soap_state* st) {
  return st && st->l && st->r && st->q_l && st->q_r && st->eig_l && st->eig_r && st->exp_avg &&
         st->exp_avg_sq;
}

// Side and matrix tables for the given state and workspace.
void soap_fill(const mfsdp_soap_set* set, const mfsdp_soap_state* st, uint8_t* ws, float tol,
               SoapTables& tb) {
  const int n = (int)set->mats.size();
  float* dmax = reinterpret_cast<float*>(ws + set->off_dmax);
  for (int pos = 0; pos < 2 * n; ++pos) {
    const int k = set->order[(size_t)pos];
    const auto& sd = set->sides[(size_t)k];
    const auto& m = set->mats[(size_t)(k % n)];
    const bool left = k < n;
    SideDev d{};
    d.orig = k;
    d.stat = (left ? st->l : st->r) + (left ? m.l_off : m.r_off);
    d.q = (left ? st->q_l : st->q_r) + (left ? m.l_off : m.r_off);
    d.eig = (left ? st->eig_l : st->eig_r) + (left ? m.el_off : m.er_off);
    d.a = reinterpret_cast<float*>(ws + sd.a);
    d.zt = reinterpret_cast<float*>(ws + sd.z);
    d.t = reinterpret_cast<float*>(ws + sd.t);
    d.j = reinterpret_cast<float*>(ws + sd.j);
    d.rot = reinterpret_cast<int32_t*>(ws + sd.rot);
    d.rank = reinterpret_cast<int32_t*>(ws + sd.rank);
    d.diag_max = dmax + k;
    d.d = sd.d;
    d.dp = sd.dp;
    d.tol = tol;
    tb.sides.push_back(d);
  }
  for (const auto& m : set->mats) tb.mats.push_back(MatDev{m.offset, m.rows * m.cols});
  for (int g = 0; g < 2; ++g) {
    const int lo = g ? set->split : 0, hi = g ? 2 * n : set->split;
    int32_t sb = 0, ab = 0, cb = 0, zb = 0;
    for (int pos = lo; pos < hi; ++pos) {
      const int32_t P = set->sides[(size_t)set->order[(size_t)pos]].dp / 64;
      tb.solve_begin[g].push_back(sb);
      tb.apply_begin[g].push_back(ab);
      tb.crit_begin[g].push_back(cb);
      tb.zrot_begin[g].push_back(zb);
      sb += P;
      ab += P * (P + 1) / 2;
      cb += 2 * P;
      zb += P * ((64 * P + kZCols - 1) / kZCols);
    }
    tb.solve_begin[g].push_back(sb);
    tb.apply_begin[g].push_back(ab);
    tb.crit_begin[g].push_back(cb);
    tb.zrot_begin[g].push_back(zb);
  }
}

// Upload `tb`'s vectors back to back (256-byte aligned) and return their device addresses.
template <typename T>
const T* put(std::vector<uint8_t>& host, size_t& at, uint8_t* dev, const std::vector<T>& v) {
  const size_t bytes = v.size() * sizeof(T);
  if (bytes) std::memcpy(host.data() + at, v.data(), bytes);
  const T* p = reinterpret_cast<const T*>(dev + at);
  at += al256(std::max<size_t>(bytes, 1));
  return p;
}

int run_gemms(const std::vector<GemmDesc>& v, const GemmDesc* dev, int ta, int tb,
              cudaStream_t st) {
  return launch_gemm(dev, v.data(), (int)v.size(), ta, tb, st);
}

}  // namespace

extern "C" int mfsdp_soap_init_state(const mfsdp_soap_set* set, const mfsdp_soap_state* state,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (set == nullptr || !state_ok(state)) return MFSDP_EINVAL;
  const int n = (int)set->mats.size();
  if (n == 0) return MFSDP_OK;
  if (workspace == nullptr || workspace_bytes < set->ws_bytes) return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SoapTables tb;
  soap_fill(set, state, ws, kDefaultJacobiTol, tb);
  std::vector<uint8_t> host(set->table_bytes);
  size_t at = 0;
  uint8_t* dev = ws + set->off_tables;
  const SideDev* d_sides = put(host, at, dev, tb.sides);
  const MatDev* d_mats = put(host, at, dev, tb.mats);
  if (cudaMemcpyAsync(dev, host.data(), at, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MFSDP_ECUDA;
  soap_init_side_kernel<<<dim3(64, 2 * (unsigned)n), 256, 0, st>>>(d_sides);
  soap_zero_kernel<<<dim3(64, (unsigned)n), 256, 0, st>>>(d_mats, state->exp_avg,
                                                          state->exp_avg_sq);
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}

extern "C" int mfsdp_soap_step(const mfsdp_soap_set* set, const float* grad, float* weights,
                               const mfsdp_soap_state* state, int64_t t,
                               const mfsdp_soap_hyper* h, int32_t* info, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (set == nullptr || grad == nullptr || weights == nullptr || !state_ok(state) ||
      h == nullptr)
    return MFSDP_EINVAL;
  if (t < 1 || h->max_sweeps < 1 || h->max_sweeps > 100 || !(h->eps >= 0.f) ||
      !(h->beta1 >= 0.f && h->beta1 < 1.f) || !(h->beta2 >= 0.f && h->beta2 < 1.f) ||
      !(h->beta_stats >= 0.f && h->beta_stats < 1.f) ||
      !(h->jacobi_tol >= 0.f && h->jacobi_tol < 1e-2f) || (h->refresh != 0 && h->refresh != 1))
    return MFSDP_EINVAL;
  const int n = (int)set->mats.size();
  if (n == 0) return MFSDP_OK;
  if (workspace == nullptr || workspace_bytes < set->ws_bytes) return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* tmp_g = reinterpret_cast<float*>(ws + set->off_tmp_g);
  float* tmp_m = reinterpret_cast<float*>(ws + set->off_tmp_m);
  float* g_rot = reinterpret_cast<float*>(ws + set->off_g_rot);
  float* m_rot = reinterpret_cast<float*>(ws + set->off_m_rot);
  JacobiCtl* ctl = reinterpret_cast<JacobiCtl*>(ws + set->off_ctl);

  SoapTables tb;
  soap_fill(set, state, ws, h->jacobi_tol > 0.f ? h->jacobi_tol : kDefaultJacobiTol, tb);
  const float bs = h->beta_stats;
  for (int i = 0; i < n; ++i) {
    const auto& m = set->mats[(size_t)i];
    const int rows = (int)m.rows, cols = (int)m.cols;
    const int64_t o = m.offset;
    float* l = state->l + m.l_off;
    float* r = state->r + m.r_off;
    float* ql = state->q_l + m.l_off;
    float* qr = state->q_r + m.r_off;
    float* tl = reinterpret_cast<float*>(ws + set->sides[(size_t)i].t);
    float* tr = reinterpret_cast<float*>(ws + set->sides[(size_t)(n + i)].t);
    float* al = reinterpret_cast<float*>(ws + set->sides[(size_t)i].a);
    float* ar = reinterpret_cast<float*>(ws + set->sides[(size_t)(n + i)].a);
    const int dpl = set->sides[(size_t)i].dp, dpr = set->sides[(size_t)(n + i)].dp;
    // L = bs L + (1 - bs) G G^T;  R = bs R + (1 - bs) G^T G
    tb.stats_l.push_back({grad + o, grad + o, l, nullptr, rows, rows, cols, cols, cols, rows,
                          1.f - bs, bs});
    tb.stats_r.push_back({grad + o, grad + o, r, nullptr, cols, cols, rows, cols, cols, cols,
                          1.f - bs, bs});
    // T = L Q;  A = Q^T T  (the statistics in the previous basis)
    tb.t.push_back({l, ql, tl, nullptr, rows, rows, rows, rows, rows, rows, 1.f, 0.f});
    tb.t.push_back({r, qr, tr, nullptr, cols, cols, cols, cols, cols, cols, 1.f, 0.f});
    tb.a.push_back({ql, tl, al, nullptr, rows, rows, rows, rows, rows, dpl, 1.f, 0.f});
    tb.a.push_back({qr, tr, ar, nullptr, cols, cols, cols, cols, cols, dpr, 1.f, 0.f});
    // after the solve: T = Z^T L (rows z_i^T L) for the Rayleigh quotients
    float* ztl = reinterpret_cast<float*>(ws + set->sides[(size_t)i].z);
    float* ztr = reinterpret_cast<float*>(ws + set->sides[(size_t)(n + i)].z);
    // the polar step: T = -Z^T Z / 2 + T (T = 1.5 I), then A = T Z^T
    tb.polar1.push_back({ztl, ztl, tl, nullptr, rows, rows, rows, dpl, dpl, rows, -0.5f, 1.f});
    tb.polar1.push_back({ztr, ztr, tr, nullptr, cols, cols, cols, dpr, dpr, cols, -0.5f, 1.f});
    tb.polar2.push_back({tl, ztl, al, nullptr, rows, rows, rows, rows, dpl, dpl, 1.f, 0.f});
    tb.polar2.push_back({tr, ztr, ar, nullptr, cols, cols, cols, cols, dpr, dpr, 1.f, 0.f});
    tb.ray.push_back({ztl, l, tl, nullptr, rows, rows, rows, dpl, rows, rows, 1.f, 0.f});
    tb.ray.push_back({ztr, r, tr, nullptr, cols, cols, cols, dpr, cols, cols, 1.f, 0.f});
    // into the new basis: Q_L^T G, Q_L^T M, then times Q_R
    tb.rot1.push_back({ql, grad + o, tmp_g + o, nullptr, rows, cols, rows, rows, cols, cols,
                       1.f, 0.f});
    tb.rot1.push_back({ql, state->exp_avg + o, tmp_m + o, nullptr, rows, cols, rows, rows, cols,
                       cols, 1.f, 0.f});
    tb.rot2.push_back({tmp_g + o, qr, g_rot + o, nullptr, rows, cols, cols, cols, cols, cols,
                       1.f, 0.f});
    tb.rot2.push_back({tmp_m + o, qr, m_rot + o, nullptr, rows, cols, cols, cols, cols, cols,
                       1.f, 0.f});
    // back out: Q_L N', then times Q_R^T (N into g_rot)
    tb.back1.push_back({ql, m_rot + o, tmp_g + o, nullptr, rows, cols, rows, rows, cols, cols,
                        1.f, 0.f});
    tb.back2.push_back({tmp_g + o, qr, g_rot + o, nullptr, rows, cols, cols, cols, cols, cols,
                        1.f, 0.f});
  }
  std::vector<uint8_t> host(set->table_bytes);
  size_t at = 0;
  uint8_t* dev = ws + set->off_tables;
  const SideDev* d_sides = put(host, at, dev, tb.sides);
  const MatDev* d_mats = put(host, at, dev, tb.mats);
  const int32_t* d_solve_begin[2] = {put(host, at, dev, tb.solve_begin[0]),
                                      put(host, at, dev, tb.solve_begin[1])};
  const int32_t* d_apply_begin[2] = {put(host, at, dev, tb.apply_begin[0]),
                                      put(host, at, dev, tb.apply_begin[1])};
  const int32_t* d_zrot_begin[2] = {put(host, at, dev, tb.zrot_begin[0]),
                                     put(host, at, dev, tb.zrot_begin[1])};
  const int32_t* d_crit_begin[2] = {put(host, at, dev, tb.crit_begin[0]),
                                     put(host, at, dev, tb.crit_begin[1])};
  const GemmDesc* d_stats_l = put(host, at, dev, tb.stats_l);
  const GemmDesc* d_stats_r = put(host, at, dev, tb.stats_r);
  const GemmDesc* d_t = put(host, at, dev, tb.t);
  const GemmDesc* d_a = put(host, at, dev, tb.a);
  const GemmDesc* d_polar1 = put(host, at, dev, tb.polar1);
  const GemmDesc* d_polar2 = put(host, at, dev, tb.polar2);
  const GemmDesc* d_ray = put(host, at, dev, tb.ray);
  const GemmDesc* d_rot1 = put(host, at, dev, tb.rot1);
  const GemmDesc* d_rot2 = put(host, at, dev, tb.rot2);
  const GemmDesc* d_back1 = put(host, at, dev, tb.back1);
  const GemmDesc* d_back2 = put(host, at, dev, tb.back2);
  if (at > set->table_bytes) return MFSDP_EWORKSPACE;
  if (cudaMemcpyAsync(dev, host.data(), at, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MFSDP_ECUDA;
  if (cudaFuncSetAttribute(jacobi_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kApplySmem) != cudaSuccess)
    return MFSDP_ECUDA;
  if (cudaFuncSetAttribute(jacobi_zrot_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)ztc::kSmem) != cudaSuccess)
    return MFSDP_ECUDA;
  const uint64_t limit_ns = wait_limit_ns();
  int* status = status_word_address();
  if (status == nullptr) return MFSDP_ECUDA;

  const unsigned ns = 2u * (unsigned)n;
  const int sweep_blocks = (int)((ns + 255) / 256);
  int e;
  // statistics
  if ((e = run_gemms(tb.stats_l, d_stats_l, 0, 1, st)) != MFSDP_OK) return e;
  if ((e = run_gemms(tb.stats_r, d_stats_r, 1, 0, st)) != MFSDP_OK) return e;
  if (h->refresh) {
    // the statistics in the previous basis, A = Q^T L Q, and Z = Q
    jacobi_setup_kernel<<<dim3(128, ns), 256, 0, st>>>(d_sides, ctl);
    if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
    if ((e = run_gemms(tb.t, d_t, 0, 0, st)) != MFSDP_OK) return e;
    if ((e = run_gemms(tb.a, d_a, 1, 0, st)) != MFSDP_OK) return e;
    diag_max_kernel<<<ns, 1024, 0, st>>>(d_sides, nullptr);
    // block Jacobi sweeps: the two groups of sides, each on two streams of its own (the
    // subproblems and A, and Z^T), as the graph's while loops, or issued sweep by sweep
    if (!set->aux) {
      bool ok = cudaStreamCreateWithFlags(&set->aux, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&set->ev_fork, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&set->ev_join, cudaEventDisableTiming) == cudaSuccess;
      for (int g = 0; g < 2 && ok; ++g) {
        ok = cudaStreamCreateWithFlags(&set->zst[g], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&set->ev_zjoin[g], cudaEventDisableTiming) == cudaSuccess &&
             cudaStreamCreateWithFlags(&set->rst[g], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&set->ev_rest[g], cudaEventDisableTiming) == cudaSuccess;
        for (int b = 0; b < 2 && ok; ++b)
          ok = cudaEventCreateWithFlags(&set->ev_j[g][b], cudaEventDisableTiming) ==
                   cudaSuccess &&
               cudaEventCreateWithFlags(&set->ev_z[g][b], cudaEventDisableTiming) == cudaSuccess;
      }
      if (!ok) return MFSDP_ECUDA;
    }
    const cudaStream_t gst[2] = {st, set->aux};
    const int goff[2] = {0, set->split}, gn[2] = {set->split, (int)ns - set->split};
    const int nb_max = std::max(set->nb_max_group[0], set->nb_max_group[1]);
    cudaError_t ce = cudaSuccess;
    auto ok = [&](cudaError_t x) { if (ce == cudaSuccess) ce = x; };
    // Round r of group g, its `rounds`-th overall: the subproblems, then A's block pairs, on
    // the group's stream `ms`; Z^T's rows on the group's Z^T stream `zs` once the round's
    // rotations are written.  The rotations alternate between two buffers, so a round waits
    // only for the Z^T rotations of the round two before it (the last reader of its buffer).
    auto round_launches = [&](int g, int r, long& rounds, cudaStream_t ms, cudaStream_t rs,
                              cudaStream_t zs) {
      const int b = (int)(rounds & 1);
      if (rounds >= 2) ok(cudaStreamWaitEvent(ms, set->ev_z[g][b], 0));
      jacobi_solve_kernel<<<(unsigned)tb.solve_begin[g].back(), kSolveThreads, 0, ms>>>(
          d_sides + goff[g], d_solve_begin[g], gn[g], ctl + goff[g], r, b);
      ok(cudaEventRecord(set->ev_j[g][b], ms));
      // A's critical block pairs once the previous round's others are done; the others beside
      // the next round's subproblems
      if (rounds >= 1) ok(cudaStreamWaitEvent(ms, set->ev_rest[g], 0));
      jacobi_apply_kernel<<<(unsigned)tb.crit_begin[g].back(), kJThreads, kApplySmem, ms>>>(
          d_sides + goff[g], d_crit_begin[g], gn[g], ctl + goff[g], r, b, 1);
      ok(cudaStreamWaitEvent(rs, set->ev_j[g][b], 0));
      jacobi_apply_kernel<<<(unsigned)tb.apply_begin[g].back(), kJThreads, kApplySmem, rs>>>(
          d_sides + goff[g], d_apply_begin[g], gn[g], ctl + goff[g], r, b, 2);
      ok(cudaEventRecord(set->ev_rest[g], rs));
      ok(cudaStreamWaitEvent(zs, set->ev_j[g][b], 0));
      jacobi_zrot_tc_kernel<<<(unsigned)tb.zrot_begin[g].back(), 128, ztc::kSmem, zs>>>(
          d_sides + goff[g], d_zrot_begin[g], gn[g], ctl + goff[g], r, b, limit_ns, status);
      ok(cudaEventRecord(set->ev_z[g][b], zs));
      ++rounds;
    };
    auto sweep_end = [&](int g, cudaStream_t ms) {
      jacobi_sweep_end_kernel<<<(gn[g] + 255) / 256, 256, 0, ms>>>(ctl + goff[g], gn[g]);
      diag_max_kernel<<<(unsigned)gn[g], 1024, 0, ms>>>(d_sides + goff[g], ctl + goff[g]);
    };
    // Build the graph: per group a while node; its body, captured from the group's two
    // streams, is one sweep followed by the loop condition.
    auto build_graph = [&]() -> bool {
      if (set->jgraph) cudaGraphExecDestroy(set->jgraph);
      set->jgraph = nullptr;
      cudaGraph_t top = nullptr;
      if (cudaGraphCreate(&top, 0) != cudaSuccess) return false;
      bool good = true;
      for (int g = 0; g < 2 && good; ++g) {
        if (gn[g] == 0) continue;
        cudaGraphConditionalHandle hnd;
        good = cudaGraphConditionalHandleCreate(&hnd, top, 1u, cudaGraphCondAssignDefault) ==
               cudaSuccess;
        cudaGraphNodeParams np{};
        np.type = cudaGraphNodeTypeConditional;
        np.conditional.handle = hnd;
        np.conditional.type = cudaGraphCondTypeWhile;
        np.conditional.size = 1;
        cudaGraphNode_t node;
        good = good && cudaGraphAddNode(&node, top, nullptr, nullptr, 0, &np) == cudaSuccess;
        if (!good) break;
        const cudaStream_t cs = set->aux, czs = set->zst[g], crs = set->rst[g];
        if (cudaStreamBeginCaptureToGraph(cs, np.conditional.phGraph_out[0], nullptr, nullptr, 0,
                                          cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
          good = false;
          break;
        }
        ce = cudaSuccess;
        ok(cudaEventRecord(set->ev_fork, cs));
        ok(cudaStreamWaitEvent(czs, set->ev_fork, 0));
        ok(cudaStreamWaitEvent(crs, set->ev_fork, 0));
        long rounds = 0;
        for (int r = 0; r < set->nb_max_group[g] - 1; ++r)
          round_launches(g, r, rounds, cs, crs, czs);
        ok(cudaEventRecord(set->ev_zjoin[g], czs));
        ok(cudaStreamWaitEvent(cs, set->ev_zjoin[g], 0));
        ok(cudaStreamWaitEvent(cs, set->ev_rest[g], 0));
        sweep_end(g, cs);
        jacobi_loop_kernel<<<1, 256, 0, cs>>>(ctl + goff[g], gn[g], h->max_sweeps, hnd);
        ok(cudaGetLastError());
        cudaGraph_t captured = nullptr;
        const cudaError_t ec = cudaStreamEndCapture(cs, &captured);
        good = ce == cudaSuccess && ec == cudaSuccess;
      }
      good = good && cudaGraphInstantiate(&set->jgraph, top, 0) == cudaSuccess;
      cudaGraphDestroy(top);
      ce = cudaSuccess;
      if (!good) {
        cudaGetLastError();
        if (set->jgraph) cudaGraphExecDestroy(set->jgraph);
        set->jgraph = nullptr;
        return false;
      }
      set->jgraph_ws = workspace;
      set->jgraph_sweeps = h->max_sweeps;
      return true;
    };
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return MFSDP_ECUDA;
    // MFSDP_SOAP_SWEEP_GRAPH=0 in the environment issues the sweeps one by one (profilers
    // that do not see kernels inside conditional graph nodes list them then)
    static const bool graph_env_off = [] {
      const char* v = std::getenv("MFSDP_SOAP_SWEEP_GRAPH");
      return v != nullptr && v[0] == '0';
    }();
    bool use_graph = !set->jgraph_off && !graph_env_off && cap == cudaStreamCaptureStatusNone;
    if (use_graph && (!set->jgraph || set->jgraph_ws != workspace ||
                      set->jgraph_sweeps != h->max_sweeps)) {
      use_graph = build_graph();
      if (!use_graph) set->jgraph_off = true;
    }
    if (use_graph) {
      if (cudaGraphLaunch(set->jgraph, st) != cudaSuccess) return MFSDP_ECUDA;
    } else {
      // the same launches issued sweep by sweep on the streams, forked from and joined back
      // into `st`; sweeps after a side has converged find it converged and return at once
      ok(cudaEventRecord(set->ev_fork, st));
      ok(cudaStreamWaitEvent(set->aux, set->ev_fork, 0));
      for (int g = 0; g < 2; ++g) {
        ok(cudaStreamWaitEvent(set->zst[g], set->ev_fork, 0));
        ok(cudaStreamWaitEvent(set->rst[g], set->ev_fork, 0));
      }
      long rounds[2] = {0, 0};
      for (int sw = 0; sw < h->max_sweeps; ++sw) {
        for (int r = 0; r < nb_max - 1; ++r)
          for (int g = 0; g < 2; ++g) {
            if (gn[g] == 0 || r >= set->nb_max_group[g] - 1) continue;
            round_launches(g, r, rounds[g], gst[g], set->rst[g], set->zst[g]);
          }
        for (int g = 0; g < 2; ++g)
          if (gn[g] > 0) sweep_end(g, gst[g]);
      }
      ok(cudaEventRecord(set->ev_join, set->aux));
      ok(cudaStreamWaitEvent(st, set->ev_join, 0));
      for (int g = 0; g < 2; ++g) {
        ok(cudaEventRecord(set->ev_zjoin[g], set->zst[g]));
        ok(cudaStreamWaitEvent(st, set->ev_zjoin[g], 0));
        ok(cudaEventRecord(set->ev_zjoin[g], set->rst[g]));
        ok(cudaStreamWaitEvent(st, set->ev_zjoin[g], 0));
      }
    }
    if (ce != cudaSuccess) return MFSDP_ECUDA;
    if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
    // the final polar step on Z^T (every side, converged at once or not)
    polar_prep_kernel<<<dim3(64, ns), 256, 0, st>>>(d_sides);
    if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
    if ((e = run_gemms(tb.polar1, d_polar1, 0, 1, st)) != MFSDP_OK) return e;
    if ((e = run_gemms(tb.polar2, d_polar2, 0, 0, st)) != MFSDP_OK) return e;
    polar_copy_kernel<<<dim3(64, ns), 256, 0, st>>>(d_sides);
    // eigenvalues (Rayleigh quotients) in descending order, the basis columns with them
    // (T = Z^T L with the symmetric L read as its own transpose: both operands K-major)
    if ((e = run_gemms(tb.ray, d_ray, 0, 1, st)) != MFSDP_OK) return e;
    rayleigh_kernel<<<dim3(64, ns), 256, 0, st>>>(d_sides);
    eig_rank_kernel<<<dim3((unsigned)((set->d_max + 255) / 256), ns), 256, 0, st>>>(d_sides);
    {
      const unsigned tiles = (unsigned)((set->d_max + 31) / 32);
      eig_scatter_kernel<<<dim3(tiles, tiles, ns), 256, 0, st>>>(d_sides);
    }
    if (info) jacobi_info_kernel<<<sweep_blocks, 256, 0, st>>>(d_sides, ctl, (int)ns, info);
  } else if (info && cudaMemsetAsync(info, 0, sizeof(int32_t) * ns, st) != cudaSuccess) {
    return MFSDP_ECUDA;
  }
  // Adam in the eigenbasis
  soap_moment_kernel<<<dim3(128, (unsigned)n), 256, 0, st>>>(d_mats, state->exp_avg, grad,
                                                             h->beta1);
  if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
  if ((e = run_gemms(tb.rot1, d_rot1, 1, 0, st)) != MFSDP_OK) return e;
  if ((e = run_gemms(tb.rot2, d_rot2, 0, 0, st)) != MFSDP_OK) return e;
  const float bc1 = (float)(1.0 - std::pow((double)h->beta1, (double)t));
  const float bc2 = (float)(1.0 - std::pow((double)h->beta2, (double)t));
  soap_adam_kernel<<<dim3(128, (unsigned)n), 256, 0, st>>>(d_mats, g_rot, m_rot,
                                                           state->exp_avg_sq, h->beta2, bc1,
                                                           bc2, h->eps);
  if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
  if ((e = run_gemms(tb.back1, d_back1, 0, 0, st)) != MFSDP_OK) return e;
  if ((e = run_gemms(tb.back2, d_back2, 0, 1, st)) != MFSDP_OK) return e;
  const float decay = (float)(1.0 - (double)h->lr * (double)h->weight_decay);
  soap_update_kernel<<<dim3(128, (unsigned)n), 256, 0, st>>>(d_mats, weights, g_rot, decay,
                                                             h->lr, status);
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}
