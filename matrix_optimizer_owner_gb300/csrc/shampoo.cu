// Owner Shampoo: full left / right preconditioners with an inverse fourth root, on the owner's
// whole matrices.
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding", §5.7:
// with every 2D matrix whole on its owner, the owner can run Shampoo, with full left and
// right preconditioners and their inverse fourth roots, in place of Muon.  Per owned matrix G (rows x
// cols), the original Shampoo update:
//     L += G G^T,  R += G^T G             (L_0 = R_0 = eps I)
//     P  = L^{-1/4} G R^{-1/4}
//     W  = W (1 - lr wd) - lr P
// The inverse fourth roots come from the coupled Newton iteration for the inverse p-th root
// (Guo and Higham, "A Schur–Newton method for the matrix p-th root and its inverse", 2006):
// with c = ||A||_F,  X_0 = c^{-1/4} I,  M_0 = A / c, and for k = 0 .. iters-1
//     T_k = (5 I - M_k) / 4,  X_{k+1} = X_k T_k,  M_{k+1} = T_k^4 M_k,
// so M_k -> I and X_k -> A^{-1/4}; an eigenvalue ratio of 1e-8 converges in 26 iterations.
//
// Two precisions.  fp32: the products run on the batched fp32 GEMM (tcgen05 kind::tf32 with
// three split products per multiply, "3xTF32", fp32 accumulation; a launch runs a product for
// every owned matrix, X' and T^2 together), the iteration's T = (5I - M) / 4 written by the
// epilogue of the product that forms M.  Split-bf16: the statistics as above, the root
// iteration and P on the tensor cores through the Newton-Schulz path's CTA-pair kernel in its
// split mode (values held as bf16 pairs hi + lo, three MMAs per product, fp32 accumulation,
// 256 x 256 tiles), symmetric side products as upper-triangle tiles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

// ||A||_F of each matrix (fp64, fixed order: per-thread strided sums, then a tree).
struct NormDesc {
  const float* a;
  int64_t numel;
  double* out;
};

__global__ void __launch_bounds__(1024) frob_kernel(const NormDesc* descs) {
  __shared__ double red[1024];
  const NormDesc d = descs[blockIdx.x];
  double s = 0.0;
  for (int64_t i = threadIdx.x; i < d.numel; i += blockDim.x) {
    const double v = d.a[i];
    s += v * v;
  }
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if ((int)threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *d.out = sqrt(red[0]);
}

// Start of the iteration for each matrix: X = c^{-1/4} I, M = A / c, T = (5I - M) / 4.
struct PrepDesc {
  const float* a;
  float* x;
  float* m;
  float* t;
  const double* norm;
  int32_t dim;
};

__global__ void root_prep_kernel(const PrepDesc* descs) {
  const PrepDesc d = descs[blockIdx.y];
  const int64_t n = (int64_t)d.dim * d.dim;
  const double c = *d.norm;
  const float inv_c = (float)(1.0 / c), x0 = (float)pow(c, -0.25);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const bool diag = (e / d.dim) == (e % d.dim);
    const float mv = d.a[e] * inv_c;
    d.m[e] = mv;
    d.t[e] = ((diag ? 5.f : 0.f) - mv) * 0.25f;
    d.x[e] = diag ? x0 : 0.f;
  }
}

// A = eps I for every state matrix.
__global__ void scaled_identity_kernel(float* base, const int64_t* offs, const int32_t* dims,
                                       float eps) {
  const int i = blockIdx.y;
  const int64_t n = (int64_t)dims[i] * dims[i];
  float* a = base + offs[i];
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x)
    a[e] = (e / dims[i]) == (e % dims[i]) ? eps : 0.f;
}

// One atomic per warp whose lanes saw a non-finite update (the device status word).
__device__ __forceinline__ void flag_non_finite(bool bad, int* status) {
  if (__any_sync(__activemask(), bad) && (threadIdx.x & 31) == 0)
    atomicOr(status, kStatusNonFinite);
}

// W = W (1 - lr wd) - lr P over the flat owner buffer.
__global__ void shampoo_update_kernel(float* w, const float* p, int64_t n, float decay,
                                      float lr, int* status) {
  bool bad = false;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    bad |= !isfinite(p[e]);
    w[e] = fmaf(w[e], decay, -lr * p[e]);
  }
  flag_non_finite(bad, status);
}

// ---------------------------------------------------------------- split-bf16 root path
// A value v is held as two bf16, hi = rn(v) and lo = rn(v - hi) (16 significant bits); the
// Newton–Schulz GEMM's split mode multiplies such pairs with three tensor-core products
// (hi*hi + hi*lo + lo*hi, fp32 accumulation) and writes its output the same way.
__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  hi = __bfloat16_as_ushort(h);
  lo = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
}
__device__ __forceinline__ float join_bf16(uint16_t hi, uint16_t lo) {
  return __uint_as_float((uint32_t)hi << 16) + __uint_as_float((uint32_t)lo << 16);
}

struct SplitDesc {   // a rows x cols fp32 matrix (pitch lds) to / from a split pair (pitch ldd)
  const float* src;
  uint16_t* hi;
  uint16_t* lo;
  int32_t rows, cols, lds, ldd;
};

// hi / lo of a fp32 matrix (the gradient G).
__global__ void to_split_kernel(const SplitDesc* descs) {
  const SplitDesc d = descs[blockIdx.y];
  const int64_t n = (int64_t)d.rows * d.cols;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / d.cols, c = e % d.cols;
    uint16_t h, l;
    split_bf16(d.src[r * d.lds + c], h, l);
    d.hi[r * d.ldd + c] = h;
    d.lo[r * d.ldd + c] = l;
  }
}

struct RootPrepDesc {
  const float* a;        // the statistics matrix, dim x dim, pitch dim
  const double* norm;    // ||A||_F
  uint16_t *x_hi, *x_lo, *m_hi, *m_lo, *t_hi, *t_lo;  // pitch ld
  int32_t dim, ld;
};

// X = c^{-1/4} I, M = A / c, T = (5I - M) / 4 as split pairs.
__global__ void root_prep_split_kernel(const RootPrepDesc* descs) {
  const RootPrepDesc d = descs[blockIdx.y];
  const int64_t n = (int64_t)d.dim * d.dim;
  const double c = *d.norm;
  const float inv_c = (float)(1.0 / c), x0 = (float)pow(c, -0.25);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / d.dim, col = e % d.dim, o = r * d.ld + col;
    const bool diag = r == col;
    uint16_t h, l;
    split_bf16(d.a[e] * inv_c, h, l);
    d.m_hi[o] = h;
    d.m_lo[o] = l;
    const float mv = join_bf16(h, l);
    split_bf16(((diag ? 5.f : 0.f) - mv) * 0.25f, h, l);
    d.t_hi[o] = h;
    d.t_lo[o] = l;
    split_bf16(diag ? x0 : 0.f, h, l);
    d.x_hi[o] = h;
    d.x_lo[o] = l;
  }
}

// W = W (1 - lr wd) - lr (P_hi + P_lo) for one matrix (P pitch ldp).
__global__ void update_split_kernel(float* w, const uint16_t* p_hi, const uint16_t* p_lo,
                                    int32_t rows, int32_t cols, int32_t ldp, float decay,
                                    float lr, int* status) {
  const int64_t n = (int64_t)rows * cols;
  bool bad = false;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e / cols, c = e % cols, o = r * ldp + c;
    const float pv = join_bf16(p_hi[o], p_lo[o]);
    bad |= !isfinite(pv);
    w[e] = fmaf(w[e], decay, -lr * pv);
  }
  flag_non_finite(bad, status);
}

}  // namespace

}  // namespace mfsdp

using namespace mfsdp;

// ------------------------------------------------------------------------------------------
// The owned-matrix set of the Shampoo step and its workspace layout.
// ------------------------------------------------------------------------------------------
struct mfsdp_shampoo_set {
  struct Mat {
    int64_t rows, cols, offset;  // in the flat owner buffers (weights, gradient, P)
    int64_t l_off, r_off;        // in the flat L and R state buffers
  };
  std::vector<Mat> mats;
  int64_t numel = 0, l_numel = 0, r_numel = 0;
  // workspace: per side (L of every matrix, then R of every matrix) X0, X1, M0, M1, T, T2, T4
  // (dim^2 floats each), then P and Y (numel floats each), norms, descriptor tables
  std::vector<int64_t> side_off;  // float offset of each side's seven buffers
  std::vector<int32_t> side_dim;
  int64_t floats = 0;
  size_t off_norms = 0, off_tables = 0, table_bytes = 0, ws_bytes = 0;
  // split-bf16 (tensor-core) layout: per side the same seven buffers as (hi, lo) bf16 pairs of
  // pitch side_ld; per matrix G, Y, P as pairs of pitch mat_ld; then norms, the epilogue's
  // (unused) per-problem scale array, tensor maps and launch tables
  std::vector<size_t> tc_side_off, tc_mat_off;
  std::vector<int32_t> side_ld, mat_ld;
  size_t tc_off_norms = 0, tc_off_fnorm = 0, tc_off_tables = 0, tc_table_bytes = 0;
  size_t tc_ws_bytes = 0;
  mutable int tc_pairs = 0, tc_pairs_dev = -1;  // co-resident pairs of the split pair kernel
};

namespace {

constexpr int kSideBufs = 7;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

namespace {

// Split-kernel launches of a step.  One root iteration is three launches over every side:
// kXT (X' = T X and T2 = T T, both from the current T), kT4 (T4 = T2 T2) and kTM (M' = T4 M,
// whose epilogue also writes the next T = (5I - M') / 4); the last iteration runs only the X'
// tiles of kXT.
// Every side product is a polynomial in the statistics matrix, so symmetric: only the tiles
// touching the upper triangle run and the epilogue mirrors them.
constexpr int kTcLaunches = 7;
enum TcLaunch { kXT0, kXT1, kT4, kTM0, kTM1, kY, kP };

int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

// Tensor-map index of buffer b of side k (hi half; +kMapsPerHalf: lo) or of matrix i's G, Y, P.
int tc_side_map(int k, int b) { return (k * kSideBufs + b) * 2 * kMapsPerHalf; }
int tc_mat_map(int n, int i, int b) { return (2 * n * kSideBufs + i * 3 + b) * 2 * kMapsPerHalf; }
int tc_n_maps(int n) { return (2 * n * kSideBufs + 3 * n) * 2 * kMapsPerHalf; }

struct TcTables {
  std::vector<NsProblem> probs[kTcLaunches];
  std::vector<NsTile> tiles[kTcLaunches];
  int32_t x_tiles[2] = {0, 0};  // leading X' tiles of kXT0 / kXT1
};

// Orders tiles [from, end) of a launch for the pair kernel's static schedule, in which pair p
// runs table entries p, p + P, p + 2P, ...  The sides' contraction lengths differ (768 … 3072
// on a transformer layer), so the plain order can leave one pair with well over the average
// work.  Wave by wave (P consecutive entries, one per pair), the longest remaining tiles go to
// the pairs with the least work so far; `load` carries each pair's work in k-blocks (plus a
// fixed cost for the epilogue) from the entries before `from`.
void balance_tiles(std::vector<NsTile>& tiles, size_t from, const std::vector<NsProblem>& probs,
                   int P, std::vector<int64_t>& load) {
  constexpr int64_t kTileFixed = 2;  // the epilogue's share of a tile, in k-block units
  auto cost = [&](const NsTile& t) { return (probs[(size_t)t.prob].K + 63) / 64 + kTileFixed; };
  std::stable_sort(tiles.begin() + (std::ptrdiff_t)from, tiles.end(),
                   [&](const NsTile& x, const NsTile& y) { return cost(x) > cost(y); });
  std::vector<size_t> pos;
  for (size_t i0 = from; i0 < tiles.size(); i0 += (size_t)P) {
    const size_t w = std::min((size_t)P, tiles.size() - i0);
    const std::vector<NsTile> wave(tiles.begin() + (std::ptrdiff_t)i0,
                                   tiles.begin() + (std::ptrdiff_t)(i0 + w));
    pos.resize(w);
    for (size_t j = 0; j < w; ++j) pos[j] = i0 + j;
    std::stable_sort(pos.begin(), pos.end(),
                     [&](size_t a, size_t b) { return load[a % P] < load[b % P]; });
    for (size_t j = 0; j < w; ++j) {
      tiles[pos[j]] = wave[j];
      load[pos[j] % P] += cost(wave[j]);
    }
  }
}

// Problems and tiles of every split-kernel launch; buffer addresses from the workspace `base`,
// or null when only the counts are wanted.  With `pairs` > 0 each launch's tiles are ordered
// for that many co-resident CTA pairs (any order gives the same result).
void tc_tables(const mfsdp_shampoo_set* s, uint8_t* base, int root_iters, int pairs,
               TcTables& tt) {
  const int n = (int)s->mats.size();
  auto sbuf = [&](int k, int b, int h) -> uint16_t* {
    if (!base) return nullptr;
    const int64_t d = s->side_dim[(size_t)k], p = s->side_ld[(size_t)k];
    return reinterpret_cast<uint16_t*>(base + s->tc_side_off[(size_t)k]) + (b * 2 + h) * d * p;
  };
  auto mbuf = [&](int i, int b, int h) -> uint16_t* {
    if (!base) return nullptr;
    const auto& m = s->mats[(size_t)i];
    return reinterpret_cast<uint16_t*>(base + s->tc_mat_off[(size_t)i]) +
           (b * 2 + h) * m.rows * s->mat_ld[(size_t)i];
  };
  enum { X0 = 0, X1 = 1, M0 = 2, M1 = 3, T = 4, T2 = 5, T4 = 6 };
  // out (M x N) = A B: A as K-major rows (M x K), B as MN-major rows (K x N) when b_mn = 1,
  // as K-major rows (N x K, i.e. B^T stored) when b_mn = 0
  auto prob = [&](int M, int N, int K, int b_mn, int sym, int mat, int ma, int mb, uint16_t* oh,
                  uint16_t* ol, int64_t ldo) {
    NsProblem p{};
    p.M = M; p.N = N; p.K = K;
    p.a_mn = 0; p.b_mn = b_mn; p.sym = sym; p.kind = kApply; p.first = 0; p.mat = mat;
    p.map_a = ma; p.map_b = mb; p.mn3d = 0; p.map_o = 0;
    p.d_hi = nullptr; p.d_lo = nullptr; p.ldd = 0;  // no addend: the launches run with a = 0
    p.o_hi = oh; p.o_lo = ol; p.ldo = ldo;
    return p;
  };
  auto side = [&](int k, int a, int b, int o) {  // side product o = a b of side k
    const int d = s->side_dim[(size_t)k], p = s->side_ld[(size_t)k];
    return prob(d, d, d, 1, 1, k, tc_side_map(k, a), tc_side_map(k, b), sbuf(k, o, 0),
                sbuf(k, o, 1), p);
  };
  for (int par = 0; par < 2; ++par) {
    const int xi = par ? X1 : X0, xo = par ? X0 : X1, mi = par ? M1 : M0, mo = par ? M0 : M1;
    auto& xt = tt.probs[par ? kXT1 : kXT0];
    for (int k = 0; k < 2 * n; ++k) xt.push_back(side(k, T, xi, xo));
    for (int k = 0; k < 2 * n; ++k) xt.push_back(side(k, T, T, T2));
    for (int k = 0; k < 2 * n; ++k) {  // M' = T4 M, and from its epilogue T = (5I - M') / 4
      NsProblem p = side(k, T4, mi, mo);
      p.t_hi = sbuf(k, T, 0);
      p.t_lo = sbuf(k, T, 1);
      tt.probs[par ? kTM1 : kTM0].push_back(p);
    }
  }
  for (int k = 0; k < 2 * n; ++k) tt.probs[kT4].push_back(side(k, T2, T2, T4));
  // P = X_L G X_R with the roots in X[root_iters & 1]: Y = X_L G, P = Y X_R
  const int xf = root_iters & 1;
  for (int i = 0; i < n; ++i) {
    const auto& m = s->mats[(size_t)i];
    const int rows = (int)m.rows, cols = (int)m.cols, pc = s->mat_ld[(size_t)i];
    tt.probs[kY].push_back(prob(rows, cols, rows, 1, 0, i, tc_side_map(i, xf),
                                tc_mat_map(n, i, 0), mbuf(i, 1, 0), mbuf(i, 1, 1), pc));
    tt.probs[kP].push_back(prob(rows, cols, cols, 1, 0, i, tc_mat_map(n, i, 1),
                                tc_side_map(n + i, xf), mbuf(i, 2, 0), mbuf(i, 2, 1), pc));
  }
  for (int l = 0; l < kTcLaunches; ++l)
    for (size_t q = 0; q < tt.probs[l].size(); ++q) {
      const NsProblem& p = tt.probs[l][q];
      add_tiles(tt.tiles[l], (int32_t)q, p.M, p.N, p.sym != 0, kPairBM);
      if ((l == kXT0 || l == kXT1) && q + 1 == (size_t)(2 * n))
        tt.x_tiles[l == kXT1] = (int32_t)tt.tiles[l].size();
    }
  if (pairs <= 0) return;
  for (int l = 0; l < kTcLaunches; ++l) {
    std::vector<int64_t> load((size_t)pairs, 0);
    auto& t = tt.tiles[l];
    if (l == kXT0 || l == kXT1) {
      // the X' tiles stay a prefix (the last iteration runs them alone), balanced on their
      // own; the T^2 tiles continue from the loads they leave
      const size_t x = (size_t)tt.x_tiles[l == kXT1];
      std::vector<NsTile> rest(t.begin() + (std::ptrdiff_t)x, t.end());
      t.resize(x);
      balance_tiles(t, 0, tt.probs[l], pairs, load);
      t.insert(t.end(), rest.begin(), rest.end());
      balance_tiles(t, x, tt.probs[l], pairs, load);
    } else {
      balance_tiles(t, 0, tt.probs[l], pairs, load);
    }
  }
}

size_t tc_table_bytes(const TcTables& tt, int n) {
  size_t b = align256(sizeof(CUtensorMap) * (size_t)tc_n_maps(n));
  for (int l = 0; l < kTcLaunches; ++l)
    b += align256(sizeof(NsProblem) * std::max<size_t>(tt.probs[l].size(), 1)) +
         align256(sizeof(NsTile) * std::max<size_t>(tt.tiles[l].size(), 1));
  b += align256(sizeof(GemmDesc) * 2 * (size_t)n) + align256(sizeof(NormDesc) * 2 * (size_t)n) +
       align256(sizeof(RootPrepDesc) * 2 * (size_t)n) + align256(sizeof(SplitDesc) * (size_t)n);
  return b;
}

void tc_layout(mfsdp_shampoo_set* s) {
  const int n = (int)s->mats.size();
  size_t off = 0;
  for (int sd = 0; sd < 2; ++sd)
    for (const auto& m : s->mats) {
      const int64_t d = sd == 0 ? m.rows : m.cols;
      s->side_ld.push_back((int32_t)round8(d));
      s->tc_side_off.push_back(off);
      off = align256(off + sizeof(uint16_t) * 2 * kSideBufs * (size_t)d * (size_t)round8(d));
    }
  for (const auto& m : s->mats) {
    s->mat_ld.push_back((int32_t)round8(m.cols));
    s->tc_mat_off.push_back(off);
    off = align256(off + sizeof(uint16_t) * 6 * (size_t)m.rows * (size_t)round8(m.cols));
  }
  s->tc_off_norms = off;
  s->tc_off_fnorm = align256(off + sizeof(double) * 2 * (size_t)std::max(n, 1));
  s->tc_off_tables = align256(s->tc_off_fnorm + sizeof(float) * 2 * (size_t)std::max(n, 1));
  s->tc_off_tables = (s->tc_off_tables + 1023) & ~size_t(1023);  // tensor maps: 64-byte aligned
  TcTables tt;
  tc_tables(s, nullptr, 1, 0, tt);
  s->tc_table_bytes = tc_table_bytes(tt, std::max(n, 1));
  s->tc_ws_bytes = align256(s->tc_off_tables + s->tc_table_bytes);
}

}  // namespace

extern "C" int mfsdp_shampoo_set_create(const mfsdp_matrix* mats, int32_t n_mats,
                                        mfsdp_shampoo_set** out) {
  if (out == nullptr || n_mats < 0 || (n_mats > 0 && mats == nullptr)) return MFSDP_EINVAL;
  auto* s = new mfsdp_shampoo_set();
  int64_t lo = 0, ro = 0;
  for (int32_t i = 0; i < n_mats; ++i) {
    const mfsdp_matrix& m = mats[i];
    if (m.rows <= 0 || m.cols <= 0 || m.offset < 0 || m.rows > (1 << 16) || m.cols > (1 << 16)) {
      delete s;
      return MFSDP_ESHAPE;
    }
    s->mats.push_back({m.rows, m.cols, m.offset, lo, ro});
    lo += m.rows * m.rows;
    ro += m.cols * m.cols;
    s->numel = std::max(s->numel, m.offset + m.rows * m.cols);
  }
  s->l_numel = lo;
  s->r_numel = ro;
  int64_t f = 0;
  for (int side = 0; side < 2; ++side)
    for (const auto& m : s->mats) {
      const int64_t d = side == 0 ? m.rows : m.cols;
      s->side_off.push_back(f);
      s->side_dim.push_back((int32_t)d);
      f += kSideBufs * d * d;
    }
  f += 2 * s->numel;  // P and Y
  s->floats = f;
  const int n = n_mats;
  s->off_norms = align256((size_t)f * sizeof(float));
  s->off_tables = align256(s->off_norms + sizeof(double) * 2 * (size_t)std::max(n, 1));
  // tables: stats (2n), the iteration's 4 products x 2n for each parity, P (2n), norms (2n),
  // prep (2n); the state-initialisation offsets and dims fit in the same space
  s->table_bytes = sizeof(GemmDesc) * (size_t)(20 * std::max(n, 1)) +
                   sizeof(NormDesc) * 2 * (size_t)std::max(n, 1) +
                   sizeof(PrepDesc) * 2 * (size_t)std::max(n, 1);
  s->ws_bytes = align256(s->off_tables + s->table_bytes);
  tc_layout(s);
  s->ws_bytes = std::max(s->ws_bytes, s->tc_ws_bytes);
  *out = s;
  return MFSDP_OK;
}

extern "C" int mfsdp_shampoo_set_destroy(mfsdp_shampoo_set* set) {
  delete set;
  return MFSDP_OK;
}

extern "C" int mfsdp_shampoo_set_sizes(const mfsdp_shampoo_set* set, size_t* workspace_bytes,
                                       int64_t* l_numel, int64_t* r_numel) {
  if (set == nullptr) return MFSDP_EINVAL;
  if (workspace_bytes) *workspace_bytes = set->ws_bytes;
  if (l_numel) *l_numel = set->l_numel;
  if (r_numel) *r_numel = set->r_numel;
  return MFSDP_OK;
}

extern "C" int mfsdp_shampoo_init_state(const mfsdp_shampoo_set* set, float eps, float* l,
                                        float* r, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (set == nullptr || !(eps > 0.f) || l == nullptr || r == nullptr) return MFSDP_EINVAL;
  const int n = (int)set->mats.size();
  if (n == 0) return MFSDP_OK;
  if (workspace == nullptr || workspace_bytes < set->ws_bytes) return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // offsets and dims of L then R, staged in the workspace's table area
  std::vector<int64_t> offs(2 * (size_t)n);
  std::vector<int32_t> dims(2 * (size_t)n);
  for (int i = 0; i < n; ++i) {
    offs[i] = set->mats[i].l_off;
    dims[i] = (int32_t)set->mats[i].rows;
    offs[n + i] = set->mats[i].r_off;
    dims[n + i] = (int32_t)set->mats[i].cols;
  }
  uint8_t* tab = static_cast<uint8_t*>(workspace) + set->off_tables;
  const size_t ob = offs.size() * sizeof(int64_t);
  if (ob + dims.size() * sizeof(int32_t) > set->table_bytes) return MFSDP_EWORKSPACE;
  if (cudaMemcpyAsync(tab, offs.data(), ob, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(tab + ob, dims.data(), dims.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MFSDP_ECUDA;
  const auto* doffs = reinterpret_cast<const int64_t*>(tab);
  const auto* ddims = reinterpret_cast<const int32_t*>(tab + ob);
  scaled_identity_kernel<<<dim3(64, (unsigned)n), 256, 0, st>>>(l, doffs, ddims, eps);
  scaled_identity_kernel<<<dim3(64, (unsigned)n), 256, 0, st>>>(r, doffs + n, ddims + n, eps);
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}

namespace {

// The Shampoo step with the root iterations and the preconditioning on the tensor cores
// (split-bf16 operands, fp32 accumulation); statistics and norms as in the fp32 path.
int shampoo_step_split(const mfsdp_shampoo_set* set, const float* grad, float* l, float* r,
                       float* weights, float lr, float weight_decay, int32_t root_iters,
                       uint8_t* ws, cudaStream_t st) {
  const int n = (int)set->mats.size();
  if (ns_prepare_kernels() != cudaSuccess) return MFSDP_ECUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MFSDP_ECUDA;
  if (set->tc_pairs <= 0 || set->tc_pairs_dev != dev) {
    set->tc_pairs = ns_pair_max_clusters(sms, true);
    set->tc_pairs_dev = dev;
    if (set->tc_pairs <= 0) return MFSDP_ECUDA;
  }
  const int pairs = set->tc_pairs;
  TcTables tt;
  tc_tables(set, ws, root_iters, pairs, tt);
  double* norms = reinterpret_cast<double*>(ws + set->tc_off_norms);
  float* fnorm = reinterpret_cast<float*>(ws + set->tc_off_fnorm);
  auto sbuf = [&](int k, int b, int h) {
    const int64_t d = set->side_dim[(size_t)k], p = set->side_ld[(size_t)k];
    return reinterpret_cast<uint16_t*>(ws + set->tc_side_off[(size_t)k]) + (b * 2 + h) * d * p;
  };
  auto mbuf = [&](int i, int b, int h) {
    return reinterpret_cast<uint16_t*>(ws + set->tc_mat_off[(size_t)i]) +
           (b * 2 + h) * set->mats[(size_t)i].rows * set->mat_ld[(size_t)i];
  };
  enum { X0 = 0, X1 = 1, M0 = 2, M1 = 3, T = 4 };

  // tensor maps: the 64 x 64 box (MN-major operand) and the 128 x 64 box (K-major operand) of
  // every hi and lo half
  std::vector<CUtensorMap> maps((size_t)tc_n_maps(n));
  std::memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
  auto put_maps = [&](int idx, const uint16_t* hi, const uint16_t* lo, int64_t rows, int64_t cols,
                      int64_t ld) {
    for (int h = 0; h < 2; ++h) {
      CUtensorMap* mp = maps.data() + idx + h * kMapsPerHalf;
      const uint16_t* b = h ? lo : hi;
      if (!encode_map(mp, b, rows, cols, ld, 64u) || !encode_map(mp + 1, b, rows, cols, ld, 128u))
        return false;
    }
    return true;
  };
  for (int k = 0; k < 2 * n; ++k)
    for (int b = 0; b < kSideBufs; ++b)
      if (!put_maps(tc_side_map(k, b), sbuf(k, b, 0), sbuf(k, b, 1), set->side_dim[(size_t)k],
                    set->side_dim[(size_t)k], set->side_ld[(size_t)k]))
        return MFSDP_ECUDA;
  for (int i = 0; i < n; ++i)
    for (int b = 0; b < 2; ++b)  // G and Y are operands; P only an output
      if (!put_maps(tc_mat_map(n, i, b), mbuf(i, b, 0), mbuf(i, b, 1), set->mats[(size_t)i].rows,
                    set->mats[(size_t)i].cols, set->mat_ld[(size_t)i]))
        return MFSDP_ECUDA;

  std::vector<GemmDesc> stats(2 * (size_t)n);
  std::vector<NormDesc> nd(2 * (size_t)n);
  std::vector<RootPrepDesc> pd(2 * (size_t)n);
  std::vector<SplitDesc> sp((size_t)n);
  for (int i = 0; i < n; ++i) {
    const auto& m = set->mats[(size_t)i];
    const float* g = grad + m.offset;
    const int rows = (int)m.rows, cols = (int)m.cols;
    stats[i] = {g, g, l + m.l_off, nullptr, rows, rows, cols, cols, cols, rows, 1.f, 1.f};
    stats[n + i] = {g, g, r + m.r_off, nullptr, cols, cols, rows, cols, cols, cols, 1.f, 1.f};
    sp[i] = {g, mbuf(i, 0, 0), mbuf(i, 0, 1), rows, cols, cols, set->mat_ld[(size_t)i]};
  }
  for (int k = 0; k < 2 * n; ++k) {
    const int i = k % n, d = set->side_dim[(size_t)k], ld = set->side_ld[(size_t)k];
    const auto& m = set->mats[(size_t)i];
    float* a = k < n ? l + m.l_off : r + m.r_off;
    nd[k] = {a, (int64_t)d * d, norms + k};
    pd[k] = {a, norms + k, sbuf(k, X0, 0), sbuf(k, X0, 1), sbuf(k, M0, 0), sbuf(k, M0, 1),
             sbuf(k, T, 0), sbuf(k, T, 1), d, ld};
  }

  // one upload, in the layout the table area is sized for
  std::vector<uint8_t> host(set->tc_table_bytes, 0);
  size_t at = 0;
  auto put = [&](const void* src, size_t bytes) {
    const size_t o = at;
    std::memcpy(host.data() + at, src, bytes);
    at += align256(std::max<size_t>(bytes, 1));
    return o;
  };
  const size_t o_maps = put(maps.data(), maps.size() * sizeof(CUtensorMap));
  size_t o_probs[kTcLaunches], o_tiles[kTcLaunches];
  for (int q = 0; q < kTcLaunches; ++q) {
    o_probs[q] = put(tt.probs[q].data(), tt.probs[q].size() * sizeof(NsProblem));
    o_tiles[q] = put(tt.tiles[q].data(), tt.tiles[q].size() * sizeof(NsTile));
  }
  const size_t o_stats = put(stats.data(), stats.size() * sizeof(GemmDesc));
  const size_t o_norm = put(nd.data(), nd.size() * sizeof(NormDesc));
  const size_t o_prep = put(pd.data(), pd.size() * sizeof(RootPrepDesc));
  const size_t o_split = put(sp.data(), sp.size() * sizeof(SplitDesc));
  if (at > set->tc_table_bytes) return MFSDP_EWORKSPACE;
  uint8_t* tab = ws + set->tc_off_tables;
  if (cudaMemcpyAsync(tab, host.data(), at, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemsetAsync(fnorm, 0, sizeof(float) * 2 * (size_t)n, st) != cudaSuccess)
    return MFSDP_ECUDA;
  int* status = status_word_address();
  if (status == nullptr) return MFSDP_ECUDA;

  auto ns = [&](int q, int32_t ntiles) {
    NsLaunchParams lp{};
    lp.probs = reinterpret_cast<const NsProblem*>(tab + o_probs[q]);
    lp.tiles = reinterpret_cast<const NsTile*>(tab + o_tiles[q]);
    lp.ntiles = ntiles;
    lp.maps = reinterpret_cast<const CUtensorMap*>(tab + o_maps);
    lp.norm = fnorm;
    lp.eps = 1.f;
    lp.a = 0.f;  // out = acc: no addend
    lp.b = 0.f;
    lp.c = 1.f;
    lp.wait_limit_ns = wait_limit_ns();
    lp.status = status;
    return launch_ns_pair_split(lp, pairs, st) == cudaSuccess;
  };
  auto all = [&](int q) { return (int32_t)tt.tiles[q].size(); };
  const unsigned nb = (unsigned)n;
  int e;
  // statistics: L += G G^T, R += G^T G (fp32), and G as a split pair
  const GemmDesc* d_stats = reinterpret_cast<const GemmDesc*>(tab + o_stats);
  if ((e = launch_gemm(d_stats, stats.data(), n, 0, 1, st)) != MFSDP_OK) return e;
  if ((e = launch_gemm(d_stats + n, stats.data() + n, n, 1, 0, st)) != MFSDP_OK) return e;
  to_split_kernel<<<dim3(128, nb), 256, 0, st>>>(reinterpret_cast<const SplitDesc*>(tab + o_split));
  frob_kernel<<<2 * n, 1024, 0, st>>>(reinterpret_cast<const NormDesc*>(tab + o_norm));
  root_prep_split_kernel<<<dim3(256, 2 * nb), 256, 0, st>>>(
      reinterpret_cast<const RootPrepDesc*>(tab + o_prep));
  if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
  for (int it = 0; it < root_iters; ++it) {
    const int par = it & 1;
    const bool last = it + 1 == root_iters;
    if (!ns(par ? kXT1 : kXT0, last ? tt.x_tiles[par] : all(par ? kXT1 : kXT0))) return MFSDP_ECUDA;
    if (last) break;
    if (!ns(kT4, all(kT4)) || !ns(par ? kTM1 : kTM0, all(par ? kTM1 : kTM0))) return MFSDP_ECUDA;
  }
  // P = X_L G X_R
  if (!ns(kY, all(kY)) || !ns(kP, all(kP))) return MFSDP_ECUDA;
  const float decay = (float)(1.0 - (double)lr * (double)weight_decay);
  for (int i = 0; i < n; ++i) {
    const auto& m = set->mats[(size_t)i];
    const int blocks = (int)std::min<int64_t>((m.rows * m.cols + 255) / 256, 4096);
    update_split_kernel<<<blocks, 256, 0, st>>>(weights + m.offset, mbuf(i, 2, 0), mbuf(i, 2, 1),
                                                (int32_t)m.rows, (int32_t)m.cols,
                                                set->mat_ld[(size_t)i], decay, lr, status);
  }
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}

}  // namespace

extern "C" int mfsdp_shampoo_step(const mfsdp_shampoo_set* set, const float* grad, float* l,
                                  float* r, float* weights, float lr, float weight_decay,
                                  int32_t root_iters, int32_t precision, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (set == nullptr || grad == nullptr || l == nullptr || r == nullptr || weights == nullptr)
    return MFSDP_EINVAL;
  if (root_iters < 1 || root_iters > 200) return MFSDP_EINVAL;
  if (precision != MFSDP_SHAMPOO_FP32 && precision != MFSDP_SHAMPOO_SPLIT_BF16)
    return MFSDP_EINVAL;
  const int n = (int)set->mats.size();
  if (n == 0) return MFSDP_OK;
  if (workspace == nullptr || workspace_bytes < set->ws_bytes) return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (precision == MFSDP_SHAMPOO_SPLIT_BF16)
    return shampoo_step_split(set, grad, l, r, weights, lr, weight_decay, root_iters,
                              static_cast<uint8_t*>(workspace), st);
  float* wsf = static_cast<float*>(workspace);
  double* norms = reinterpret_cast<double*>(static_cast<uint8_t*>(workspace) + set->off_norms);
  float* pbuf = wsf + (set->floats - 2 * set->numel);
  float* ybuf = pbuf + set->numel;
  auto side = [&](int sd, int i, int b) {  // buffer b of side sd (0 = L, 1 = R) of matrix i
    return wsf + set->side_off[(size_t)(sd * n + i)] +
           (int64_t)b * set->side_dim[(size_t)(sd * n + i)] * set->side_dim[(size_t)(sd * n + i)];
  };
  enum { X0 = 0, X1 = 1, M0 = 2, M1 = 3, T = 4, T2 = 5, T4 = 6 };

  // Host tables, uploaded once per step.
  std::vector<GemmDesc> stats(2 * (size_t)n), iter(4 * 2 * (size_t)n), pre(2 * (size_t)n);
  std::vector<NormDesc> nd(2 * (size_t)n);
  std::vector<PrepDesc> pd(2 * (size_t)n);
  for (int i = 0; i < n; ++i) {
    const auto& m = set->mats[i];
    const float* g = grad + m.offset;
    const int rows = (int)m.rows, cols = (int)m.cols;
    // L += G G^T (A = G, op(B) = G^T)   R += G^T G (op(A) = G^T, B = G)
    stats[i] = {g, g, l + m.l_off, nullptr, rows, rows, cols, cols, cols, rows, 1.f, 1.f};
    stats[n + i] = {g, g, r + m.r_off, nullptr, cols, cols, rows, cols, cols, cols, 1.f, 1.f};
    for (int sd = 0; sd < 2; ++sd) {
      const int k = sd * n + i, d = sd == 0 ? rows : cols;
      nd[k] = {sd == 0 ? l + m.l_off : r + m.r_off, (int64_t)d * d, norms + k};
      pd[k] = {sd == 0 ? l + m.l_off : r + m.r_off, side(sd, i, X0), side(sd, i, M0),
               side(sd, i, T), norms + k, d};
    }
    // P = X_L G X_R: Y = X_L G, P = Y X_R (root buffers chosen below by iteration parity)
  }
  // the iteration ping-pongs X and M: after `root_iters` iterations the result is in
  // X[root_iters & 1]
  const int xf = root_iters & 1;
  for (int i = 0; i < n; ++i) {
    const auto& m = set->mats[i];
    const int rows = (int)m.rows, cols = (int)m.cols;
    pre[i] = {side(0, i, xf), grad + m.offset, ybuf + m.offset, nullptr, rows, cols, rows, rows,
              cols, cols, 1.f, 0.f};
    pre[n + i] = {ybuf + m.offset, side(1, i, xf), pbuf + m.offset, nullptr, rows, cols, cols,
                  cols, cols, cols, 1.f, 0.f};
  }
  // Iteration products for both parities of k: even k reads X0 / M0 and writes X1 / M1, odd
  // k the reverse.
  std::vector<GemmDesc> iter_odd(4 * 2 * (size_t)n);
  for (int par = 0; par < 2; ++par) {
    std::vector<GemmDesc>& tbl = par == 0 ? iter : iter_odd;
    const int xi = par == 0 ? X0 : X1, xo = par == 0 ? X1 : X0;
    const int mi = par == 0 ? M0 : M1, mo = par == 0 ? M1 : M0;
    for (int sd = 0; sd < 2; ++sd)
      for (int i = 0; i < n; ++i) {
        const int k = sd * n + i;
        const int d = set->side_dim[(size_t)k];
        // X_{k+1} = X_k T,  T2 = T T,  T4 = T2 T2,  M_{k+1} = T4 M_k (and T = (5I - M)/4)
        tbl[0 * 2 * n + k] = {side(sd, i, xi), side(sd, i, T), side(sd, i, xo), nullptr,
                              d, d, d, d, d, d, 1.f, 0.f};
        tbl[1 * 2 * n + k] = {side(sd, i, T), side(sd, i, T), side(sd, i, T2), nullptr,
                              d, d, d, d, d, d, 1.f, 0.f};
        tbl[2 * 2 * n + k] = {side(sd, i, T2), side(sd, i, T2), side(sd, i, T4), nullptr,
                              d, d, d, d, d, d, 1.f, 0.f};
        tbl[3 * 2 * n + k] = {side(sd, i, T4), side(sd, i, mi), side(sd, i, mo),
                              side(sd, i, T), d, d, d, d, d, d, 1.f, 0.f};
      }
  }
  // One upload of every table: stats | even iteration | odd iteration | P | norms | prep.
  const size_t g_bytes = sizeof(GemmDesc) * (size_t)(20 * n);
  std::vector<uint8_t> host(g_bytes + sizeof(NormDesc) * 2 * (size_t)n +
                            sizeof(PrepDesc) * 2 * (size_t)n);
  if (host.size() > set->table_bytes) return MFSDP_EWORKSPACE;
  {
    uint8_t* h = host.data();
    auto put = [&](const void* src, size_t bytes) {
      std::memcpy(h, src, bytes);
      h += bytes;
    };
    put(stats.data(), sizeof(GemmDesc) * stats.size());
    put(iter.data(), sizeof(GemmDesc) * iter.size());
    put(iter_odd.data(), sizeof(GemmDesc) * iter_odd.size());
    put(pre.data(), sizeof(GemmDesc) * pre.size());
    put(nd.data(), sizeof(NormDesc) * nd.size());
    put(pd.data(), sizeof(PrepDesc) * pd.size());
  }
  uint8_t* tab = static_cast<uint8_t*>(workspace) + set->off_tables;
  if (cudaMemcpyAsync(tab, host.data(), host.size(), cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MFSDP_ECUDA;
  const GemmDesc* d_stats = reinterpret_cast<const GemmDesc*>(tab);
  const GemmDesc* d_even = d_stats + 2 * n;
  const GemmDesc* d_odd = d_even + 8 * n;
  const GemmDesc* d_pre = d_odd + 8 * n;
  const NormDesc* d_norm = reinterpret_cast<const NormDesc*>(d_pre + 2 * n);
  const PrepDesc* d_prep = reinterpret_cast<const PrepDesc*>(d_norm + 2 * n);

  int e;
  // statistics: L += G G^T, R += G^T G
  if ((e = launch_gemm(d_stats, stats.data(), n, 0, 1, st)) != MFSDP_OK) return e;
  if ((e = launch_gemm(d_stats + n, stats.data() + n, n, 1, 0, st)) != MFSDP_OK) return e;
  // inverse fourth roots of every L and R
  frob_kernel<<<2 * n, 1024, 0, st>>>(d_norm);
  root_prep_kernel<<<dim3(256, (unsigned)(2 * n)), 256, 0, st>>>(d_prep);
  if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
  // Three launches per iteration: X' = X T with T2 = T T (both read only the current T, so
  // they share one launch of 4n problems), then T4 = T2 T2, then M' = T4 M (whose epilogue
  // writes the next T).  Every right factor (T, T2, M) is a polynomial in the statistics
  // matrix, so symmetric: it is read as its own transpose (trans_b = 1), which puts both
  // operands K-major and lets the GEMM load them by TMA.
  for (int it = 0; it < root_iters; ++it) {
    const GemmDesc* tbl = (it & 1) ? d_odd : d_even;
    const GemmDesc* htbl = (it & 1) ? iter_odd.data() : iter.data();
    if ((e = launch_gemm(tbl, htbl, 4 * n, 0, 1, st)) != MFSDP_OK) return e;
    for (int prod = 2; prod < 4; ++prod)
      if ((e = launch_gemm(tbl + prod * 2 * n, htbl + prod * 2 * n, 2 * n, 0, 1, st)) !=
          MFSDP_OK)
        return e;
  }
  // P = L^{-1/4} G R^{-1/4} (R^{-1/4} symmetric: read as its own transpose)
  if ((e = launch_gemm(d_pre, pre.data(), n, 0, 0, st)) != MFSDP_OK) return e;
  if ((e = launch_gemm(d_pre + n, pre.data() + n, n, 0, 1, st)) != MFSDP_OK) return e;
  // W = W (1 - lr wd) - lr P, matrix by matrix
  int* status = status_word_address();
  if (status == nullptr) return MFSDP_ECUDA;
  const float decay = (float)(1.0 - (double)lr * (double)weight_decay);
  for (const auto& m : set->mats) {
    const int64_t cnt = m.rows * m.cols;
    const int blocks = (int)std::min<int64_t>((cnt + 255) / 256, 4096);
    shampoo_update_kernel<<<blocks, 256, 0, st>>>(weights + m.offset, pbuf + m.offset, cnt,
                                                  decay, lr, status);
  }
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}
