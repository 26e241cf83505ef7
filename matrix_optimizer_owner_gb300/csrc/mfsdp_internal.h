// Internal declarations shared by the host API and the kernels of libmfsdp.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

namespace mfsdp {

// ---- device status word bits (kept in one __device__ int per device) ----------------------
constexpr int kStatusTimeout = 1;
constexpr int kStatusNonFinite = 2;
constexpr int kStatusTmemMismatch = 4;  // a CTA pair received different tensor-memory bases

// ---- streaming kernels (gradient deposit + momentum + norm, update) -----------------------
constexpr int kMaxContrib = 64;
constexpr int kStreamThreads = 256;
constexpr int kVec = 8;                                   // elements per thread per access
constexpr int kVecsPerThread = 8;                         // vectors per thread per CTA
constexpr int kChunk = kStreamThreads * kVec * kVecsPerThread;  // 16384 elements per CTA

struct DevMat {            // one owned matrix, as the streaming kernels see it
  int64_t offset;          // element offset in the flat owner buffers
  int64_t numel;
  int64_t rows, cols;
  int32_t cta_begin;       // first CTA of this matrix in the per-matrix CTA partition
  int32_t split;           // 1: NS input / output carry a low bf16 half
  float scale_original;    // sqrt(max(1, rows/cols))
  float scale_rms;         // 0.2 * sqrt(max(rows, cols))
};

struct ContribPtrs {
  const void* p[kMaxContrib];
};

constexpr int kMaxBulkStages = 8;
constexpr size_t kBulkStageBudget = 48 * 1024;   // bytes of one bulk-copy stage
constexpr size_t kBulkSmemBudget = 192 * 1024;   // bytes of all stages of one CTA

struct BulkCfg {           // bulk-copy pipeline shape of the deposit kernel
  int32_t sub_elems;       // elements per stage
  int32_t stage_bytes;
  int32_t stages;
  int32_t pad_;
  uint64_t wait_limit_ns;
};

struct ReduceParams {
  ContribPtrs contrib;
  int32_t W;
  int32_t n_mats;
  int32_t total_ctas;
  int32_t nesterov;
  int32_t offsets_aligned;  // every matrix offset is a multiple of 8 elements
  int32_t pad_;
  uint64_t wait_limit_ns;
  int* status;
  const DevMat* mats;
  float grad_scale, mu, one_minus_mu;
  float* momentum;
  uint16_t* uhat;
  uint16_t* uhat_lo;       // nullable
  float* grad;             // nullable
  float* partials;         // [total_ctas]
};

struct NormParams {
  const DevMat* mats;
  int32_t n_mats;
  const float* partials;
  float* norm;             // [n_mats]
  int* status;
};

struct UpdateParams {
  const DevMat* mats;
  int32_t n_mats;
  int32_t total_ctas;
  int32_t lr_adjust;
  float decay;             // 1 - lr * weight_decay
  float lr;
  float* weights;
  const uint16_t* ortho;
  const uint16_t* ortho_lo;  // nullable
};

struct AdamParams {
  ContribPtrs contrib;
  int32_t W;
  int64_t n;
  float grad_scale;
  float decay;             // 1 - lr * weight_decay
  float b1, one_minus_b1, b2, one_minus_b2;
  float step_size;         // lr / (1 - b1^t)
  float inv_sqrt_bc2;      // 1 / sqrt(1 - b2^t)
  float eps;
  float* p;
  float* m;
  float* v;
};

struct CopyParams {        // strided 2D bf16 copy (pack / unpack of unaligned matrices)
  const uint16_t* src;
  uint16_t* dst;
  int64_t rows, cols, ld_src, ld_dst;
};

cudaError_t launch_reduce_momentum(const ReduceParams& p, int contrib_dtype, cudaStream_t s);
cudaError_t launch_norm_finalize(const NormParams& p, cudaStream_t s);
cudaError_t launch_apply_update(const UpdateParams& p, cudaStream_t s);
cudaError_t launch_adamw(const AdamParams& p, int contrib_dtype, cudaStream_t s);
cudaError_t launch_copy2d(const CopyParams& p, cudaStream_t s);
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* status, cudaStream_t s);
int* status_word_address();  // device address of this device's status word (nullptr on error)
uint64_t wait_limit_ns();    // limit of every bounded device-side wait (mfsdp_set_wait_limit_ns)

// ---- batched fp32 GEMM on the tensor cores, 3xTF32 (second-order optimizers) --------------
struct GemmDesc {          // C = alpha op(A) op(B) + beta C, row-major, one problem
  const float* a;
  const float* b;
  float* c;
  float* t_out;            // nullable: also write (5 delta_ij - C_ij) / 4 here
  int32_t m, n, k;
  int32_t lda, ldb, ldc;
  float alpha, beta;
};
// Every problem of the table in one persistent launch (one per 480 problems); ta / tb: op =
// transpose.  host_descs is the host copy of the device table dev_descs (the host orders the
// tiles from it).  Returns an MFSDP status.
int launch_gemm(const GemmDesc* dev_descs, const GemmDesc* host_descs, int nprob, int ta,
                int tb, cudaStream_t st);

// ---- Newton–Schulz grouped GEMM (tcgen05 / TMEM / TMA) ------------------------------------
constexpr int kBM = 128;   // tile rows    = UMMA M (one CTA, TMEM lanes 0..127)
constexpr int kBN = 256;   // tile columns = UMMA N
constexpr int kBK = 64;    // k per pipeline stage = one 128-byte swizzle atom of bf16
constexpr int kPairBM = 256;  // tile rows of the CTA-pair kernel (128 per CTA)
constexpr int kMapsPerHalf = 4;  // tensor maps per buffer half (see NsProblem::map_a)
constexpr int kNsThreads = 320;  // warp 0 TMA producer, warp 1 MMA issuer, warps 2-9 epilogue

enum NsKind : int32_t { kGram = 0, kPoly = 1, kApply = 2 };

struct NsProblem {         // one output matrix of one Newton–Schulz phase
  int32_t M, N, K;         // output M x N, contraction length K
  int32_t a_mn, b_mn;      // operand storage: 0 = K-major rows, 1 = MN-major rows
  int32_t sym;             // symmetric output: only tiles touching the upper triangle run
  int32_t kind;            // NsKind: epilogue out = alpha*acc + beta*D (see fold_a)
  int32_t first;           // first iteration: fold s = 1/(norm + eps) into alpha / beta
  int32_t mat;             // matrix index (norm)
  int32_t map_a, map_b;    // tensor-map indices of the hi operands (2D 64x64 box); +1: 2D
                           // 64x128 box, +2: 3D 64x64x2 MN-major view, +3: 2D 32x32 box with
                           // 64-byte swizzle (stores), +kMapsPerHalf: the lo half's maps
  int32_t mn3d;            // bit 0 / bit 1: the A / B operand is MN-major and has the 3D view
  int32_t map_o;           // tensor-map index of the output's 32x32 store box (hi, 64B swizzle)
  int32_t fold_a;          // 1: a X is folded into B' = a I + B (kPoly adds a on the diagonal,
                           // kApply has no addend); 0: kApply adds a * alpha * D
  const uint16_t* d_hi;    // epilogue addend D (kPoly: A, kApply without fold_a: X), pitch ldd
  const uint16_t* d_lo;
  int64_t ldd;
  uint16_t* o_hi;          // output, row pitch ldo
  uint16_t* o_lo;
  int64_t ldo;
  uint16_t* t_hi;          // split epilogue only, nullable: also T = (5 I - out) / 4 (pitch ldo)
  uint16_t* t_lo;
};

struct NsTile {
  int32_t prob, tm, tn, pad_;
};

struct NsLaunchParams {
  const NsProblem* probs;
  const NsTile* tiles;
  int32_t ntiles;
  int32_t pad_;
  const CUtensorMap* maps;
  const float* norm;
  float eps, a, b, c;
  uint64_t wait_limit_ns;
  int* status;
};

cudaError_t ns_prepare_kernels();  // set the dynamic shared memory attribute once per device
// co-resident CTA pairs of the pair kernel, bf16 or split operands (-1: error)
int ns_pair_max_clusters(int num_sms, bool split = false);
// split: single-CTA kernel, `grid` CTAs; else the CTA-pair kernel, `grid` pairs.
cudaError_t launch_ns_phase(const NsLaunchParams& p, bool split, int grid, cudaStream_t s);
// The CTA-pair kernel with split (hi + lo) operands and outputs: 256 x 256 tiles (tiles built
// with 256-row blocks), `pairs` pairs.
cudaError_t launch_ns_pair_split(const NsLaunchParams& p, int pairs, cudaStream_t s);

// 2D bf16 tensor map over a rows x cols row-major buffer of pitch ld elements (box_rows x
// box_cols boxes; 128-byte swizzle, or 64-byte for the epilogue's store boxes) and the 3D
// MN-major view; false when the driver refuses the map.
bool encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                uint32_t box_rows, uint32_t box_cols = 64, bool swizzle128 = true);
bool encode_map3d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld);
// 2D fp32 tensor map (boxes of 32 columns x box_rows rows, 128-byte swizzle); false when the
// driver refuses it (the base must be 16-byte aligned and ld a multiple of 4).
bool encode_map_f32(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t box_rows);
// Output tiles (bm x kBN) of one problem in the rasterised order; `sym` keeps the tiles that
// reach the upper triangle.
void add_tiles(std::vector<NsTile>& out, int32_t prob, int64_t M, int64_t N, bool sym,
               int64_t bm);

}  // namespace mfsdp
