/*
 * mfsdp.h — C ABI of the owner-local Muon optimizer step on one GB300 (sm_103a).
 *
 * Source: "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding"
 * (academ.us/article/2607.05895).  Under owner-shaped ZeRO-3 placement (§3) every 2D weight is
 * whole on one owner rank, so after the backward gradient reduction has deposited the full
 * gradient there, the owner's Muon step needs no communication (§3, §4.4).  This library is
 * that owner-local step:
 *
 *   mfsdp_plan_owner_set          owner assignment + segment table (host only)   §4.1
 *   mfsdp_score_plan              per-rank resource estimates, gamma_B (host)     §4.1, §4.2
 *   mfsdp_plan_cost_aware         CostAware: scope plan within a workspace cap    §4.1
 *   mfsdp_pack_owner_shards /     canonical axis <-> owner shards (reshard load)  §4.4
 *   mfsdp_unpack_owner_shards
 *   mfsdp_shampoo_step            owner Shampoo (L/R inverse fourth roots)         §5.7
 *   mfsdp_soap_step               owner SOAP (Adam in the Shampoo eigenbasis)      §5.7
 *   mfsdp_owner_reduce_momentum   W-way gradient deposit + Nesterov momentum + norm  §3, §4.2
 *   mfsdp_newton_schulz           quintic Newton–Schulz of every owned matrix      §2
 *   mfsdp_apply_update            scaled update with decoupled weight decay        §5.1
 *   mfsdp_adamw_tail              AdamW on the packed non-2D tail                  §3, §5.1
 *
 * Conventions shared by every call:
 *   - Pointers named *_dev / buffers are DEVICE pointers (cudaMalloc'd or torch tensors on the
 *     current device); descriptor arrays (mfsdp_param_desc, mfsdp_matrix, contribution pointer
 *     lists) are HOST arrays read during the call and not retained.
 *   - The caller owns all memory, including the workspace.  The library never allocates or
 *     frees device memory.  Its only device-side global state is one status word per device.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work is enqueued on
 *     it and the call returns without synchronising.
 *   - Every argument is validated before anything is launched; a negative mfsdp_status is
 *     returned and nothing is enqueued.  MFSDP_ECUDA reports a CUDA runtime failure.
 *     Conditions found on the device (a bounded wait that ran out, a non-finite norm) are
 *     recorded in the device status word and returned by mfsdp_query_status.
 *   - bf16 buffers hold IEEE bfloat16 values (uint16_t storage).  fp32 buffers are float.
 *     All device buffers must be 16-byte aligned.
 *   - Matrices are row-major rows x cols.  m = min(rows, cols), n = max(rows, cols).
 */
#ifndef MFSDP_H
#define MFSDP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MFSDP_OK = 0,
  MFSDP_EINVAL = -1,      /* null pointer, bad enum, bad count, unbound set, mismatched buffer */
  MFSDP_ESHAPE = -2,      /* negative or oversized dimension, overlapping matrices */
  MFSDP_EALIGN = -3,      /* a device pointer is not 16-byte aligned, workspace not 256-aligned */
  MFSDP_ENOTCONTIG = -4,  /* a plan would give a parameter more than one local segment */
  MFSDP_EWORKSPACE = -5,  /* workspace smaller than mfsdp_owner_set_workspace_bytes() */
  MFSDP_ECUDA = -6,       /* a CUDA runtime / driver call failed */
  MFSDP_ETIMEOUT = -7,    /* device status: a bounded device-side wait ran out */
  MFSDP_ENONFINITE = -8,  /* device status: a matrix norm (Muon) or update (Shampoo, SOAP) was
                             NaN or Inf */
  MFSDP_ENODEVICE = -9    /* no usable sm_103 device for a device call */
} mfsdp_status;

/* ------------------------------------------------------------------------------------------
 * Owner planning (§3, §4.1, §4.2).  Host only; needs no GPU.
 * ------------------------------------------------------------------------------------------ */

typedef struct {
  int64_t rows;       /* >= 0 */
  int64_t cols;       /* >= 0; vectors use cols = 1 */
  int32_t block;      /* FSDP unit id; blocks are visited in order of first appearance */
  int32_t is_matrix;  /* 1 = 2D weight (Muon role of its own), 0 = joins the block's tail role */
} mfsdp_param_desc;

typedef struct {
  int32_t owner;         /* owner rank in [0, world_size) */
  int32_t role;          /* role id: blocks in order, roles by first declaration index */
  int64_t local_offset;  /* element offset in the owner's block-local shard */
  int64_t rank_offset;   /* element offset in the owner's flat matrix buffer (matrices) or
                            flat tail buffer (vectors); both in (block, declaration) order */
  int64_t numel;
} mfsdp_segment;

typedef enum {
  MFSDP_POLICY_ROLE_GREEDY = 0,  /* per block, largest role first, to the least-loaded rank */
  MFSDP_POLICY_SCOPE_GREEDY = 1  /* the same rule over the roles of all blocks pooled */
} mfsdp_policy;

/*
 * Assign every role (one per 2D matrix, one packed non-2D tail per block; §3) to an owner
 * rank and lay out the owned segments (§4.1).  The load is the numel resident on the owner; ties go to
 * the lowest rank.  Within each (block, rank) the owned roles are laid out by first
 * declaration index, a role's parameters in declaration order, unpadded, so every parameter
 * has one contiguous local segment and a tail is one whole segment.
 *
 *   params          [n_params] host array, declaration order.
 *   seg_out         [n_params] host array, written.
 *   block_rank_numel_out  nullable host array of capacity n_params * world_size; on return
 *                   entry [k * world_size + r] = O_{B_k, r} (§4.2), numel of the k-th block
 *                   (first-appearance order) resident on rank r.
 *   n_blocks_out    nullable; receives the number of distinct blocks.
 * Errors: MFSDP_EINVAL (null params/seg_out with n_params > 0, world_size <= 0, bad policy),
 *         MFSDP_ESHAPE (negative dimension or numel overflow).
 * Deterministic and thread-safe.
 */
int mfsdp_plan_owner_set(const mfsdp_param_desc* params, int64_t n_params, int32_t world_size,
                         int32_t policy, mfsdp_segment* seg_out, int64_t* block_rank_numel_out,
                         int64_t* n_blocks_out);

/* Element sizes and step length the resource scorer prices a plan with. */
typedef struct {
  int32_t param_bytes;  /* bytes per parameter element (2 = bf16) */
  int32_t grad_bytes;   /* bytes per gradient element */
  int32_t state_bytes;  /* bytes per optimizer-state element (4 = fp32) */
  int32_t ns_steps;     /* Newton–Schulz iterations per optimizer step */
} mfsdp_cost_model;

/* Per-rank estimates of a plan (§4.1 resource scorer).  The pages name these quantities but
 * give no formulas; with O_{B,r} the numel of block B owned by rank r, P_B the numel of
 * block B and W the world size:
 *   param_bytes / grad_bytes  owned numel x element size;
 *   state_bytes               (owned matrix numel + 2 x owned tail numel) x state size
 *                             (Muon momentum; AdamW first and second moments);
 *   comm_bytes                one owner-segment collective over every block (materialise or
 *                             gradient reduce), sent + received:
 *                             sum_B ((W - 1) O_{B,r} + P_B - O_{B,r}) x param_bytes;
 *   workspace_bytes           receive buffers of the gradient reduce into the rank's owner
 *                             segments: max_B (W - 1) O_{B,r} x grad_bytes;
 *   optimizer_flops           nominal Newton–Schulz FLOPs of the owned matrices,
 *                             ns_steps x (4 m^2 n + 2 m^3), m = min(rows, cols), n = max. */
typedef struct {
  int64_t param_bytes;
  int64_t grad_bytes;
  int64_t state_bytes;
  int64_t comm_bytes;
  int64_t workspace_bytes;
  double optimizer_flops;
} mfsdp_rank_resources;

/*
 * Score a plan made by mfsdp_plan_owner_set (or any segment table with one owner per
 * parameter).
 *   segs       [n_params] host array; only owner and numel are read.
 *   model      element sizes (each >= 1) and ns_steps (>= 0).
 *   ranks_out  [world_size] host array, written.
 *   gamma_out  nullable host array of capacity n_params; entry k = gamma_{B_k} =
 *              max_r O_{B_k,r} / (P_{B_k} / W) (§4.2) for the k-th block in first-appearance
 *              order, 0 for an empty block.
 *   n_blocks_out  nullable; receives the number of blocks.
 * Errors: MFSDP_EINVAL (null arrays with n_params > 0, world_size <= 0, bad model, an owner
 *         outside [0, world_size)), MFSDP_ESHAPE (negative dimension, numel != rows x cols,
 *         byte-count overflow).
 */
int mfsdp_score_plan(const mfsdp_param_desc* params, int64_t n_params, int32_t world_size,
                     const mfsdp_segment* segs, const mfsdp_cost_model* model,
                     mfsdp_rank_resources* ranks_out, double* gamma_out, int64_t* n_blocks_out);

/*
 * CostAware (§4.1): plan with RoleGreedy and with ScopeGreedy and take the scope plan only if
 * its largest per-rank workspace_bytes (as scored above) is at most workspace_cap_bytes; a
 * cap <= 0 stands for the role plan's own largest workspace.  Otherwise the role plan.
 *   seg_out     [n_params] host array, written with the plan taken.
 *   policy_out  nullable; receives MFSDP_POLICY_SCOPE_GREEDY or MFSDP_POLICY_ROLE_GREEDY.
 * Errors: as mfsdp_plan_owner_set and mfsdp_score_plan.
 */
int mfsdp_plan_cost_aware(const mfsdp_param_desc* params, int64_t n_params, int32_t world_size,
                          const mfsdp_cost_model* model, int64_t workspace_cap_bytes,
                          mfsdp_segment* seg_out, int32_t* policy_out);

/* ------------------------------------------------------------------------------------------
 * Owner-segment repacking (§4.1, §4.2, §4.4): moving parameters (or gradients, or optimizer
 * state of the same shape) between the canonical axis and owner shards.
 *
 * Layouts.  Canonical buffer: the parameters back to back in declaration order, parameter i
 * at sum_{j<i} numel_j elements.  Owner shard of rank r: r's block-local shards back to back
 * in block order (first appearance), parameter i (owned by r) at
 * sum_{B' before B} O_{B',r} + segs[i].local_offset elements — the concatenation of the
 * FSDP block shards a plan from mfsdp_plan_owner_set gives rank r.
 *
 * Reshard load (§4.4) is mfsdp_unpack_owner_shards under the saved plan followed by
 * mfsdp_pack_owner_shards under the target plan and world size.
 *
 * Common arguments:
 *   params, segs   [n_params] host arrays; segs as written by mfsdp_plan_owner_set (owner,
 *                  local_offset, numel are read; numel must equal rows x cols and each
 *                  segment must lie inside its block-local shard).
 *   elem_bytes     element size: 1, 2, 4 or 8.  Elements are copied bit for bit.
 *   shards         host array of world_size DEVICE pointers, one owner shard per rank; a NULL
 *                  entry skips that rank (a rank that holds only its own shard passes the
 *                  others as NULL).
 *   canonical      DEVICE pointer to the canonical buffer.
 *   workspace      DEVICE buffer of at least mfsdp_repack_workspace_bytes(n_params) bytes for
 *                  the copy table; reused by the next call on the same stream.
 * Buffers may start at any element boundary; ranges whose source and destination share their
 * alignment mod 16 bytes move as 16-byte vectors.  Source and destination must not overlap.
 * Errors: MFSDP_EINVAL (null arrays, world_size <= 0, bad elem_bytes, owner out of range),
 *         MFSDP_ESHAPE (numel mismatch, a segment outside its shard), MFSDP_EWORKSPACE,
 *         MFSDP_ECUDA.  Enqueued on `stream`; returns without synchronising.
 * ------------------------------------------------------------------------------------------ */

int mfsdp_repack_workspace_bytes(int64_t n_params, size_t* bytes_out);

/* Canonical buffer -> the owner shard of every rank whose shards[r] is not NULL. */
int mfsdp_pack_owner_shards(const mfsdp_param_desc* params, int64_t n_params,
                            const mfsdp_segment* segs, int32_t world_size, int32_t elem_bytes,
                            const void* canonical, void* const* shards, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Owner shards of the ranks whose shards[r] is not NULL -> their parameters' places in the
 * canonical buffer (the rest of the canonical buffer is left as it was). */
int mfsdp_unpack_owner_shards(const mfsdp_param_desc* params, int64_t n_params,
                              const mfsdp_segment* segs, int32_t world_size, int32_t elem_bytes,
                              const void* const* shards, void* canonical, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------------------------
 * The owned-matrix set.  Built once from the owner's matrix table; its launch tables, tensor
 * maps and Newton–Schulz scratch live in a caller-provided device workspace.
 * ------------------------------------------------------------------------------------------ */

typedef struct {
  int64_t rows, cols;  /* >= 0; an empty matrix is skipped by every call */
  int64_t offset;      /* element offset of the matrix in the flat owner buffers */
} mfsdp_matrix;

/* ------------------------------------------------------------------------------------------
 * Owner Shampoo (§5.7): the owner's whole matrices preconditioned with full left and right
 * statistics and their inverse fourth roots, in place of Muon.  For every matrix G (rows x
 * cols) of the set, one step is
 *     L += G G^T,   R += G^T G                     (L, R start at eps I)
 *     P  = L^{-1/4} G R^{-1/4}
 *     W  = W (1 - lr weight_decay) - lr P
 * The pages name the preconditioners and the inverse fourth root only; this is the original
 * Shampoo update.  The roots come from `root_iters` steps of the coupled Newton iteration for
 * the inverse p-th root (p = 4), started from X = c^{-1/4} I, M = A / c with c = ||A||_F; an
 * eigenvalue ratio of 1e-8 converges within 26 steps.
 *
 * `precision` selects where the products run:
 *   MFSDP_SHAMPOO_FP32        every product an fp32 GEMM on the tcgen05 tensor cores in
 *                             3xTF32 (mfsdp_gemm_f32_batched below: about 21 significant
 *                             bits per product, the accuracy of an fp32 FFMA GEMM);
 *   MFSDP_SHAMPOO_SPLIT_BF16  the statistics as above; the root iteration and P = X_L G X_R on
 *                             the tcgen05 tensor cores with split-bf16 operands (value = hi +
 *                             lo, three products per multiply, fp32 accumulation: about 16
 *                             significant bits per stored value, so the roots carry a relative
 *                             error near 1e-4 where the fp32 path reaches 1e-6).  It resolves
 *                             statistics whose eigenvalues span about four decades: below
 *                             ~1e-5 of the largest, bf16 pairs hold only rounding noise, which
 *                             can be negative and make the iteration diverge (then the
 *                             non-finite status below is set); use the fp32 precision, or a
 *                             larger eps, for statistics spread wider than that.
 *
 * Buffers (DEVICE, fp32, caller-owned): `grad` and `weights` are the flat owner buffers the
 * matrix table's offsets index (grad = the deposited gradient, e.g. the reduced_grad_out of
 * mfsdp_owner_reduce_momentum); `l` / `r` hold every matrix's L (rows^2) / R (cols^2) back to
 * back in table order (sizes from mfsdp_shampoo_set_sizes).  The workspace holds the root
 * iteration's buffers (7 x (rows^2 + cols^2) values per matrix), P, the tensor maps and the
 * launch tables; its size covers both precisions.
 * A non-finite P sets MFSDP_ENONFINITE in the device status word (mfsdp_query_status).
 * Errors: MFSDP_EINVAL (null pointers, eps <= 0, root_iters outside [1, 200], unknown
 * precision), MFSDP_ESHAPE
 * (rows or cols outside [1, 65536], negative offset), MFSDP_EWORKSPACE, MFSDP_ECUDA.
 * ------------------------------------------------------------------------------------------ */

typedef struct mfsdp_shampoo_set mfsdp_shampoo_set;

#define MFSDP_SHAMPOO_FP32 0
#define MFSDP_SHAMPOO_SPLIT_BF16 1

int mfsdp_shampoo_set_create(const mfsdp_matrix* mats, int32_t n_mats, mfsdp_shampoo_set** out);
int mfsdp_shampoo_set_destroy(mfsdp_shampoo_set* set);
/* Workspace bytes and the numel of the flat L and R buffers (any output may be NULL). */
int mfsdp_shampoo_set_sizes(const mfsdp_shampoo_set* set, size_t* workspace_bytes,
                            int64_t* l_numel, int64_t* r_numel);
/* L = R = eps I for every matrix. */
int mfsdp_shampoo_init_state(const mfsdp_shampoo_set* set, float eps, float* l, float* r,
                             void* workspace, size_t workspace_bytes, void* stream);
/* One Shampoo step of every matrix in the set (enqueued on `stream`). */
int mfsdp_shampoo_step(const mfsdp_shampoo_set* set, const float* grad, float* l, float* r,
                       float* weights, float lr, float weight_decay, int32_t root_iters,
                       int32_t precision, void* workspace, size_t workspace_bytes,
                       void* stream);


/* ------------------------------------------------------------------------------------------
 * Batched fp32 GEMM on the tensor cores (§5.7: the contractions of the second-order owner
 * optimizers, G G^T and G^T G for the statistics, the products of the root iteration and of
 * the preconditioning, the rotations into and out of an eigenbasis).  For every problem i:
 *     C_i = alpha_i op(A_i) op(B_i) + beta_i C_i,    op(A_i): m x k,  op(B_i): k x n
 * op(A) = A (stored m x k, pitch lda >= k) or A^T when trans_a (A stored k x m, lda >= m);
 * op(B) = B (stored k x n, ldb >= n) or B^T when trans_b (B stored n x k, ldb >= k); C is
 * m x n with pitch ldc >= n.  All row-major fp32 in DEVICE memory; C may not overlap A or B
 * (beta = 0: C is not read).  The problems run in persistent tcgen05 launches (up to 480
 * problems each; with trans_a = 0, trans_b = 1, 16-byte-aligned A and B and lda, ldb
 * multiples of 4, up to 64 each, the operand tiles then loaded by TMA):
 * values are cut into a TF32 high part and an fp32 remainder and each multiply is three
 * TF32 products (hi hi + hi lo + lo hi) accumulated in fp32, about 21 significant bits per
 * product.  `workspace` (DEVICE, >= mfsdp_gemm_f32_workspace_bytes(n_probs) bytes, 256-byte
 * aligned) receives the problem table.  n_probs == 0 or an empty problem is no work.
 * Errors: MFSDP_EINVAL (null table or pointers, negative sizes, a pitch below its minimum),
 * MFSDP_EWORKSPACE, MFSDP_ECUDA; a wait that runs out on the device sets MFSDP_ETIMEOUT in the
 * status word.
 * ------------------------------------------------------------------------------------------ */

typedef struct {
  const float* a;
  const float* b;
  float* c;
  int32_t m, n, k;
  int32_t lda, ldb, ldc;
  float alpha, beta;
} mfsdp_gemm_problem;

size_t mfsdp_gemm_f32_workspace_bytes(int32_t n_probs);
int mfsdp_gemm_f32_batched(const mfsdp_gemm_problem* probs, int32_t n_probs, int32_t trans_a,
                           int32_t trans_b, void* workspace, size_t workspace_bytes,
                           void* stream);

/* ------------------------------------------------------------------------------------------
 * Owner SOAP (§5.7): Adam run in the eigenbasis of the Shampoo statistics, on the owner's
 * whole matrices, in place of Muon.  For every matrix G (rows x cols) of the set and step
 * t >= 1 (the pages name the method only; this is the SOAP update with the eigenbasis taken
 * exactly at every step):
 *     L = bs L + (1 - bs) G G^T,   R = bs R + (1 - bs) G^T G
 *     Q_L, Q_R = eigenvectors of L, R (columns), in descending eigenvalue order
 *     M = b1 M + (1 - b1) G                      (parameter coordinates)
 *     G' = Q_L^T G Q_R,  M' = Q_L^T M Q_R
 *     V = b2 V + (1 - b2) G'^2                   (eigenbasis coordinates)
 *     N = Q_L [ (M' / (1 - b1^t)) / (sqrt(V / (1 - b2^t)) + eps) ] Q_R^T
 *     W = W (1 - lr weight_decay) - lr N
 * The eigenbases come from cyclic block Jacobi on Q^T L Q, started from the basis the state
 * holds (the previous step's), until a sweep rotates nothing or `max_sweeps` sweeps ran;
 * each solve ends with one polar step on its basis (Z <- Z (3I - Z^T Z) / 2); the statistics,
 * Q^T L Q, that polar step, the Rayleigh quotients and the rotations into and out of the
 * eigenbasis are fp32 GEMMs on the tensor cores (3xTF32, as mfsdp_gemm_f32_batched); the
 * Jacobi rotations of Q^T L Q run in fp32 on the CUDA cores, those of the basis on the tensor
 * cores (3xTF32).  Eigenvectors are fixed up to sign, and N does not
 * depend on the signs.  The Jacobi sweeps run as a CUDA graph that the set builds at its
 * first refresh step for a given workspace and max_sweeps and launches on `stream`: per group
 * of sides a while loop whose body is one sweep, ending on the device once every side of the
 * group has converged.  While `stream` is being captured (or if the graph cannot be built)
 * the same sweeps are issued one by one on `stream` and three internal streams of the set,
 * forked from and joined back into `stream` with events, so a capture of `stream` takes them
 * all; so does MFSDP_SOAP_SWEEP_GRAPH=0 in the environment (read once per process), for
 * profilers that do not list kernels inside conditional graph nodes.  Streams, events and the
 * graph are created on the device current at the first step; a set serves one host thread at
 * a time.
 *
 * State (DEVICE, fp32, caller-owned, updated in place): `l`, `q_l` hold every matrix's L and
 * Q_L (rows^2 each) back to back in table order, `r`, `q_r` its R and Q_R (cols^2); `eig_l`
 * (sum of rows) and `eig_r` (sum of cols) the eigenvalues, descending per matrix;
 * `exp_avg` (M) and `exp_avg_sq` (V) are flat owner buffers indexed like the weights.
 * mfsdp_soap_init_state sets L = R = 0, Q = I, eigenvalues, M and V to 0; a caller may write
 * any symmetric positive semi-definite L, R and any orthogonal Q there instead.
 * `grad` and `weights` are the flat owner buffers (fp32).  `info` (DEVICE, nullable,
 * 2 x n_mats int32: L sides, then R sides) receives the sweeps each solve used, negated when
 * it stopped at max_sweeps (0 for every side when the step does not refresh).  A non-finite
 * N sets MFSDP_ENONFINITE in the device status word.
 * Errors: MFSDP_EINVAL (null pointers, t < 1, max_sweeps outside [1, 100], a beta outside
 * [0, 1), eps < 0, jacobi_tol outside [0, 1e-2), refresh not 0 or 1), MFSDP_ESHAPE (rows or cols outside [1, 65536], negative offset),
 * MFSDP_EWORKSPACE, MFSDP_ECUDA.
 * ------------------------------------------------------------------------------------------ */

typedef struct mfsdp_soap_set mfsdp_soap_set;

typedef struct {
  float* l;
  float* r;
  float* q_l;
  float* q_r;
  float* eig_l;
  float* eig_r;
  float* exp_avg;
  float* exp_avg_sq;
} mfsdp_soap_state;

typedef struct {
  float lr, beta1, beta2, beta_stats, eps, weight_decay;
  int32_t max_sweeps;
  float jacobi_tol;  /* couplings below jacobi_tol * ||L|| are not rotated; 0: 1e-6 */
  int32_t refresh;   /* 1: recompute the eigenbases this step; 0: keep the state's Q and
                        eigenvalues (SOAP's preconditioning frequency: refresh every f steps) */
} mfsdp_soap_hyper;

int mfsdp_soap_set_create(const mfsdp_matrix* mats, int32_t n_mats, mfsdp_soap_set** out);
int mfsdp_soap_set_destroy(mfsdp_soap_set* set);
/* Workspace bytes and the numel of the flat L (= Q_L), R (= Q_R) and eigenvalue buffers. */
int mfsdp_soap_set_sizes(const mfsdp_soap_set* set, size_t* workspace_bytes, int64_t* l_numel,
                         int64_t* r_numel, int64_t* eig_l_numel, int64_t* eig_r_numel);
int mfsdp_soap_init_state(const mfsdp_soap_set* set, const mfsdp_soap_state* state,
                          void* workspace, size_t workspace_bytes, void* stream);
/* One SOAP step of every matrix in the set (enqueued on `stream`). */
int mfsdp_soap_step(const mfsdp_soap_set* set, const float* grad, float* weights,
                    const mfsdp_soap_state* state, int64_t t, const mfsdp_soap_hyper* hyper,
                    int32_t* info, void* workspace, size_t workspace_bytes, void* stream);

typedef struct mfsdp_owner_set_s mfsdp_owner_set;

/*
 * Describe the owner's matrices.  `mats` [n_mats] host array: each matrix occupies
 * [offset, offset + rows*cols) of every flat per-element buffer (weights, momentum, NS input,
 * NS output); ranges must not overlap.  Matrices with rows*cols <= split_max_numel run
 * Newton–Schulz with split bf16 operands (value = hi + lo, three products per multiply,
 * about 16 significant bits); the others use plain bf16 operands with fp32 accumulation.
 * No device work; *out is a host object owned by the caller (mfsdp_owner_set_destroy).
 * Errors: MFSDP_EINVAL, MFSDP_ESHAPE (negative size, overlap, dimension >= 2^31).
 */
int mfsdp_owner_set_create(const mfsdp_matrix* mats, int32_t n_mats, int64_t split_max_numel,
                           mfsdp_owner_set** out);
int mfsdp_owner_set_destroy(mfsdp_owner_set* set);

/* Device workspace bytes the set needs (launch tables, norm partials, tensor maps, the
 * Newton–Schulz ping buffer and the m x m Gram / polynomial buffers of every matrix). */
int mfsdp_owner_set_workspace_bytes(const mfsdp_owner_set* set, size_t* bytes_out);

/* Number of matrices that run in split (hi + lo) precision. */
int mfsdp_owner_set_split_count(const mfsdp_owner_set* set, int32_t* count_out);

/*
 * Bind the set to its device buffers on the current device and write its launch tables and
 * TMA tensor maps into `workspace` (enqueued on `stream`).  The workspace must stay untouched
 * by the caller while the set is bound.  ns_input / ortho_out are the flat bf16 buffers of
 * mfsdp_owner_reduce_momentum's output and mfsdp_newton_schulz's output; ns_input_lo /
 * ortho_lo are their low halves, required iff the set has split matrices (else may be NULL).
 * ns_input must not alias ortho_out.  Re-binding replaces the previous binding.
 * Errors: MFSDP_EINVAL, MFSDP_EALIGN, MFSDP_EWORKSPACE, MFSDP_ECUDA, MFSDP_ENODEVICE.
 */
int mfsdp_owner_set_bind(mfsdp_owner_set* set, void* workspace, size_t workspace_bytes,
                         const void* ns_input, const void* ns_input_lo, void* ortho_out,
                         void* ortho_lo, void* stream);

/* ------------------------------------------------------------------------------------------
 * The owner-local step.  All calls need a bound set; buffers are flat over the set.
 * ------------------------------------------------------------------------------------------ */

typedef enum { MFSDP_DTYPE_F32 = 0, MFSDP_DTYPE_BF16 = 1 } mfsdp_dtype;

/*
 * Owner gradient deposit fused with Nesterov momentum and the Frobenius norm (§3, §4.2: the
 * reduced full gradient lands in the owner segment; §2: Muon's input is the momentum-
 * buffered gradient).  Per element e of every matrix:
 *     G = grad_scale * sum_{w<W} contrib[w][e]          (fp32, w in order)
 *     B = momentum * B + (1 - momentum) * G             (momentum_buf, updated in place)
 *     U = nesterov ? (1 - momentum) * G + momentum * B : B
 *     ns_input[e] = bf16_rne(U);  ns_input_lo[e] = bf16_rne(U - ns_input[e])  (split matrices)
 *     reduced_grad_out[e] = G                            (nullable)
 * and per matrix i: norm_out[i] = ||U_i||_F of the fp32 U, reduced in a fixed order (per-CTA
 * fp32 partial sums, then an fp64 sum in index order): bitwise reproducible run to run.
 *   contrib  host array of W device pointers to flat contribution buffers (dtype contrib_dtype).
 *   W in [1, 64].  momentum_buf fp32 [flat]; ns_input bf16 [flat] (must be the bound buffer).
 *   norm_out fp32 [n_mats] device.
 * A non-finite norm sets MFSDP_ENONFINITE in the device status word.
 */
int mfsdp_owner_reduce_momentum(const mfsdp_owner_set* set, const void* const* contrib, int32_t W,
                                int32_t contrib_dtype, float grad_scale, float momentum,
                                int32_t nesterov, float* momentum_buf, void* ns_input,
                                void* ns_input_lo, float* reduced_grad_out, float* norm_out,
                                void* stream);

/*
 * Quintic Newton–Schulz orthogonalisation of every owned matrix (§2: steps built from
 * products such as X X^T that couple all rows).  Per matrix, with s = 1/(norm[i] + eps):
 *     X = s * U  (U = ns_input, + ns_input_lo for split matrices), transposed if rows > cols;
 *     repeat `steps` times:  A = X X^T;  B = b*A + c*A A;  X = a*X + B X
 *     with bf16 operands computed as A = X X^T;  B' = a*I + b*A + c*A A;  X = B' X
 *     (a X + B X = (a I + B) X); split matrices compute B and a X + B X as written.
 *     ortho_out = X (transposed back), ortho_lo = low half for split matrices.
 * Runs as three grouped, persistent tcgen05 GEMM launches per iteration over all matrices;
 * only the upper-triangle tiles of the symmetric A and A A are computed.  Operands are bf16
 * (or split bf16), accumulation fp32 in tensor memory; each phase's output is rounded to
 * bf16 once.  ns_input / ortho_out must be the bound buffers.  steps in [1, 64].
 * A device wait that runs out sets MFSDP_ETIMEOUT in the status word.
 */
int mfsdp_newton_schulz(const mfsdp_owner_set* set, const void* ns_input, const void* ns_input_lo,
                        const float* norm, int32_t steps, float a, float b, float c, float eps,
                        void* ortho_out, void* ortho_lo, void* stream);

typedef enum {
  MFSDP_LR_ORIGINAL = 0,        /* scale s = sqrt(max(1, rows/cols)) */
  MFSDP_LR_MATCH_RMS_ADAMW = 1  /* scale s = 0.2 * sqrt(max(rows, cols)) */
} mfsdp_lr_adjust;

/*
 * Scaled update with decoupled weight decay (§5.1: torch.optim.Muon semantics):
 *     W = W * (1 - lr*weight_decay) - lr * s(rows, cols) * (ortho + ortho_lo)
 * weights fp32 [flat] in place; ortho bf16 [flat]; ortho_lo bf16 [flat] or NULL (used only on
 * split matrices).
 */
int mfsdp_apply_update(const mfsdp_owner_set* set, float* weights, const void* ortho,
                       const void* ortho_lo, float lr, float weight_decay, int32_t lr_adjust,
                       void* stream);

/*
 * AdamW on a packed non-2D tail of n elements (§3: the tail is one whole segment on its
 * owner and stays on AdamW; §5.1 hyperparameters).  g = grad_scale * sum_w contrib[w];
 *     p = p*(1 - lr*wd);  m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g^2;
 *     p = p - lr * (m / (1 - b1^step)) / (sqrt(v / (1 - b2^step)) + eps)
 * param, exp_avg, exp_avg_sq fp32 [n] device, updated in place; step >= 1 (shared by the
 * whole tail).  Stateless: needs no owner set.  n == 0 returns MFSDP_OK without a launch.
 */
int mfsdp_adamw_tail(const void* const* contrib, int32_t W, int32_t contrib_dtype,
                     float grad_scale, int64_t n, float* param, float* exp_avg,
                     float* exp_avg_sq, int64_t step, float lr, float beta1, float beta2,
                     float eps, float weight_decay, void* stream);

/* ------------------------------------------------------------------------------------------
 * Gradient deposit without any allocation.  The paper has no counterpart to this call; it
 * exists for callers of this library that cannot allocate device memory: code running under
 * another system's memory manager (a framework or serving runtime that owns all device memory
 * and gives extensions no cudaMalloc), and processes that reserve memory once at start-up and
 * must not allocate on the step path.  They cannot provide the workspace of
 * mfsdp_owner_set_bind.
 * ------------------------------------------------------------------------------------------ */

#define MFSDP_NOALLOC_SCRATCH_BYTES (4u << 20) /* fixed per-device scratch, held until exit */
#define MFSDP_NOALLOC_MAX_MATRICES 4096

/*
 * Same computation and outputs as mfsdp_owner_reduce_momentum, for the matrices of the host
 * table `mats` [n_mats] (as in mfsdp_owner_set_create: rows, cols, element offset into the
 * flat buffers; ranges must not overlap).  Matrices with 0 < rows*cols <= split_max_numel
 * also get the low bf16 half in ns_input_lo (nullable: then no low half is written).  Needs no
 * owner set and no workspace: its scratch — the matrix table and one fp32 norm partial per
 * 16384 elements — lives in a fixed MFSDP_NOALLOC_SCRATCH_BYTES array in the library's own
 * device memory, and the call allocates nothing (no cudaMalloc / cudaFree, no allocating
 * library routine, no host heap).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture begins.
 *   - All calls on a device share the one array, and it keeps the last call's contents.
 *     Nothing in it needs to start at zero (every call rewrites the table, and each partial
 *     is written before it is read).  Calls whose work overlaps on the GPU — in different
 *     streams, or from different host threads — race on the array and give wrong results;
 *     order them on one stream.
 * Limits: n_mats <= MFSDP_NOALLOC_MAX_MATRICES and sum_i ceil(rows_i*cols_i / 16384) <=
 * (MFSDP_NOALLOC_SCRATCH_BYTES - MFSDP_NOALLOC_MAX_MATRICES*48) / 4 (about 16.4e9 elements);
 * larger problems return MFSDP_EWORKSPACE before anything is enqueued.
 * Other errors as mfsdp_owner_reduce_momentum.
 */
int mfsdp_owner_reduce_momentum_noalloc(const mfsdp_matrix* mats, int32_t n_mats,
                                        int64_t split_max_numel, const void* const* contrib,
                                        int32_t W, int32_t contrib_dtype, float grad_scale,
                                        float momentum, int32_t nesterov, float* momentum_buf,
                                        void* ns_input, void* ns_input_lo,
                                        float* reduced_grad_out, float* norm_out, void* stream);

/* ------------------------------------------------------------------------------------------
 * Status and diagnostics.
 * ------------------------------------------------------------------------------------------ */

/* Synchronise `stream`, read and clear the current device's status word.  *device_status_out
 * is MFSDP_OK, MFSDP_ETIMEOUT or MFSDP_ENONFINITE (timeout wins).  Returns MFSDP_ECUDA if the
 * synchronisation itself failed. */
int mfsdp_query_status(void* stream, int32_t* device_status_out);

/* Static description of a status code. */
const char* mfsdp_status_string(int status);

/* Limit, in nanoseconds, of every bounded device-side wait launched afterwards by this process
 * (default 2e9).  0 restores the default. */
int mfsdp_set_wait_limit_ns(uint64_t limit_ns);

/* Failure-detection check: launch one CTA that waits on an mbarrier nothing will arrive at,
 * bounded by limit_ns.  The wait runs out, the kernel records MFSDP_ETIMEOUT in the status
 * word and returns; the context stays usable. */
int mfsdp_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Library ABI version (major * 100 + minor). */
int mfsdp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MFSDP_H */
