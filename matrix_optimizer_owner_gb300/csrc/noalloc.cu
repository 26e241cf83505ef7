// mfsdp_owner_reduce_momentum_noalloc: the gradient deposit + momentum + norm call for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs under another system's device-memory manager (a host framework
// or serving runtime that owns every byte of device memory and gives plugins no way to call
// cudaMalloc), and processes that reserve device memory once at start-up and must never
// allocate on the training-step path.  Such callers cannot provide the workspace that
// mfsdp_owner_set_bind needs.  This entry point keeps its scratch (the matrix table and the
// per-CTA norm partials) in one fixed array in the library's own device memory instead; it
// allocates nothing, on the device or the host.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds its
// 4 MiB until the process exits.  In host code its name is only a stand-in, not a device
// address, so the address is looked up with cudaGetSymbolAddress once per device (the first
// call on a device does this, with that device current) and passed to the kernels.
#include <cstring>
#include <mutex>

#include "mfsdp.h"
#include "mfsdp_internal.h"

// The scratch of every call on this device: [matrix table | per-CTA norm partials].
static __device__ __align__(256) unsigned char g_noalloc_scratch[MFSDP_NOALLOC_SCRATCH_BYTES];

namespace mfsdp {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kTableBytes = (size_t)MFSDP_NOALLOC_MAX_MATRICES * sizeof(DevMat);
static_assert(kTableBytes % 256 == 0 && kTableBytes < MFSDP_NOALLOC_SCRATCH_BYTES, "layout");

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MFSDP_ENODEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MFSDP_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MFSDP_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Up to 64 table entries travel as one kernel's parameters (3 KB) and one thread per entry
// stores them into the scratch table.  The runtime copies a launch's parameters when the launch
// is issued, so the table never depends on host memory after this call returns.
constexpr int kTableBatch = 64;
struct TableBatch {
  DevMat m[kTableBatch];
  int32_t first, count;
};
static_assert(sizeof(TableBatch) <= 4000, "table batch must fit the kernel parameter space");

__global__ void write_table_kernel(const TableBatch b, DevMat* table) {
  const int k = threadIdx.x;
  if (k < b.count) table[b.first + k] = b.m[k];
}

}  // namespace
}  // namespace mfsdp

using namespace mfsdp;

extern "C" int mfsdp_owner_reduce_momentum_noalloc(
    const mfsdp_matrix* mats, int32_t n_mats, int64_t split_max_numel, const void* const* contrib,
    int32_t W, int32_t contrib_dtype, float grad_scale, float momentum, int32_t nesterov,
    float* momentum_buf, void* ns_input, void* ns_input_lo, float* reduced_grad_out,
    float* norm_out, void* stream) {
  if (n_mats < 0 || (n_mats > 0 && !mats)) return MFSDP_EINVAL;
  if (n_mats > MFSDP_NOALLOC_MAX_MATRICES) return MFSDP_EWORKSPACE;
  // Shapes, overlap, and the number of per-CTA partials the scratch must hold.
  int64_t ctas = 0;
  for (int32_t i = 0; i < n_mats; ++i) {
    const mfsdp_matrix& q = mats[i];
    if (q.rows < 0 || q.cols < 0 || q.offset < 0 || q.rows >= (1ll << 31) || q.cols >= (1ll << 31))
      return MFSDP_ESHAPE;
    ctas += (q.rows * q.cols + kChunk - 1) / kChunk;
    if ((size_t)ctas * sizeof(float) > MFSDP_NOALLOC_SCRATCH_BYTES - kTableBytes)
      return MFSDP_EWORKSPACE;
  }
  for (int32_t i = 0; i < n_mats; ++i) {
    const int64_t ni = mats[i].rows * mats[i].cols;
    for (int32_t j = i + 1; j < n_mats && ni > 0; ++j) {
      const int64_t nj = mats[j].rows * mats[j].cols;
      if (nj > 0 && mats[i].offset < mats[j].offset + nj && mats[j].offset < mats[i].offset + ni)
        return MFSDP_ESHAPE;
    }
  }
  if (!contrib || W < 1 || W > kMaxContrib) return MFSDP_EINVAL;
  if (contrib_dtype != MFSDP_DTYPE_F32 && contrib_dtype != MFSDP_DTYPE_BF16) return MFSDP_EINVAL;
  if (!momentum_buf || !ns_input || !norm_out) return MFSDP_EINVAL;
  for (int32_t w = 0; w < W; ++w) {
    if (!contrib[w]) return MFSDP_EINVAL;
    if (!aligned16(contrib[w])) return MFSDP_EALIGN;
  }
  if (!aligned16(momentum_buf) || !aligned16(ns_input) || !aligned16(norm_out) ||
      (ns_input_lo && !aligned16(ns_input_lo)) || (reduced_grad_out && !aligned16(reduced_grad_out)))
    return MFSDP_EALIGN;
  if (n_mats == 0) return MFSDP_OK;

  void* scratch = nullptr;
  int st = scratch_address(&scratch);
  if (st != MFSDP_OK) return st;
  int* status = status_word_address();
  if (!status) return MFSDP_ECUDA;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevMat* table = static_cast<DevMat*>(scratch);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(scratch) + kTableBytes);

  // The matrix table, written in batches of 64 entries by a one-CTA kernel that receives them
  // as its parameters (no host allocation, and no copy from host memory that must outlive the
  // call).
  TableBatch batch;
  int32_t cta = 0;
  for (int32_t i0 = 0; i0 < n_mats; i0 += kTableBatch) {
    const int32_t cnt = n_mats - i0 < kTableBatch ? n_mats - i0 : kTableBatch;
    std::memset(&batch, 0, sizeof(batch));
    batch.first = i0;
    batch.count = cnt;
    for (int32_t k = 0; k < cnt; ++k) {
      const mfsdp_matrix& q = mats[i0 + k];
      DevMat& d = batch.m[k];
      d.offset = q.offset;
      d.numel = q.rows * q.cols;
      d.rows = q.rows;
      d.cols = q.cols;
      d.cta_begin = cta;
      d.split = d.numel > 0 && d.numel <= split_max_numel;
      cta += (int32_t)((d.numel + kChunk - 1) / kChunk);
    }
    write_table_kernel<<<1, kTableBatch, 0, s>>>(batch, table);
    if (cudaGetLastError() != cudaSuccess) return MFSDP_ECUDA;
  }

  // Every partial is written by its CTA before the norm kernel reads it, so nothing in the
  // scratch has to start at zero.
  ReduceParams p{};
  for (int32_t w = 0; w < W; ++w) p.contrib.p[w] = contrib[w];
  p.W = W;
  p.n_mats = n_mats;
  p.total_ctas = cta;
  p.nesterov = nesterov ? 1 : 0;
  p.offsets_aligned = 1;
  for (int32_t i = 0; i < n_mats; ++i)
    if (mats[i].rows * mats[i].cols > 0 && mats[i].offset % 8 != 0) p.offsets_aligned = 0;
  p.wait_limit_ns = wait_limit_ns();
  p.status = status;
  p.mats = table;
  p.grad_scale = grad_scale;
  p.mu = momentum;
  p.one_minus_mu = (float)(1.0 - (double)momentum);
  p.momentum = momentum_buf;
  p.uhat = static_cast<uint16_t*>(ns_input);
  p.uhat_lo = static_cast<uint16_t*>(ns_input_lo);
  p.grad = reduced_grad_out;
  p.partials = partials;
  if (launch_reduce_momentum(p, contrib_dtype, s) != cudaSuccess) return MFSDP_ECUDA;
  NormParams q{};
  q.mats = table;
  q.n_mats = n_mats;
  q.partials = partials;
  q.norm = norm_out;
  q.status = status;
  return launch_norm_finalize(q, s) == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}
