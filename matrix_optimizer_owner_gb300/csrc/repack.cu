// Owner-segment repacking: canonical parameter axis <-> owner shards (host tables + one copy
// kernel).
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":
//   §4.1 every parameter has one contiguous local segment on its owner, inside the owner's
//        block-local shard of its FSDP block;
//   §4.2 owner-segment collectives move only the nonempty segments;
//   §4.4 reshard load rebuilds each parameter on its canonical [0, numel) axis from the saved
//        segments and repacks it into the target owner assignment and world size.
// Layouts: the canonical buffer holds the parameters back to back in declaration order; the
// owner shard of rank r holds r's block-local shards back to back in block order (first
// appearance), parameter i at sum_{B' before B} O_{B',r} + local_offset_i.
//
// Every call reduces to a list of contiguous byte ranges to copy (one per parameter whose
// destination is present).  The list goes to the caller's device workspace and one
// persistent kernel copies it: the concatenated bytes are cut into 32 KB pieces, CTAs take
// pieces round-robin, and each range is copied with 16-byte vectors wherever source and
// destination share their alignment (element copies otherwise).  The kernel is a plain
// HBM stream: read + write of every byte once.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <limits>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "mfsdp.h"
#include "mfsdp_internal.h"

namespace mfsdp {
namespace {

constexpr int kCopyThreads = 256;
constexpr int64_t kPiece = 32 * 1024;  // bytes per work item
constexpr int kCopyCtasPerSm = 4;

struct CopyDesc {
  const uint8_t* src;
  uint8_t* dst;
  int64_t bytes;
  int64_t start;  // offset of this range in the concatenated byte stream
};

// Up to kInlineDescs ranges travel in the launch's parameter space (no upload, no host wait);
// longer lists go through the caller's workspace.
constexpr int kInlineDescs = 800;

struct CopyParams {
  const CopyDesc* descs;  // the workspace table, or nullptr when the ranges are inline
  int64_t n_descs;
  int64_t total;  // bytes
  int32_t elem_bytes;
  CopyDesc inline_descs[kInlineDescs];
};
static_assert(sizeof(CopyParams) <= 32000, "kernel parameter space");

__device__ __forceinline__ int64_t find_desc(const CopyDesc* d, int64_t n, int64_t pos) {
  int64_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (d[mid].start <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void copy_elem(uint8_t* t, const uint8_t* s, int64_t k, int eb) {
  if (eb == 8)
    *reinterpret_cast<uint64_t*>(t + k) = *reinterpret_cast<const uint64_t*>(s + k);
  else if (eb == 4)
    *reinterpret_cast<uint32_t*>(t + k) = *reinterpret_cast<const uint32_t*>(s + k);
  else if (eb == 2)
    *reinterpret_cast<uint16_t*>(t + k) = *reinterpret_cast<const uint16_t*>(s + k);
  else
    t[k] = s[k];
}

// Copy bytes [a, b) of one range (a, b multiples of the element size).
__device__ void copy_part(const CopyDesc& d, int64_t a, int64_t b, int eb) {
  const uint8_t* s = d.src + a;
  uint8_t* t = d.dst + a;
  int64_t n = b - a;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(s), ta = reinterpret_cast<uintptr_t>(t);
  if (((sa ^ ta) & 15u) == 0) {
    // same alignment: element head up to a 16-byte boundary, vector body, element tail
    const int64_t h16 = (int64_t)((16u - (sa & 15u)) & 15u);
    const int64_t head = n < h16 ? n : h16;
    for (int64_t k = (int64_t)threadIdx.x * eb; k < head; k += (int64_t)kCopyThreads * eb)
      copy_elem(t, s, k, eb);
    s += head;
    t += head;
    n -= head;
    const int64_t nv = n >> 4;
    const uint4* sv = reinterpret_cast<const uint4*>(s);
    uint4* tv = reinterpret_cast<uint4*>(t);
    int64_t v = threadIdx.x;
    // 8 loads in flight per thread, then 8 stores
    for (; v + 7 * kCopyThreads < nv; v += 8 * kCopyThreads) {
      uint4 r[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) r[u] = __ldcs(sv + v + u * kCopyThreads);
#pragma unroll
      for (int u = 0; u < 8; ++u) __stcs(tv + v + u * kCopyThreads, r[u]);
    }
    for (; v < nv; v += kCopyThreads) __stcs(tv + v, __ldcs(sv + v));
    s += nv << 4;
    t += nv << 4;
    n -= nv << 4;
  }
  for (int64_t k = (int64_t)threadIdx.x * eb; k < n; k += (int64_t)kCopyThreads * eb)
    copy_elem(t, s, k, eb);
}

__global__ void __launch_bounds__(kCopyThreads) segment_copy_kernel(
    const __grid_constant__ CopyParams P) {
  const CopyDesc* descs = P.descs ? P.descs : P.inline_descs;
  const int64_t npieces = (P.total + kPiece - 1) / kPiece;
  for (int64_t pc = blockIdx.x; pc < npieces; pc += gridDim.x) {
    const int64_t p0 = pc * kPiece, p1 = P.total < p0 + kPiece ? P.total : p0 + kPiece;
    int64_t k = find_desc(descs, P.n_descs, p0);
    for (int64_t pos = p0; pos < p1 && k < P.n_descs; ++k) {
      const CopyDesc d = descs[k];
      const int64_t a = pos - d.start, b = d.bytes < p1 - d.start ? d.bytes : p1 - d.start;
      if (b > a) copy_part(d, a, b, P.elem_bytes);
      pos = d.start + d.bytes;
    }
  }
}

bool mul_ok(int64_t a, int64_t b) {
  return a >= 0 && b >= 0 && (a == 0 || b <= std::numeric_limits<int64_t>::max() / a);
}

// Canonical offsets and owner-shard offsets of every parameter (see the header comment).
int layout(const mfsdp_param_desc* params, int64_t n, const mfsdp_segment* segs, int32_t W,
           std::vector<int64_t>& canon, std::vector<int64_t>& shard) {
  canon.assign((size_t)n, 0);
  shard.assign((size_t)n, 0);
  std::unordered_map<int32_t, int32_t> pos;
  std::vector<int32_t> bpos((size_t)n);
  int64_t c = 0;
  for (int64_t i = 0; i < n; ++i) {
    const mfsdp_param_desc& p = params[i];
    if (!mul_ok(p.rows, p.cols)) return MFSDP_ESHAPE;
    const int64_t ne = p.rows * p.cols;
    if (segs[i].numel != ne || segs[i].local_offset < 0) return MFSDP_ESHAPE;
    if (segs[i].owner < 0 || segs[i].owner >= W) return MFSDP_EINVAL;
    canon[(size_t)i] = c;
    if (ne > std::numeric_limits<int64_t>::max() - c) return MFSDP_ESHAPE;
    c += ne;
    bpos[(size_t)i] = pos.emplace(p.block, (int32_t)pos.size()).first->second;
  }
  const int64_t nb = (int64_t)pos.size();
  std::vector<int64_t> o((size_t)(nb * W), 0), base((size_t)(nb * W), 0);
  for (int64_t i = 0; i < n; ++i) o[(size_t)(bpos[(size_t)i] * W + segs[i].owner)] += segs[i].numel;
  for (int32_t r = 0; r < W; ++r) {
    int64_t acc = 0;
    for (int64_t b = 0; b < nb; ++b) {
      base[(size_t)(b * W + r)] = acc;
      acc += o[(size_t)(b * W + r)];
    }
  }
  for (int64_t i = 0; i < n; ++i) {
    const size_t k = (size_t)(bpos[(size_t)i] * W + segs[i].owner);
    if (segs[i].local_offset + segs[i].numel > o[k]) return MFSDP_ESHAPE;  // outside its shard
    shard[(size_t)i] = base[k] + segs[i].local_offset;
  }
  return MFSDP_OK;
}

size_t desc_bytes(int64_t n) { return (size_t)std::max<int64_t>(n, 1) * sizeof(CopyDesc); }

int run_copies(std::vector<CopyDesc>& d, int32_t eb, void* ws, size_t ws_bytes, void* stream) {
  int64_t total = 0;
  std::vector<CopyDesc> live;
  live.reserve(d.size());
  for (CopyDesc& x : d) {
    if (x.bytes <= 0) continue;
    x.start = total;
    total += x.bytes;
    live.push_back(x);
  }
  if (live.empty()) return MFSDP_OK;
  if (ws_bytes < desc_bytes((int64_t)live.size())) return MFSDP_EWORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  static CopyParams p;  // large: kept off the stack; filled and launched under one lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  p.n_descs = (int64_t)live.size();
  p.total = total;
  p.elem_bytes = eb;
  if (live.size() <= (size_t)kInlineDescs) {
    p.descs = nullptr;
    std::copy(live.begin(), live.end(), p.inline_descs);
  } else {
    if (cudaMemcpyAsync(ws, live.data(), live.size() * sizeof(CopyDesc), cudaMemcpyHostToDevice,
                        st) != cudaSuccess)
      return MFSDP_ECUDA;
    p.descs = static_cast<const CopyDesc*>(ws);
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MFSDP_ECUDA;
  const int64_t npieces = (total + kPiece - 1) / kPiece;
  const int grid = (int)std::min<int64_t>(npieces, (int64_t)sms * kCopyCtasPerSm);
  segment_copy_kernel<<<grid, kCopyThreads, 0, st>>>(p);
  // (a copy from pageable host memory has read the host table when cudaMemcpyAsync returns)
  return cudaGetLastError() == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA;
}

int repack(const mfsdp_param_desc* params, int64_t n, const mfsdp_segment* segs, int32_t W,
           int32_t eb, const void* canonical_src, void* canonical_dst,
           const void* const* shards_src, void* const* shards_dst, void* ws, size_t ws_bytes,
           void* stream) {
  if (n < 0 || W <= 0 || (eb != 1 && eb != 2 && eb != 4 && eb != 8)) return MFSDP_EINVAL;
  if (n > 0 && (params == nullptr || segs == nullptr)) return MFSDP_EINVAL;
  if (n == 0) return MFSDP_OK;
  if (ws == nullptr) return MFSDP_EWORKSPACE;
  std::vector<int64_t> canon, shard;
  const int st = layout(params, n, segs, W, canon, shard);
  if (st != MFSDP_OK) return st;
  std::vector<CopyDesc> d;
  d.reserve((size_t)n);
  for (int64_t i = 0; i < n; ++i) {
    const int32_t r = segs[i].owner;
    const int64_t bytes = segs[i].numel * eb;
    if (canonical_src) {  // pack
      if (!shards_dst[r]) continue;
      d.push_back({static_cast<const uint8_t*>(canonical_src) + canon[(size_t)i] * eb,
                   static_cast<uint8_t*>(shards_dst[r]) + shard[(size_t)i] * eb, bytes, 0});
    } else {  // unpack
      if (!shards_src[r]) continue;
      d.push_back({static_cast<const uint8_t*>(shards_src[r]) + shard[(size_t)i] * eb,
                   static_cast<uint8_t*>(canonical_dst) + canon[(size_t)i] * eb, bytes, 0});
    }
  }
  return run_copies(d, eb, ws, ws_bytes, stream);
}

}  // namespace
}  // namespace mfsdp

using namespace mfsdp;

extern "C" int mfsdp_repack_workspace_bytes(int64_t n_params, size_t* bytes_out) {
  if (n_params < 0 || bytes_out == nullptr) return MFSDP_EINVAL;
  *bytes_out = desc_bytes(n_params);
  return MFSDP_OK;
}

extern "C" int mfsdp_pack_owner_shards(const mfsdp_param_desc* params, int64_t n_params,
                                       const mfsdp_segment* segs, int32_t world_size,
                                       int32_t elem_bytes, const void* canonical,
                                       void* const* shards, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  if (n_params > 0 && (canonical == nullptr || shards == nullptr)) return MFSDP_EINVAL;
  return repack(params, n_params, segs, world_size, elem_bytes, canonical, nullptr, nullptr,
                shards, workspace, workspace_bytes, stream);
}

extern "C" int mfsdp_unpack_owner_shards(const mfsdp_param_desc* params, int64_t n_params,
                                         const mfsdp_segment* segs, int32_t world_size,
                                         int32_t elem_bytes, const void* const* shards,
                                         void* canonical, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (n_params > 0 && (canonical == nullptr || shards == nullptr)) return MFSDP_EINVAL;
  return repack(params, n_params, segs, world_size, elem_bytes, nullptr, canonical, shards,
                nullptr, workspace, workspace_bytes, stream);
}
