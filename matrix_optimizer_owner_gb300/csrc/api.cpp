// C ABI of libmfsdp: argument validation, the owned-matrix set (launch tables, workspace
// layout, TMA tensor maps) and the launch sequence of each step call.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "mfsdp.h"
#include "mfsdp_internal.h"

using namespace mfsdp;

namespace {

constexpr int kSlotU = 0, kSlotP = 1, kSlotO = 2, kSlotA = 3, kSlotB = 4, kSlots = 5;
// Per slot and half (hi, lo): [2D 64x64 box, 2D 64x128 box, 3D 64x64x2 box, 2D 32x32 box].
// 64x64 boxes and the 3D view serve MN-major operands (the 3D view, 64 elements x rows x
// 64-element chunks with a 128-byte chunk stride, loads a 128-wide half-tile in one operation;
// it exists only when the row length is a multiple of 64, so it never reaches past a row);
// 64x128 boxes load a 128-row K-major half-tile; unswizzled 32x32 boxes carry the epilogue's
// TMA stores (a warp's 32 rows x 32 columns).
constexpr int kMapsPerMatrix = 2 * kMapsPerHalf * kSlots;
constexpr int kGroupRows = 8;               // tile-row group of the rasterised tile order

// Problem-array variants: which X buffer a phase reads and writes.
enum Variant { kP1U, kP1O, kP1P, kP2, kP3UO, kP3UP, kP3OP, kP3PO, kVariants };

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct MatInfo {
  int64_t rows, cols, offset, numel, m, n;
  bool tr;        // rows > cols: Newton–Schulz runs on X = U^T, kept in U's own layout
  bool split;     // hi + lo operands
  bool aligned;   // offset % 8 == 0 and cols % 8 == 0: TMA reads/writes the caller buffers
  int64_t ldx;    // pitch of the workspace X buffers (= cols when aligned)
  int64_t ldm;    // pitch of the m x m buffers
  int32_t cta_begin;
  size_t ws[kSlots][2];  // workspace offsets of slot buffers (0 = not in the workspace)
};

}  // namespace

struct mfsdp_owner_set_s {
  std::vector<MatInfo> mats;
  int64_t split_max = 0;
  int32_t total_ctas = 0;
  int32_t n_split = 0;
  bool any_unaligned = false;
  bool offsets_aligned = true;      // every matrix offset is a multiple of 8 elements
  std::vector<NsTile> tiles[3][2];  // [phase][split]
  size_t off_devmats = 0, off_partials = 0, off_maps = 0, off_probs = 0, off_tiles = 0;
  size_t tile_off[3][2] = {};
  size_t ws_total = 0;
  // binding
  bool bound = false;
  int device = -1;
  int num_sms = 0;
  int pair_clusters = 0;            // co-resident CTA pairs of the pair kernel
  int* status = nullptr;
  char* ws = nullptr;
  const void* ns_input = nullptr;
  const void* ns_input_lo = nullptr;
  void* ortho = nullptr;
  void* ortho_lo = nullptr;
};

namespace mfsdp {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2D bf16 tensor map over a rows x cols row-major buffer of pitch ld elements: 64 x box_rows boxes,
// 128-byte swizzle, zero fill outside the tensor.
// 3D view of the same buffer for MN-major loads: (64 within a chunk, rows, cols / 64 chunks).
bool encode_map3d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * 2), 128};
  cuuint32_t box[3] = {64, 64, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 tensor map over a row-major rows x cols buffer of pitch ld elements: boxes of 32
// columns (128 bytes) x box_rows rows with a 128-byte swizzle, zero fill outside the tensor
// (the 3xTF32 GEMM's K-major operand tiles).
bool encode_map_f32(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
  cuuint32_t box[2] = {32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D bf16 tensor map over a row-major rows x cols buffer of pitch ld; boxes of box_rows x
// box_cols with a 128-byte swizzle (operand loads) or a 64-byte swizzle (the epilogue's
// 32 x 32 staging blocks).
bool encode_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld,
                uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output tiles of one problem in a rasterised order: groups of kGroupRows tile-rows, each group
// walked column by column, so the CTAs running at the same time share operand panels in L2.
void add_tiles(std::vector<NsTile>& out, int32_t prob, int64_t M, int64_t N, bool sym,
               int64_t bm) {
  const int64_t tm_n = (M + bm - 1) / bm, tn_n = (N + kBN - 1) / kBN;
  for (int64_t g0 = 0; g0 < tm_n; g0 += kGroupRows) {
    const int64_t g1 = std::min(tm_n, g0 + kGroupRows);
    for (int64_t tn = 0; tn < tn_n; ++tn)
      for (int64_t tm = g0; tm < g1; ++tm) {
        if (sym && tm * bm >= (tn + 1) * kBN) continue;  // entirely below the diagonal
        out.push_back(NsTile{prob, (int32_t)tm, (int32_t)tn, 0});
      }
  }
}

}  // namespace mfsdp

namespace {

int check_device(const mfsdp_owner_set* set) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFSDP_ENODEVICE;
  if (set && dev != set->device) return MFSDP_EINVAL;
  return MFSDP_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MFSDP_OK : MFSDP_ECUDA; }

}  // namespace

uint64_t mfsdp::wait_limit_ns() { return g_wait_limit_ns.load(); }

extern "C" {

int mfsdp_version(void) { return 100; }

const char* mfsdp_status_string(int st) {
  switch (st) {
    case MFSDP_OK: return "ok";
    case MFSDP_EINVAL: return "invalid argument";
    case MFSDP_ESHAPE: return "invalid shape";
    case MFSDP_EALIGN: return "misaligned pointer";
    case MFSDP_ENOTCONTIG: return "non-contiguous local segment";
    case MFSDP_EWORKSPACE: return "workspace too small";
    case MFSDP_ECUDA: return "CUDA error";
    case MFSDP_ETIMEOUT: return "device wait timed out";
    case MFSDP_ENONFINITE: return "non-finite norm or update";
    case MFSDP_ENODEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

int mfsdp_set_wait_limit_ns(uint64_t limit_ns) {
  g_wait_limit_ns.store(limit_ns ? limit_ns : 2000000000ull);
  return MFSDP_OK;
}

int mfsdp_owner_set_create(const mfsdp_matrix* mats, int32_t n_mats, int64_t split_max_numel,
                           mfsdp_owner_set** out) {
  if (!out || n_mats < 0 || (n_mats > 0 && !mats)) return MFSDP_EINVAL;
  *out = nullptr;
  mfsdp_owner_set* s = new (std::nothrow) mfsdp_owner_set_s();
  if (!s) return MFSDP_EINVAL;
  s->split_max = split_max_numel;
  s->mats.resize(n_mats);
  int64_t ctas = 0;
  for (int32_t i = 0; i < n_mats; ++i) {
    const mfsdp_matrix& q = mats[i];
    MatInfo& mi = s->mats[i];
    if (q.rows < 0 || q.cols < 0 || q.offset < 0 || q.rows >= (1ll << 31) ||
        q.cols >= (1ll << 31)) {
      delete s;
      return MFSDP_ESHAPE;
    }
    mi.rows = q.rows;
    mi.cols = q.cols;
    mi.offset = q.offset;
    mi.numel = q.rows * q.cols;
    mi.m = std::min(q.rows, q.cols);
    mi.n = std::max(q.rows, q.cols);
    mi.tr = q.rows > q.cols;
    mi.split = mi.numel > 0 && mi.numel <= split_max_numel;
    mi.aligned = (q.offset % 8 == 0) && (q.cols % 8 == 0);
    mi.ldx = round_up(std::max<int64_t>(q.cols, 1), 8);
    mi.ldm = round_up(std::max<int64_t>(mi.m, 1), 8);
    mi.cta_begin = (int32_t)ctas;
    ctas += (mi.numel + kChunk - 1) / kChunk;
    if (ctas >= (1ll << 31)) {
      delete s;
      return MFSDP_ESHAPE;
    }
    s->n_split += mi.split;
    if (mi.numel > 0 && !mi.aligned) s->any_unaligned = true;
    if (mi.numel > 0 && q.offset % 8 != 0) s->offsets_aligned = false;
  }
  s->total_ctas = (int32_t)ctas;
  // Ranges must not overlap.
  std::vector<std::pair<int64_t, int64_t>> r;
  for (const MatInfo& m : s->mats)
    if (m.numel > 0) r.emplace_back(m.offset, m.offset + m.numel);
  std::sort(r.begin(), r.end());
  for (size_t k = 1; k < r.size(); ++k)
    if (r[k].first < r[k - 1].second) {
      delete s;
      return MFSDP_ESHAPE;
    }

  // Tile lists, matrices ordered by contraction length (longest first) within each phase.
  std::vector<int32_t> order(n_mats);
  for (int32_t i = 0; i < n_mats; ++i) order[i] = i;
  for (int ph = 0; ph < 3; ++ph) {
    std::vector<int32_t> o = order;
    std::stable_sort(o.begin(), o.end(), [&](int32_t x, int32_t y) {
      const int64_t kx = ph == 0 ? s->mats[x].n : s->mats[x].m;
      const int64_t ky = ph == 0 ? s->mats[y].n : s->mats[y].m;
      return kx > ky;
    });
    for (int32_t i : o) {
      const MatInfo& m = s->mats[i];
      if (m.numel == 0) continue;
      // bf16 matrices run on CTA pairs (256-row tiles), split ones on single CTAs (128 rows)
      auto& dst = s->tiles[ph][m.split ? 1 : 0];
      const int64_t bm = m.split ? kBM : kPairBM;
      if (ph < 2)
        add_tiles(dst, i, m.m, m.m, true, bm);
      else
        add_tiles(dst, i, m.tr ? m.n : m.m, m.tr ? m.m : m.n, false, bm);
    }
  }

  // Workspace layout.
  size_t off = 0;
  auto take = [&](size_t bytes, size_t align) {
    off = (off + align - 1) / align * align;
    const size_t at = off;
    off += bytes;
    return at;
  };
  s->off_devmats = take(sizeof(DevMat) * std::max(n_mats, 1), 256);
  s->off_partials = take(sizeof(float) * std::max<int64_t>(ctas, 1), 256);
  s->off_maps = take(sizeof(CUtensorMap) * kMapsPerMatrix * std::max(n_mats, 1), 1024);
  s->off_probs = take(sizeof(NsProblem) * kVariants * std::max(n_mats, 1), 256);
  size_t ntiles = 0;
  for (int ph = 0; ph < 3; ++ph)
    for (int p = 0; p < 2; ++p) {
      s->tile_off[ph][p] = ntiles;
      ntiles += s->tiles[ph][p].size();
    }
  s->off_tiles = take(sizeof(NsTile) * std::max<size_t>(ntiles, 1), 256);
  for (MatInfo& m : s->mats) {
    std::memset(m.ws, 0, sizeof(m.ws));
    if (m.numel == 0) continue;
    const int halves = m.split ? 2 : 1;
    const size_t xb = (size_t)m.rows * m.ldx * 2, mb = (size_t)m.m * m.ldm * 2;
    for (int h = 0; h < halves; ++h) {
      m.ws[kSlotP][h] = take(xb, 256);
      if (!m.aligned) {
        m.ws[kSlotU][h] = take(xb, 256);
        m.ws[kSlotO][h] = take(xb, 256);
      }
      m.ws[kSlotA][h] = take(mb, 256);
      m.ws[kSlotB][h] = take(mb, 256);
    }
  }
  s->ws_total = (off + 255) / 256 * 256;
  *out = s;
  return MFSDP_OK;
}

int mfsdp_owner_set_destroy(mfsdp_owner_set* set) {
  delete set;
  return MFSDP_OK;
}

int mfsdp_owner_set_workspace_bytes(const mfsdp_owner_set* set, size_t* bytes_out) {
  if (!set || !bytes_out) return MFSDP_EINVAL;
  *bytes_out = set->ws_total;
  return MFSDP_OK;
}

int mfsdp_owner_set_split_count(const mfsdp_owner_set* set, int32_t* count_out) {
  if (!set || !count_out) return MFSDP_EINVAL;
  *count_out = set->n_split;
  return MFSDP_OK;
}

int mfsdp_owner_set_bind(mfsdp_owner_set* set, void* workspace, size_t workspace_bytes,
                         const void* ns_input, const void* ns_input_lo, void* ortho_out,
                         void* ortho_lo, void* stream) {
  if (!set || !workspace || !ns_input || !ortho_out) return MFSDP_EINVAL;
  if (set->n_split > 0 && (!ns_input_lo || !ortho_lo)) return MFSDP_EINVAL;
  if (ns_input == ortho_out) return MFSDP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MFSDP_EALIGN;
  if (!aligned16(ns_input) || !aligned16(ortho_out) || (ns_input_lo && !aligned16(ns_input_lo)) ||
      (ortho_lo && !aligned16(ortho_lo)))
    return MFSDP_EALIGN;
  if (workspace_bytes < set->ws_total) return MFSDP_EWORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFSDP_ENODEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MFSDP_ENODEVICE;
  if (prop.major != 10 || prop.minor != 3) return MFSDP_ENODEVICE;
  if (!encode_fn()) return MFSDP_ECUDA;
  if (ns_prepare_kernels() != cudaSuccess) return MFSDP_ECUDA;
  const int pair_clusters = ns_pair_max_clusters(prop.multiProcessorCount);
  if (pair_clusters < 1) return MFSDP_ECUDA;
  int* status = status_word_address();
  if (!status) return MFSDP_ECUDA;

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const int32_t n = (int32_t)set->mats.size();

  // Streaming-kernel matrix table.
  std::vector<DevMat> dm(std::max(n, 1));
  for (int32_t i = 0; i < n; ++i) {
    const MatInfo& m = set->mats[i];
    dm[i].offset = m.offset;
    dm[i].numel = m.numel;
    dm[i].rows = m.rows;
    dm[i].cols = m.cols;
    dm[i].cta_begin = m.cta_begin;
    dm[i].split = m.split;
    dm[i].scale_original =
        m.cols > 0 ? (float)std::sqrt(std::max(1.0, (double)m.rows / (double)m.cols)) : 1.f;
    dm[i].scale_rms = (float)(0.2 * std::sqrt((double)std::max(m.rows, m.cols)));
  }

  // Buffers of each slot.
  auto slot_ptr = [&](const MatInfo& m, int slot, int h) -> uint16_t* {
    if (m.ws[slot][h] || slot == kSlotP || slot == kSlotA || slot == kSlotB)
      return reinterpret_cast<uint16_t*>(ws + m.ws[slot][h]);
    const void* b = slot == kSlotU ? (h ? ns_input_lo : ns_input) : (h ? ortho_lo : ortho_out);
    return const_cast<uint16_t*>(static_cast<const uint16_t*>(b)) + m.offset;
  };
  auto slot_ld = [&](const MatInfo& m, int slot) -> int64_t {
    if (slot == kSlotA || slot == kSlotB) return m.ldm;
    if (slot == kSlotP || !m.aligned) return m.ldx;
    return m.cols;
  };

  // Whether a slot buffer has the 3D MN-major view (its row length is a multiple of 64).
  auto view3d = [&](const MatInfo& m, int slot) -> bool {
    return ((slot == kSlotA || slot == kSlotB) ? m.m : m.cols) % 64 == 0;
  };

  // Tensor maps.
  std::vector<CUtensorMap> maps((size_t)kMapsPerMatrix * std::max(n, 1));
  std::memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
  for (int32_t i = 0; i < n; ++i) {
    const MatInfo& m = set->mats[i];
    if (m.numel == 0) continue;
    for (int slot = 0; slot < kSlots; ++slot)
      for (int h = 0; h < (m.split ? 2 : 1); ++h) {
        const bool sq = slot == kSlotA || slot == kSlotB;
        const int64_t rows = sq ? m.m : m.rows, cols = sq ? m.m : m.cols;
        CUtensorMap* mp = &maps[(size_t)i * kMapsPerMatrix + 2 * kMapsPerHalf * slot + kMapsPerHalf * h];
        if (!encode_map(mp, slot_ptr(m, slot, h), rows, cols, slot_ld(m, slot), 64u) ||
            !encode_map(mp + 1, slot_ptr(m, slot, h), rows, cols, slot_ld(m, slot), 128u) ||
            !encode_map(mp + 3, slot_ptr(m, slot, h), rows, cols, slot_ld(m, slot), 32u, 32u,
                        false))
          return MFSDP_ECUDA;
        if (cols % 64 == 0 && !encode_map3d(mp + 2, slot_ptr(m, slot, h), rows, cols,
                                            slot_ld(m, slot)))
          return MFSDP_ECUDA;
      }
  }

  // Problem variants.
  std::vector<NsProblem> probs((size_t)kVariants * std::max(n, 1));
  std::memset(probs.data(), 0, probs.size() * sizeof(NsProblem));
  for (int32_t i = 0; i < n; ++i) {
    const MatInfo& m = set->mats[i];
    if (m.numel == 0) continue;
    const int mb = i * kMapsPerMatrix;
    auto gram = [&](int src, int first) {
      NsProblem p{};
      p.M = p.N = (int32_t)m.m;
      p.K = (int32_t)m.n;
      p.a_mn = p.b_mn = m.tr ? 1 : 0;
      p.sym = 1;
      p.kind = kGram;
      p.first = first;
      p.mat = i;
      p.map_a = p.map_b = mb + 2 * kMapsPerHalf * src;
      p.mn3d = m.tr && view3d(m, src) ? 3 : 0;
      p.o_hi = slot_ptr(m, kSlotA, 0);
      p.o_lo = m.split ? slot_ptr(m, kSlotA, 1) : nullptr;
      p.ldo = m.ldm;
      p.map_o = mb + 2 * kMapsPerHalf * kSlotA + 3;  // 32x32 store box (64-byte swizzle)
      return p;
    };
    auto apply = [&](int src, int dst, int first) {
      NsProblem p{};
      if (!m.tr) {  // X' = B' X (or a X + B X): B' rows (K-major) times X (MN-major)
        p.M = (int32_t)m.m;
        p.N = (int32_t)m.n;
        p.a_mn = 0;
        p.b_mn = 1;
        p.map_a = mb + 2 * kMapsPerHalf * kSlotB;
        p.map_b = mb + 2 * kMapsPerHalf * src;
        p.mn3d = view3d(m, src) ? 2 : 0;
      } else {      // Y' = Y B' (or a Y + Y B), Y = X^T in the caller's layout: both K-major
        p.M = (int32_t)m.n;
        p.N = (int32_t)m.m;
        p.a_mn = 0;
        p.b_mn = 0;
        p.map_a = mb + 2 * kMapsPerHalf * src;
        p.map_b = mb + 2 * kMapsPerHalf * kSlotB;
      }
      p.K = (int32_t)m.m;
      p.kind = kApply;
      p.first = first;
      p.mat = i;
      p.fold_a = m.split ? 0 : 1;  // bf16 operands: a X is folded into B' = a I + B
      if (m.split) {               // split operands: X' = a X + B X, X as the addend
        p.d_hi = slot_ptr(m, src, 0);
        p.d_lo = slot_ptr(m, src, 1);
        p.ldd = slot_ld(m, src);
      }
      p.o_hi = slot_ptr(m, dst, 0);
      p.o_lo = m.split ? slot_ptr(m, dst, 1) : nullptr;
      p.ldo = slot_ld(m, dst);
      p.map_o = mb + 2 * kMapsPerHalf * dst + 3;  // 32x32 store box (64-byte swizzle)
      return p;
    };
    NsProblem poly{};
    poly.M = poly.N = poly.K = (int32_t)m.m;
    poly.sym = 1;
    poly.kind = kPoly;
    poly.fold_a = m.split ? 0 : 1;
    poly.mat = i;
    poly.map_a = poly.map_b = mb + 2 * kMapsPerHalf * kSlotA;
    poly.d_hi = slot_ptr(m, kSlotA, 0);
    poly.d_lo = m.split ? slot_ptr(m, kSlotA, 1) : nullptr;
    poly.ldd = m.ldm;
    poly.map_o = mb + 2 * kMapsPerHalf * kSlotB + 3;  // 32x32 store box (64-byte swizzle)
    poly.o_hi = slot_ptr(m, kSlotB, 0);
    poly.o_lo = m.split ? slot_ptr(m, kSlotB, 1) : nullptr;
    poly.ldo = m.ldm;
    probs[(size_t)kP1U * n + i] = gram(kSlotU, 1);
    probs[(size_t)kP1O * n + i] = gram(kSlotO, 0);
    probs[(size_t)kP1P * n + i] = gram(kSlotP, 0);
    probs[(size_t)kP2 * n + i] = poly;
    probs[(size_t)kP3UO * n + i] = apply(kSlotU, kSlotO, 1);
    probs[(size_t)kP3UP * n + i] = apply(kSlotU, kSlotP, 1);
    probs[(size_t)kP3OP * n + i] = apply(kSlotO, kSlotP, 0);
    probs[(size_t)kP3PO * n + i] = apply(kSlotP, kSlotO, 0);
  }

  std::vector<NsTile> tiles;
  for (int ph = 0; ph < 3; ++ph)
    for (int p = 0; p < 2; ++p) tiles.insert(tiles.end(), set->tiles[ph][p].begin(), set->tiles[ph][p].end());

  cudaError_t e = cudaSuccess;
  auto put = [&](size_t off, const void* src, size_t bytes) {
    if (e == cudaSuccess && bytes) e = cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, st);
  };
  put(set->off_devmats, dm.data(), sizeof(DevMat) * n);
  put(set->off_maps, maps.data(), sizeof(CUtensorMap) * maps.size());
  put(set->off_probs, probs.data(), sizeof(NsProblem) * probs.size());
  put(set->off_tiles, tiles.data(), sizeof(NsTile) * tiles.size());
  if (e != cudaSuccess) return MFSDP_ECUDA;

  set->bound = true;
  set->device = dev;
  set->num_sms = prop.multiProcessorCount;
  set->pair_clusters = pair_clusters;
  set->status = status;
  set->ws = ws;
  set->ns_input = ns_input;
  set->ns_input_lo = ns_input_lo;
  set->ortho = ortho_out;
  set->ortho_lo = ortho_lo;
  return MFSDP_OK;
}

int mfsdp_owner_reduce_momentum(const mfsdp_owner_set* set, const void* const* contrib, int32_t W,
                                int32_t contrib_dtype, float grad_scale, float momentum,
                                int32_t nesterov, float* momentum_buf, void* ns_input,
                                void* ns_input_lo, float* reduced_grad_out, float* norm_out,
                                void* stream) {
  if (!set || !set->bound || !contrib || W < 1 || W > kMaxContrib) return MFSDP_EINVAL;
  if (contrib_dtype != MFSDP_DTYPE_F32 && contrib_dtype != MFSDP_DTYPE_BF16) return MFSDP_EINVAL;
  if (!momentum_buf || !norm_out || ns_input != set->ns_input) return MFSDP_EINVAL;
  if (set->n_split > 0 && ns_input_lo != set->ns_input_lo) return MFSDP_EINVAL;
  for (int32_t w = 0; w < W; ++w) {
    if (!contrib[w]) return MFSDP_EINVAL;
    if (!aligned16(contrib[w])) return MFSDP_EALIGN;
  }
  if (!aligned16(momentum_buf) || !aligned16(norm_out) ||
      (reduced_grad_out && !aligned16(reduced_grad_out)))
    return MFSDP_EALIGN;
  const int dst = check_device(set);
  if (dst != MFSDP_OK) return dst;
  if (set->mats.empty()) return MFSDP_OK;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  ReduceParams p{};
  for (int32_t w = 0; w < W; ++w) p.contrib.p[w] = contrib[w];
  p.W = W;
  p.n_mats = (int32_t)set->mats.size();
  p.total_ctas = set->total_ctas;
  p.nesterov = nesterov ? 1 : 0;
  p.offsets_aligned = set->offsets_aligned ? 1 : 0;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = set->status;
  p.mats = reinterpret_cast<const DevMat*>(set->ws + set->off_devmats);
  p.grad_scale = grad_scale;
  p.mu = momentum;
  p.one_minus_mu = (float)(1.0 - (double)momentum);
  p.momentum = momentum_buf;
  p.uhat = static_cast<uint16_t*>(ns_input);
  p.uhat_lo = static_cast<uint16_t*>(ns_input_lo);
  p.grad = reduced_grad_out;
  p.partials = reinterpret_cast<float*>(set->ws + set->off_partials);
  cudaError_t e = launch_reduce_momentum(p, contrib_dtype, st);
  if (e != cudaSuccess) return MFSDP_ECUDA;
  NormParams q{};
  q.mats = p.mats;
  q.n_mats = p.n_mats;
  q.partials = p.partials;
  q.norm = norm_out;
  q.status = set->status;
  return cuda_status(launch_norm_finalize(q, st));
}

int mfsdp_newton_schulz(const mfsdp_owner_set* set, const void* ns_input, const void* ns_input_lo,
                        const float* norm, int32_t steps, float a, float b, float c, float eps,
                        void* ortho_out, void* ortho_lo, void* stream) {
  if (!set || !set->bound || !norm || steps < 1 || steps > 64) return MFSDP_EINVAL;
  if (ns_input != set->ns_input || ortho_out != set->ortho) return MFSDP_EINVAL;
  if (set->n_split > 0 && (ns_input_lo != set->ns_input_lo || ortho_lo != set->ortho_lo))
    return MFSDP_EINVAL;
  if (!aligned16(norm)) return MFSDP_EALIGN;
  const int dst = check_device(set);
  if (dst != MFSDP_OK) return dst;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int32_t n = (int32_t)set->mats.size();
  if (n == 0) return MFSDP_OK;
  cudaError_t e = cudaSuccess;

  // Unaligned matrices: stage the input in a pitched workspace copy.
  if (set->any_unaligned) {
    for (const MatInfo& m : set->mats) {
      if (m.numel == 0 || m.aligned) continue;
      for (int h = 0; h < (m.split ? 2 : 1); ++h) {
        CopyParams cp{};
        cp.src = static_cast<const uint16_t*>(h ? ns_input_lo : ns_input) + m.offset;
        cp.dst = reinterpret_cast<uint16_t*>(set->ws + m.ws[kSlotU][h]);
        cp.rows = m.rows;
        cp.cols = m.cols;
        cp.ld_src = m.cols;
        cp.ld_dst = m.ldx;
        if (e == cudaSuccess) e = launch_copy2d(cp, st);
      }
    }
  }

  const NsProblem* probs = reinterpret_cast<const NsProblem*>(set->ws + set->off_probs);
  const NsTile* tiles = reinterpret_cast<const NsTile*>(set->ws + set->off_tiles);
  NsLaunchParams lp{};
  lp.maps = reinterpret_cast<const CUtensorMap*>(set->ws + set->off_maps);
  lp.norm = norm;
  lp.eps = eps;
  lp.a = a;
  lp.b = b;
  lp.c = c;
  lp.wait_limit_ns = g_wait_limit_ns.load();
  lp.status = set->status;
  auto run = [&](int phase, int variant) {
    for (int p = 0; p < 2; ++p) {
      const size_t cnt = set->tiles[phase][p].size();
      if (cnt == 0 || e != cudaSuccess) continue;
      lp.probs = probs + (size_t)variant * n;
      lp.tiles = tiles + set->tile_off[phase][p];
      lp.ntiles = (int32_t)cnt;
      const int grid = p == 1 ? (int)std::min<size_t>(cnt, (size_t)set->num_sms)
                              : set->pair_clusters;
      e = launch_ns_phase(lp, p == 1, grid, st);
    }
  };
  // X_t lives in the output slot when steps - t is even, else in the workspace ping buffer,
  // so that X_steps lands in the output slot.
  for (int t = 1; t <= steps; ++t) {
    const bool src_u = t == 1;
    const bool src_o = !src_u && ((steps - (t - 1)) % 2 == 0);
    const bool dst_o = (steps - t) % 2 == 0;
    run(0, src_u ? kP1U : (src_o ? kP1O : kP1P));
    run(1, kP2);
    run(2, src_u ? (dst_o ? kP3UO : kP3UP) : (src_o ? kP3OP : kP3PO));
  }

  if (set->any_unaligned) {
    for (const MatInfo& m : set->mats) {
      if (m.numel == 0 || m.aligned) continue;
      for (int h = 0; h < (m.split ? 2 : 1); ++h) {
        CopyParams cp{};
        cp.src = reinterpret_cast<const uint16_t*>(set->ws + m.ws[kSlotO][h]);
        cp.dst = static_cast<uint16_t*>(h ? ortho_lo : ortho_out) + m.offset;
        cp.rows = m.rows;
        cp.cols = m.cols;
        cp.ld_src = m.ldx;
        cp.ld_dst = m.cols;
        if (e == cudaSuccess) e = launch_copy2d(cp, st);
      }
    }
  }
  return cuda_status(e);
}

int mfsdp_apply_update(const mfsdp_owner_set* set, float* weights, const void* ortho,
                       const void* ortho_lo, float lr, float weight_decay, int32_t lr_adjust,
                       void* stream) {
  if (!set || !set->bound || !weights || !ortho) return MFSDP_EINVAL;
  if (lr_adjust != MFSDP_LR_ORIGINAL && lr_adjust != MFSDP_LR_MATCH_RMS_ADAMW) return MFSDP_EINVAL;
  if (!aligned16(weights) || !aligned16(ortho) || (ortho_lo && !aligned16(ortho_lo)))
    return MFSDP_EALIGN;
  const int dst = check_device(set);
  if (dst != MFSDP_OK) return dst;
  if (set->mats.empty()) return MFSDP_OK;
  UpdateParams p{};
  p.mats = reinterpret_cast<const DevMat*>(set->ws + set->off_devmats);
  p.n_mats = (int32_t)set->mats.size();
  p.total_ctas = set->total_ctas;
  p.lr_adjust = lr_adjust;
  p.decay = (float)(1.0 - (double)lr * (double)weight_decay);
  p.lr = lr;
  p.weights = weights;
  p.ortho = static_cast<const uint16_t*>(ortho);
  p.ortho_lo = static_cast<const uint16_t*>(ortho_lo);
  return cuda_status(launch_apply_update(p, static_cast<cudaStream_t>(stream)));
}

int mfsdp_adamw_tail(const void* const* contrib, int32_t W, int32_t contrib_dtype,
                     float grad_scale, int64_t n, float* param, float* exp_avg,
                     float* exp_avg_sq, int64_t step, float lr, float beta1, float beta2,
                     float eps, float weight_decay, void* stream) {
  if (n < 0 || step < 1) return MFSDP_EINVAL;
  if (n == 0) return MFSDP_OK;
  if (!contrib || W < 1 || W > kMaxContrib || !param || !exp_avg || !exp_avg_sq)
    return MFSDP_EINVAL;
  if (contrib_dtype != MFSDP_DTYPE_F32 && contrib_dtype != MFSDP_DTYPE_BF16) return MFSDP_EINVAL;
  for (int32_t w = 0; w < W; ++w) {
    if (!contrib[w]) return MFSDP_EINVAL;
    if (!aligned16(contrib[w])) return MFSDP_EALIGN;
  }
  if (!aligned16(param) || !aligned16(exp_avg) || !aligned16(exp_avg_sq)) return MFSDP_EALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MFSDP_ENODEVICE;
  AdamParams p{};
  for (int32_t w = 0; w < W; ++w) p.contrib.p[w] = contrib[w];
  p.W = W;
  p.n = n;
  p.grad_scale = grad_scale;
  p.decay = (float)(1.0 - (double)lr * (double)weight_decay);
  p.b1 = beta1;
  p.one_minus_b1 = (float)(1.0 - (double)beta1);
  p.b2 = beta2;
  p.one_minus_b2 = (float)(1.0 - (double)beta2);
  const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
  const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
  p.step_size = (float)((double)lr / bc1);
  p.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
  p.eps = eps;
  p.p = param;
  p.m = exp_avg;
  p.v = exp_avg_sq;
  return cuda_status(launch_adamw(p, contrib_dtype, static_cast<cudaStream_t>(stream)));
}

int mfsdp_query_status(void* stream, int32_t* device_status_out) {
  if (!device_status_out) return MFSDP_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MFSDP_ECUDA;
  int* addr = status_word_address();
  if (!addr) return MFSDP_ECUDA;
  int v = 0;
  if (cudaMemcpy(&v, addr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MFSDP_ECUDA;
  if (cudaMemset(addr, 0, sizeof(int)) != cudaSuccess) return MFSDP_ECUDA;
  *device_status_out = (v & kStatusTimeout)        ? MFSDP_ETIMEOUT
                       : (v & kStatusTmemMismatch) ? MFSDP_ECUDA
                       : (v & kStatusNonFinite)    ? MFSDP_ENONFINITE
                                                   : MFSDP_OK;
  return MFSDP_OK;
}

int mfsdp_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  int* addr = status_word_address();
  if (!addr) return MFSDP_ECUDA;
  return cuda_status(
      launch_wait_timeout_selftest(limit_ns, addr, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
