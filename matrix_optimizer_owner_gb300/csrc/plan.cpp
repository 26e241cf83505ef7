// Owner planner: role construction, greedy owner assignment and segment layout (host only).
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":
//   §3   one role per data-parallel-sharded 2D matrix, one packed non-2D tail role per FSDP
//        unit, each whole on one owner;
//   §4.1 the planner sees every block; the greedy load is owner-resident numel; RoleGreedy
//        (the memory-conservative default) and ScopeGreedy (roles of all blocks pooled); each
//        block layout gives every parameter one contiguous local segment;
//   §4.2 O_{B,r}, the bytes of block B owned by rank r, drives the bandwidth model.
// The assignment listing itself is not printed on the pages; this follows the prose:
// blocks in order of first appearance; roles largest first with ties by first declaration
// index (pooled over all blocks for ScopeGreedy, ordered by block position next); each role
// to the rank with the least cumulative load, ties to the lowest rank.  In each (block, rank)
// owned roles are laid out by first declaration index, members in declaration order.
#include <algorithm>
#include <cstdint>
#include <limits>
#include <unordered_map>
#include <vector>

#include "mfsdp.h"

namespace {

struct RoleRec {
  int32_t id;
  int32_t block_pos;       // position of the block in first-appearance order
  int64_t first;           // first declaration index
  int64_t numel;
  std::vector<int64_t> members;
};

bool mul_overflows(int64_t a, int64_t b) {
  return a != 0 && b > std::numeric_limits<int64_t>::max() / a;
}

}  // namespace

extern "C" int mfsdp_plan_owner_set(const mfsdp_param_desc* params, int64_t n_params,
                                    int32_t world_size, int32_t policy, mfsdp_segment* seg_out,
                                    int64_t* block_rank_numel_out, int64_t* n_blocks_out) {
  if (n_params < 0 || world_size <= 0) return MFSDP_EINVAL;
  if (n_params > 0 && (params == nullptr || seg_out == nullptr)) return MFSDP_EINVAL;
  if (policy != MFSDP_POLICY_ROLE_GREEDY && policy != MFSDP_POLICY_SCOPE_GREEDY)
    return MFSDP_EINVAL;
  std::vector<int64_t> numel(n_params);
  for (int64_t i = 0; i < n_params; ++i) {
    const mfsdp_param_desc& p = params[i];
    if (p.rows < 0 || p.cols < 0 || mul_overflows(p.rows, p.cols)) return MFSDP_ESHAPE;
    numel[i] = p.rows * p.cols;
  }

  // Blocks in order of first appearance.
  std::unordered_map<int32_t, int32_t> block_pos;
  std::vector<int32_t> blocks;
  for (int64_t i = 0; i < n_params; ++i) {
    if (block_pos.emplace(params[i].block, (int32_t)blocks.size()).second)
      blocks.push_back(params[i].block);
  }
  const int32_t nb = (int32_t)blocks.size();

  // Roles: per block, one per matrix and one tail; ids by block, then first declaration index.
  std::vector<std::vector<int64_t>> by_block(nb);
  for (int64_t i = 0; i < n_params; ++i) by_block[block_pos[params[i].block]].push_back(i);
  std::vector<RoleRec> roles;
  std::vector<int32_t> role_of(n_params, -1);
  for (int32_t b = 0; b < nb; ++b) {
    std::vector<RoleRec> local;
    RoleRec tail{0, b, -1, 0, {}};
    for (int64_t i : by_block[b]) {
      if (params[i].is_matrix) {
        local.push_back(RoleRec{0, b, i, numel[i], {i}});
      } else {
        if (tail.first < 0) tail.first = i;
        tail.members.push_back(i);
        if (tail.numel > std::numeric_limits<int64_t>::max() - numel[i]) return MFSDP_ESHAPE;
        tail.numel += numel[i];
      }
    }
    if (tail.first >= 0) local.push_back(tail);
    std::sort(local.begin(), local.end(),
              [](const RoleRec& x, const RoleRec& y) { return x.first < y.first; });
    for (RoleRec& r : local) {
      r.id = (int32_t)roles.size();
      for (int64_t i : r.members) role_of[i] = r.id;
      roles.push_back(std::move(r));
    }
  }

  // Greedy assignment.
  std::vector<int64_t> load(world_size, 0);
  std::vector<int32_t> owner(roles.size(), 0);
  auto assign = [&](const RoleRec& r) {
    int32_t best = 0;
    for (int32_t k = 1; k < world_size; ++k)
      if (load[k] < load[best]) best = k;
    owner[r.id] = best;
    load[best] += r.numel;
  };
  auto larger_first = [](const RoleRec* x, const RoleRec* y) {
    if (x->numel != y->numel) return x->numel > y->numel;
    if (x->block_pos != y->block_pos) return x->block_pos < y->block_pos;
    return x->first < y->first;
  };
  if (policy == MFSDP_POLICY_ROLE_GREEDY) {
    size_t k = 0;
    for (int32_t b = 0; b < nb; ++b) {
      std::vector<const RoleRec*> rb;
      while (k < roles.size() && roles[k].block_pos == b) rb.push_back(&roles[k++]);
      std::stable_sort(rb.begin(), rb.end(), larger_first);
      for (const RoleRec* r : rb) assign(*r);
    }
  } else {
    std::vector<const RoleRec*> all;
    for (const RoleRec& r : roles) all.push_back(&r);
    std::stable_sort(all.begin(), all.end(), larger_first);
    for (const RoleRec* r : all) assign(*r);
  }

  // Layout: per (block, rank) by first declaration index; per rank flat matrix / tail buffers.
  std::vector<int64_t> mat_off(world_size, 0), tail_off(world_size, 0);
  if (block_rank_numel_out) {
    for (int64_t k = 0; k < (int64_t)nb * world_size; ++k) block_rank_numel_out[k] = 0;
  }
  for (int32_t b = 0; b < nb; ++b) {
    std::vector<int64_t> local(world_size, 0);
    for (const RoleRec& r : roles) {
      if (r.block_pos != b) continue;
      const int32_t o = owner[r.id];
      for (int64_t i : r.members) {
        mfsdp_segment& s = seg_out[i];
        s.owner = o;
        s.role = r.id;
        s.local_offset = local[o];
        s.numel = numel[i];
        if (params[i].is_matrix) {
          s.rank_offset = mat_off[o];
          mat_off[o] += numel[i];
        } else {
          s.rank_offset = tail_off[o];
          tail_off[o] += numel[i];
        }
        local[o] += numel[i];
      }
    }
    if (block_rank_numel_out) {
      for (int32_t r = 0; r < world_size; ++r)
        block_rank_numel_out[(int64_t)b * world_size + r] = local[r];
    }
  }
  // Contiguity check (§4.1): every role's members are adjacent in the owner's block shard.
  for (const RoleRec& r : roles) {
    for (size_t k = 1; k < r.members.size(); ++k) {
      const mfsdp_segment& a = seg_out[r.members[k - 1]];
      const mfsdp_segment& c = seg_out[r.members[k]];
      if (c.local_offset != a.local_offset + a.numel) return MFSDP_ENOTCONTIG;
    }
  }
  if (n_blocks_out) *n_blocks_out = nb;
  return MFSDP_OK;
}
