// Owner planner: role construction, greedy owner assignment and segment layout (host only).
//
// "MatrixFSDP: communication-free matrix optimizers under ZeRO-3 parameter sharding":
//   §3   one role per data-parallel-sharded 2D matrix, one packed non-2D tail role per FSDP
//        unit, each whole on one owner;
//   §4.1 the planner sees every block; the greedy load is the numel resident on the owner; RoleGreedy
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

// ------------------------------------------------------------------------------------------
// Resource scorer and CostAware (§4.1), with the §4.2 quantities O_{B,r}, P_B and gamma_B.
// The pages name the estimates but give no formulas; the ones used here are stated with the
// declarations: one owner-segment collective's send + receive bytes, the gradient-reduce
// receive buffers as workspace, nominal Newton–Schulz FLOPs as optimizer compute.
// ------------------------------------------------------------------------------------------
namespace {

bool add_overflows(int64_t a, int64_t b) { return b > std::numeric_limits<int64_t>::max() - a; }

int score_impl(const mfsdp_param_desc* params, int64_t n_params, int32_t world_size,
               const mfsdp_segment* segs, const mfsdp_cost_model* model,
               mfsdp_rank_resources* ranks_out, double* gamma_out, int64_t* n_blocks_out) {
  if (n_params < 0 || world_size <= 0 || model == nullptr || ranks_out == nullptr)
    return MFSDP_EINVAL;
  if (n_params > 0 && (params == nullptr || segs == nullptr)) return MFSDP_EINVAL;
  if (model->param_bytes < 1 || model->grad_bytes < 1 || model->state_bytes < 1 ||
      model->ns_steps < 0)
    return MFSDP_EINVAL;
  const int64_t W = world_size;
  std::unordered_map<int32_t, int32_t> block_pos;
  std::vector<int64_t> pb;  // P_B
  std::vector<int32_t> pos(n_params);
  for (int64_t i = 0; i < n_params; ++i) {
    const mfsdp_param_desc& p = params[i];
    if (p.rows < 0 || p.cols < 0 || mul_overflows(p.rows, p.cols)) return MFSDP_ESHAPE;
    if (segs[i].numel != p.rows * p.cols) return MFSDP_ESHAPE;
    if (segs[i].owner < 0 || segs[i].owner >= world_size) return MFSDP_EINVAL;
    auto it = block_pos.emplace(p.block, (int32_t)pb.size());
    if (it.second) pb.push_back(0);
    pos[i] = it.first->second;
    if (add_overflows(pb[pos[i]], segs[i].numel)) return MFSDP_ESHAPE;
    pb[pos[i]] += segs[i].numel;
  }
  const int64_t nb = (int64_t)pb.size();
  std::vector<int64_t> o((size_t)(nb * W), 0);  // O_{B,r}
  std::vector<int64_t> mat(W, 0), tail(W, 0);
  std::vector<double> flops(W, 0.0);
  for (int64_t i = 0; i < n_params; ++i) {
    const int32_t r = segs[i].owner;
    const int64_t ne = segs[i].numel;
    o[(size_t)(pos[i] * W + r)] += ne;
    if (params[i].is_matrix) {
      mat[r] += ne;
      if (ne > 0) {
        const int64_t m = std::min(params[i].rows, params[i].cols);
        const int64_t n = std::max(params[i].rows, params[i].cols);
        flops[r] += (double)model->ns_steps *
                    (4.0 * (double)m * (double)m * (double)n + 2.0 * (double)(m * m * m));
      }
    } else {
      tail[r] += ne;
    }
  }
  const int64_t big = std::numeric_limits<int64_t>::max() / 4;
  for (int32_t r = 0; r < world_size; ++r) {
    const int64_t own = mat[r] + tail[r];
    int64_t comm = 0, ws = 0;
    for (int64_t b = 0; b < nb; ++b) {
      const int64_t obr = o[(size_t)(b * W + r)];
      if (obr > big / W) return MFSDP_ESHAPE;
      comm += (W - 1) * obr + (pb[b] - obr);
      if (comm > big) return MFSDP_ESHAPE;
      ws = std::max(ws, (W - 1) * obr);
    }
    if (own > big / 8 || comm > big / 8 || ws > big / 8) return MFSDP_ESHAPE;
    mfsdp_rank_resources& x = ranks_out[r];
    x.param_bytes = own * model->param_bytes;
    x.grad_bytes = own * model->grad_bytes;
    x.state_bytes = (mat[r] + 2 * tail[r]) * model->state_bytes;
    x.comm_bytes = comm * model->param_bytes;
    x.workspace_bytes = ws * model->grad_bytes;
    x.optimizer_flops = flops[r];
  }
  if (gamma_out) {
    for (int64_t b = 0; b < nb; ++b) {
      int64_t mx = 0;
      for (int32_t r = 0; r < world_size; ++r) mx = std::max(mx, o[(size_t)(b * W + r)]);
      gamma_out[b] = pb[b] > 0 ? (double)mx / ((double)pb[b] / (double)W) : 0.0;
    }
  }
  if (n_blocks_out) *n_blocks_out = nb;
  return MFSDP_OK;
}

int64_t max_workspace(const std::vector<mfsdp_rank_resources>& rs) {
  int64_t m = 0;
  for (const mfsdp_rank_resources& x : rs) m = std::max(m, x.workspace_bytes);
  return m;
}

}  // namespace

extern "C" int mfsdp_score_plan(const mfsdp_param_desc* params, int64_t n_params,
                                int32_t world_size, const mfsdp_segment* segs,
                                const mfsdp_cost_model* model, mfsdp_rank_resources* ranks_out,
                                double* gamma_out, int64_t* n_blocks_out) {
  return score_impl(params, n_params, world_size, segs, model, ranks_out, gamma_out,
                    n_blocks_out);
}

extern "C" int mfsdp_plan_cost_aware(const mfsdp_param_desc* params, int64_t n_params,
                                     int32_t world_size, const mfsdp_cost_model* model,
                                     int64_t workspace_cap_bytes, mfsdp_segment* seg_out,
                                     int32_t* policy_out) {
  if (n_params < 0 || world_size <= 0 || model == nullptr) return MFSDP_EINVAL;
  if (n_params > 0 && (params == nullptr || seg_out == nullptr)) return MFSDP_EINVAL;
  std::vector<mfsdp_segment> role((size_t)n_params), scope((size_t)n_params);
  int st = mfsdp_plan_owner_set(params, n_params, world_size, MFSDP_POLICY_ROLE_GREEDY,
                                role.data(), nullptr, nullptr);
  if (st != MFSDP_OK) return st;
  st = mfsdp_plan_owner_set(params, n_params, world_size, MFSDP_POLICY_SCOPE_GREEDY,
                            scope.data(), nullptr, nullptr);
  if (st != MFSDP_OK) return st;
  std::vector<mfsdp_rank_resources> rs_role(world_size), rs_scope(world_size);
  st = score_impl(params, n_params, world_size, role.data(), model, rs_role.data(), nullptr,
                  nullptr);
  if (st != MFSDP_OK) return st;
  st = score_impl(params, n_params, world_size, scope.data(), model, rs_scope.data(), nullptr,
                  nullptr);
  if (st != MFSDP_OK) return st;
  const int64_t cap = workspace_cap_bytes > 0 ? workspace_cap_bytes : max_workspace(rs_role);
  const bool take_scope = max_workspace(rs_scope) <= cap;
  const std::vector<mfsdp_segment>& pick = take_scope ? scope : role;
  std::copy(pick.begin(), pick.end(), seg_out);
  if (policy_out) *policy_out = take_scope ? MFSDP_POLICY_SCOPE_GREEDY : MFSDP_POLICY_ROLE_GREEDY;
  return MFSDP_OK;
}
