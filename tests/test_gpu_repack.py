"""Owner-segment repacking on the GPU against the oracle (bit-exact).

Pack (canonical axis -> owner shards), unpack (owner shards -> canonical axis) and reshard
(unpack under one plan, pack under another) of the workloads' parameter lists, for 2- and
4-byte elements, with segments at odd element offsets, with ranks skipped (NULL shard) and an
empty model.  Small cases compare every element with the oracle's numpy repacking; the
Llama-3-8B parameter list (7.0e9 elements) compares every parameter's slice on the device at
the offsets the oracle computes.
"""

import numpy as np
import pytest
import torch

from oracle import plan as oplan
from oracle import repack as orepack
from workloads import get_config

pytestmark = pytest.mark.gpu


def _params(spec):
    return [(p.rows, p.cols, p.block, p.is_matrix) for p in spec]


def _oparams(params):
    return [oplan.Param(r, c, b, m) for r, c, b, m in params]


def _segs(params, W, policy):
    from matrix_optimizer_owner_gb300 import mfsdp
    segs, _, _ = mfsdp.mfsdp_plan_owner_set(params, W, policy)
    return segs


def _osegs(segs):
    return [oplan.Segment(s["owner"], s["role"], s["local_offset"], s["rank_offset"], s["numel"])
            for s in segs]


def _ws(n):
    from matrix_optimizer_owner_gb300 import mfsdp
    return torch.empty(mfsdp.mfsdp_repack_workspace_bytes(n), dtype=torch.uint8, device="cuda")


def _random(n, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    bits = torch.randint(-(1 << 15), 1 << 15, (n * (2 if dtype == torch.int32 else 1),),
                         generator=g, device="cuda", dtype=torch.int16)
    return bits.view(dtype) if dtype == torch.int32 else bits


def _odd_params(seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(40):
        m = bool(rng.random() < 0.7)
        out.append((int(rng.integers(1, 97)), int(rng.integers(1, 61)) if m else 1,
                    int(rng.integers(0, 6)), m))
    return out


SMALL = [("tiny", _params(get_config(0).params)), ("gpt2", _params(get_config(1).params)),
         ("odd", _odd_params(5))]


@pytest.mark.parametrize("name,params", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("dtype", [torch.int16, torch.int32])
def test_pack_unpack_reshard_match_oracle(name, params, dtype):
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    ps = _oparams(params)
    total = sum(p.numel for p in ps)
    canon = _random(total, dtype, 7)
    canon_h = canon.cpu().numpy()
    ws = _ws(len(params))
    for W, pol in ((8, 0), (3, 1), (1, 0)):
        segs = _segs(params, W, pol)
        _, size = orepack.shard_offsets(ps, _osegs(segs), W)
        shards = [torch.full((max(n, 1),), 0x5A5A, dtype=torch.int32, device="cuda")
                  .view(dtype)[:n].clone() for n in size]
        mfsdp.mfsdp_pack_owner_shards(params, segs, W, canon, shards, ws)
        ref = orepack.pack(ps, _osegs(segs), W, canon_h)
        for got, want in zip(shards, ref):
            np.testing.assert_array_equal(got.cpu().numpy(), want)
        back = torch.zeros_like(canon)
        mfsdp.mfsdp_unpack_owner_shards(params, segs, W, shards, back, ws)
        np.testing.assert_array_equal(back.cpu().numpy(), canon_h)
    # reshard 8 ranks RoleGreedy -> 3 ranks ScopeGreedy through the canonical axis
    a, b = _segs(params, 8, 0), _segs(params, 3, 1)
    _, size_a = orepack.shard_offsets(ps, _osegs(a), 8)
    _, size_b = orepack.shard_offsets(ps, _osegs(b), 3)
    src = [torch.zeros(n, dtype=dtype, device="cuda") for n in size_a]
    mfsdp.mfsdp_pack_owner_shards(params, a, 8, canon, src, ws)
    mid = torch.zeros_like(canon)
    mfsdp.mfsdp_unpack_owner_shards(params, a, 8, src, mid, ws)
    dst = [torch.zeros(n, dtype=dtype, device="cuda") for n in size_b]
    mfsdp.mfsdp_pack_owner_shards(params, b, 3, mid, dst, ws)
    want = orepack.reshard(ps, _osegs(a), 8, [s.cpu().numpy() for s in src], _osegs(b), 3)
    for got, w in zip(dst, want):
        np.testing.assert_array_equal(got.cpu().numpy(), w)
    assert mfsdp.mfsdp_query_status() == 0


def test_null_shards_are_skipped_and_empty_model():
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    params = _odd_params(9)
    ps = _oparams(params)
    total = sum(p.numel for p in ps)
    canon = _random(total, torch.int16, 3)
    segs = _segs(params, 4, 0)
    _, size = orepack.shard_offsets(ps, _osegs(segs), 4)
    ws = _ws(len(params))
    only = [None, torch.full((size[1],), 77, dtype=torch.int16, device="cuda"), None, None]
    mfsdp.mfsdp_pack_owner_shards(params, segs, 4, canon, only, ws)
    want = orepack.pack(ps, _osegs(segs), 4, canon.cpu().numpy())
    np.testing.assert_array_equal(only[1].cpu().numpy(), want[1])
    # unpack of rank 1 alone writes rank 1's parameters and nothing else
    back = torch.full_like(canon, -1)
    mfsdp.mfsdp_unpack_owner_shards(params, segs, 4, only, back, ws)
    coff = orepack.canonical_offsets(ps)
    expect = np.full(total, -1, dtype=np.int16)
    ch = canon.cpu().numpy()
    for i, s in enumerate(segs):
        if s["owner"] == 1:
            expect[coff[i]:coff[i] + s["numel"]] = ch[coff[i]:coff[i] + s["numel"]]
    np.testing.assert_array_equal(back.cpu().numpy(), expect)
    mfsdp.mfsdp_pack_owner_shards([], [], 2, canon, [None, None], ws)  # no parameters: no work


def test_llama3_8b_full_model_pack_and_reshard():
    """All 7.0e9 Llama-3-8B layer parameters (bf16-sized elements): pack into the 8-rank RoleGreedy
    shards, reshard to 4 ranks ScopeGreedy, and check every parameter's slice at the
    oracle's offsets."""
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    wl = get_config(2)
    params = _params(wl.params)
    ps = _oparams(params)
    total = sum(p.numel for p in ps)
    canon = _random(total, torch.int16, 11)
    ws = _ws(len(params))
    a, b = _segs(params, 8, 0), _segs(params, 4, 1)
    offs_a, size_a = orepack.shard_offsets(ps, _osegs(a), 8)
    offs_b, size_b = orepack.shard_offsets(ps, _osegs(b), 4)
    coff = orepack.canonical_offsets(ps)
    src = [torch.empty(n, dtype=torch.int16, device="cuda") for n in size_a]
    mfsdp.mfsdp_pack_owner_shards(params, a, 8, canon, src, ws)
    mid = torch.empty_like(canon)
    mfsdp.mfsdp_unpack_owner_shards(params, a, 8, src, mid, ws)
    del src
    dst = [torch.empty(n, dtype=torch.int16, device="cuda") for n in size_b]
    mfsdp.mfsdp_pack_owner_shards(params, b, 4, mid, dst, ws)
    torch.cuda.synchronize()
    assert torch.equal(mid, canon)
    for i, s in enumerate(b):
        got = dst[s["owner"]][offs_b[i]:offs_b[i] + s["numel"]]
        assert torch.equal(got, canon[coff[i]:coff[i] + s["numel"]]), i
    assert mfsdp.mfsdp_query_status() == 0


def test_repack_plan_matches_the_plain_calls():
    from matrix_optimizer_owner_gb300 import mfsdp
    torch.cuda.set_device(0)
    params = _odd_params(13)
    ps = _oparams(params)
    total = sum(p.numel for p in ps)
    canon = _random(total, torch.int16, 5)
    segs = _segs(params, 5, 1)
    _, size = orepack.shard_offsets(ps, _osegs(segs), 5)
    ws = _ws(len(params))
    plan = mfsdp.RepackPlan(params, segs, 5)
    a = [torch.zeros(n, dtype=torch.int16, device="cuda") for n in size]
    b = [torch.zeros(n, dtype=torch.int16, device="cuda") for n in size]
    plan.pack(canon, a, ws)
    mfsdp.mfsdp_pack_owner_shards(params, segs, 5, canon, b, ws)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    back = torch.zeros_like(canon)
    plan.unpack(a, back, ws)
    assert torch.equal(back, canon)
