"""mfsdp_owner_reduce_momentum_noalloc against mfsdp_owner_reduce_momentum.

The no-allocation entry point is for callers of this library that cannot allocate device
memory — code living under another system's memory manager, or processes that reserve all
device memory up front and must not allocate on the step path — and so cannot hand the
library a workspace.  It keeps its scratch in a fixed array in the library's own device memory
that every call reuses.  These tests call it through the C ABI twice in a row (the second call
runs on the scratch the first one left behind) and compare every output with the
workspace-backed entry point on the same inputs, within the streaming tolerance of the other
parity tests (1e-5 relative).  This file runs last so that a failure here does not hide the
results of the other tests; it also passes when run on its own in a fresh process.
"""

import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    d = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / d) if d > 0 else float(np.linalg.norm(a))


def _max_rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    m = np.max(np.abs(b))
    return float(np.max(np.abs(a - b)) / m) if m > 0 else float(np.max(np.abs(a)))


def test_noalloc_matches_workspace_entry_on_two_calls():
    from matrix_optimizer_owner_gb300 import _lib, mfsdp, owner_step
    lib = _lib.load()
    # large and small, tall and wide, split and bf16-only, one matrix at an unaligned offset
    shapes = [(768, 2304), (2304, 768), (256, 64), (100, 100), (64, 64), (1, 64), (300, 700)]
    offsets, o = [], 0
    for k, (r, c) in enumerate(shapes):
        offsets.append(o)
        o += r * c + (5 if k == 3 else 0)
    split_max = 65536
    W = 4
    runner = owner_step.OwnerStep(shapes, offsets, 0, split_max_numel=split_max)
    n = runner.n
    dev = runner.device
    mom2 = torch.zeros(n, dtype=torch.float32, device=dev)
    ns2 = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    lo2 = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grad1 = torch.zeros(n, dtype=torch.float32, device=dev)
    grad2 = torch.zeros(n, dtype=torch.float32, device=dev)
    norm2 = torch.zeros(len(shapes), dtype=torch.float32, device=dev)
    table = (_lib.Matrix * len(shapes))(*[_lib.Matrix(r, c, off)
                                          for (r, c), off in zip(shapes, offsets)])
    g = torch.Generator(device=dev)
    for call in range(2):
        g.manual_seed(1234 + call)
        contribs = [(torch.randn(n, generator=g, device=dev) * 1e-3).to(torch.bfloat16)
                    for _ in range(W)]
        mfsdp.mfsdp_owner_reduce_momentum(runner.oset, contribs, 1.0, 0.95, True,
                                          runner.momentum, runner.ns_input, runner.ns_input_lo,
                                          grad1, runner.norm)
        ptrs = (C.c_void_p * W)(*[t.data_ptr() for t in contribs])
        st = lib.mfsdp_owner_reduce_momentum_noalloc(
            table, len(shapes), split_max, ptrs, W, mfsdp.DTYPE_BF16, 1.0, 0.95, 1,
            mom2.data_ptr(), ns2.data_ptr(), lo2.data_ptr(), grad2.data_ptr(), norm2.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
        assert st == 0, _lib.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        assert mfsdp.mfsdp_query_status() == 0
        for a, b in ((grad2, grad1), (mom2, runner.momentum), (ns2, runner.ns_input),
                     (lo2, runner.ns_input_lo), (norm2, runner.norm)):
            assert _rel(a, b) <= TOL and _max_rel(a, b) <= TOL, call


def test_noalloc_rejects_problems_beyond_its_scratch():
    from matrix_optimizer_owner_gb300 import _lib
    lib = _lib.load()
    ptrs = (C.c_void_p * 1)(256)
    big = (_lib.Matrix * 1)(_lib.Matrix(1 << 30, 1 << 20, 0))    # 2^50 elements
    st = lib.mfsdp_owner_reduce_momentum_noalloc(big, 1, 0, ptrs, 1, 1, 1.0, 0.95, 1, 256, 512,
                                                 None, None, 768, None)
    assert st == -5  # MFSDP_EWORKSPACE, before anything is enqueued
    many = (_lib.Matrix * 4097)(*[_lib.Matrix(1, 8, 8 * i) for i in range(4097)])
    st = lib.mfsdp_owner_reduce_momentum_noalloc(many, 4097, 0, ptrs, 1, 1, 1.0, 0.95, 1, 256,
                                                 512, None, None, 768, None)
    assert st == -5
