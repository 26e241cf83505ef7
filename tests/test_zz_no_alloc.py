"""mfsdp_owner_reduce_momentum_noalloc against mfsdp_owner_reduce_momentum.

The no-allocation entry point is for callers of this library that cannot allocate device
memory — code living under another system's memory manager, or processes that reserve all
device memory up front and must not allocate on the step path — and so cannot hand the
library a workspace.  It keeps its scratch in a fixed array in the library's own device memory
that every call reuses.  These tests call it through the C ABI twice in a row (the second call
runs on the scratch the first one left behind).  Both entry points launch the same deposit and
norm kernels over the same per-CTA partition, so every output must equal the workspace-backed
entry point's bit for bit; on the tiny four-matrix set the outputs are also held to the fp64
oracle at the streaming tolerance of the other parity tests (1e-5 relative), the second call
carrying the first call's momentum.  This file runs last so that a failure here does not hide
the results of the other tests; it also passes when run on its own in a fresh process.
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
        for name, a, b in (("grad", grad2, grad1), ("momentum", mom2, runner.momentum),
                           ("ns_input", ns2, runner.ns_input), ("ns_input_lo", lo2, runner.ns_input_lo),
                           ("norm", norm2, runner.norm)):
            assert torch.equal(a, b), (call, name, _rel(a, b), _max_rel(a, b))


def test_noalloc_matches_oracle_on_tiny_set_over_two_calls():
    """The scratch-array path on its own against the fp64 oracle: the tiny four-matrix set
    (64x64, 64x256, 256x64, 128x128, W = 4 fp32 contributions, every matrix in split
    precision), two calls in a row with momentum carried from the first to the second."""
    from matrix_optimizer_owner_gb300 import _lib, mfsdp
    from oracle import muon as omuon
    from workloads import get_config, synth
    lib = _lib.load()
    wl = get_config(0)
    hp = wl.hyper
    mats = [i for i, p in enumerate(wl.params) if p.is_matrix]
    shapes = [(wl.params[i].rows, wl.params[i].cols) for i in mats]
    offsets, o = [], 0
    for r, c in shapes:
        offsets.append(o)
        o += r * c
    n = o
    dev = torch.device("cuda", torch.cuda.current_device())
    mom = torch.zeros(n, dtype=torch.float32, device=dev)
    ns_hi = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    ns_lo = torch.zeros(n, dtype=torch.bfloat16, device=dev)
    grad = torch.zeros(n, dtype=torch.float32, device=dev)
    norm = torch.zeros(len(shapes), dtype=torch.float32, device=dev)
    table = (_lib.Matrix * len(shapes))(*[_lib.Matrix(r, c, off)
                                          for (r, c), off in zip(shapes, offsets)])
    B_ref = [np.zeros((r, c)) for r, c in shapes]
    for step in range(2):
        contribs = []
        for w in range(wl.W):
            buf = torch.empty(n, dtype=torch.float32, device=dev)
            for pi, off, (r, c) in zip(mats, offsets, shapes):
                buf[off:off + r * c] = synth.contribution(wl, step, pi, w, dev)
            contribs.append(buf)
        ptrs = (C.c_void_p * wl.W)(*[t.data_ptr() for t in contribs])
        st = lib.mfsdp_owner_reduce_momentum_noalloc(
            table, len(shapes), 65536, ptrs, wl.W, mfsdp.DTYPE_F32, hp.grad_scale, hp.momentum,
            1 if hp.nesterov else 0, mom.data_ptr(), ns_hi.data_ptr(), ns_lo.data_ptr(),
            grad.data_ptr(), norm.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert st == 0, _lib.STATUS_NAMES.get(st, st)
        torch.cuda.synchronize()
        assert mfsdp.mfsdp_query_status() == 0
        h = lambda t: t.double().cpu().numpy()
        U_dev = h(ns_hi) + h(ns_lo)
        for k, ((r, c), off) in enumerate(zip(shapes, offsets)):
            sl = slice(off, off + r * c)
            cs = [h(t[sl]).reshape(r, c) for t in contribs]
            G = omuon.reduce_contributions(cs, hp.grad_scale)
            B_ref[k] = omuon.momentum_update(B_ref[k], G, hp.momentum)
            U = omuon.nesterov_input(G, B_ref[k], hp.momentum, hp.nesterov)
            nu = omuon.frobenius_norm(U)
            for name, got, ref in (("G", h(grad[sl]), G), ("B", h(mom[sl]), B_ref[k]),
                                   ("U", U_dev[sl], U)):
                got = got.reshape(r, c)
                assert np.linalg.norm(got - ref) <= TOL * np.linalg.norm(ref), (step, k, name)
                assert np.max(np.abs(got - ref)) <= TOL * np.max(np.abs(ref)), (step, k, name)
            assert abs(float(norm[k]) - nu) <= TOL * nu, (step, k, float(norm[k]), nu)


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
