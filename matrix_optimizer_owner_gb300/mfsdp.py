"""Python binding of ``include/mfsdp.h``: the same entry points, argument marshalling only.

Tensors are torch tensors on the current CUDA device (PyTorch provides device memory and
streams; every step of the optimizer runs in the library's kernels).  Each wrapper enqueues on
``torch.cuda.current_stream()`` unless a stream is given, and raises ``MfsdpError`` on a
non-zero status.
"""

from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence, Tuple

from . import _lib
from ._lib import CostModel, GemmProblem, Matrix, ParamDesc, RankResources, Segment

POLICY_ROLE_GREEDY = 0
POLICY_SCOPE_GREEDY = 1
DTYPE_F32 = 0
DTYPE_BF16 = 1
LR_ORIGINAL = 0
LR_MATCH_RMS_ADAMW = 1


class MfsdpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {_lib.STATUS_NAMES.get(status, status)}")


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise MfsdpError(fn, st)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ptr_array(tensors: Sequence) -> C.Array:
    return (C.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise TypeError(f"contribution dtype {t.dtype} is not float32 or bfloat16")


def mfsdp_version() -> int:
    return _lib.load().mfsdp_version()


def mfsdp_status_string(status: int) -> str:
    return _lib.load().mfsdp_status_string(status).decode()


# ------------------------------------------------------------------------------- planner
def mfsdp_plan_owner_set(params: Sequence[Tuple[int, int, int, bool]], world_size: int,
                         policy: int = POLICY_ROLE_GREEDY):
    """params: (rows, cols, block, is_matrix) per parameter, declaration order.

    Returns (segments, block_rank_numel, n_blocks): segments as a list of dicts with keys
    owner, role, local_offset, rank_offset, numel; block_rank_numel[k][r] = O_{B_k, r}.
    """
    lib = _lib.load()
    n = len(params)
    pd = (ParamDesc * max(n, 1))()
    for i, (r, c, b, m) in enumerate(params):
        pd[i] = ParamDesc(r, c, b, 1 if m else 0)
    seg = (Segment * max(n, 1))()
    brn = (C.c_int64 * max(n * world_size, 1))()
    nb = C.c_int64(0)
    _check("mfsdp_plan_owner_set",
           lib.mfsdp_plan_owner_set(pd, n, world_size, policy, seg, brn, C.byref(nb)))
    segs = [{"owner": s.owner, "role": s.role, "local_offset": s.local_offset,
             "rank_offset": s.rank_offset, "numel": s.numel} for s in seg[:n]]
    table = [[brn[k * world_size + r] for r in range(world_size)] for k in range(nb.value)]
    return segs, table, nb.value


def _param_array(params):
    n = len(params)
    pd = (ParamDesc * max(n, 1))()
    for i, (r, c, b, m) in enumerate(params):
        pd[i] = ParamDesc(r, c, b, 1 if m else 0)
    return pd


def _cost_model(param_bytes, grad_bytes, state_bytes, ns_steps):
    return CostModel(param_bytes, grad_bytes, state_bytes, ns_steps)


def mfsdp_score_plan(params: Sequence[Tuple[int, int, int, bool]], world_size: int,
                     segments: Sequence[dict], param_bytes: int = 2, grad_bytes: int = 2,
                     state_bytes: int = 4, ns_steps: int = 5):
    """Per-rank resource estimates and gamma_B of a plan (segments as returned by
    ``mfsdp_plan_owner_set``).  Returns (list of per-rank dicts, gamma per block)."""
    lib = _lib.load()
    n = len(params)
    seg = (Segment * max(n, 1))()
    for i, s in enumerate(segments):
        seg[i] = Segment(s["owner"], s["role"], s["local_offset"], s["rank_offset"], s["numel"])
    out = (RankResources * world_size)()
    gam = (C.c_double * max(n, 1))()
    nb = C.c_int64(0)
    model = _cost_model(param_bytes, grad_bytes, state_bytes, ns_steps)
    _check("mfsdp_score_plan", lib.mfsdp_score_plan(_param_array(params), n, world_size, seg,
                                                    C.byref(model), out, gam, C.byref(nb)))
    ranks = [{k: getattr(x, k) for k, _ in RankResources._fields_} for x in out]
    return ranks, [gam[k] for k in range(nb.value)]


def mfsdp_plan_cost_aware(params: Sequence[Tuple[int, int, int, bool]], world_size: int,
                          workspace_cap_bytes: int = 0, param_bytes: int = 2, grad_bytes: int = 2,
                          state_bytes: int = 4, ns_steps: int = 5):
    """CostAware plan.  Returns (segments, policy taken)."""
    lib = _lib.load()
    n = len(params)
    seg = (Segment * max(n, 1))()
    pol = C.c_int32(-1)
    model = _cost_model(param_bytes, grad_bytes, state_bytes, ns_steps)
    _check("mfsdp_plan_cost_aware",
           lib.mfsdp_plan_cost_aware(_param_array(params), n, world_size, C.byref(model),
                                     workspace_cap_bytes, seg, C.byref(pol)))
    segs = [{"owner": s.owner, "role": s.role, "local_offset": s.local_offset,
             "rank_offset": s.rank_offset, "numel": s.numel} for s in seg[:n]]
    return segs, pol.value


# ------------------------------------------------------------------------------- repacking
def _segment_array(segments):
    seg = (Segment * max(len(segments), 1))()
    for i, s in enumerate(segments):
        seg[i] = Segment(s["owner"], s["role"], s["local_offset"], s["rank_offset"], s["numel"])
    return seg


def mfsdp_repack_workspace_bytes(n_params: int) -> int:
    out = C.c_size_t(0)
    _check("mfsdp_repack_workspace_bytes",
           _lib.load().mfsdp_repack_workspace_bytes(n_params, C.byref(out)))
    return out.value


class RepackPlan:
    """A parameter list and its segment table marshalled once, for repeated pack / unpack
    calls (the per-call marshalling of a long list costs more host time than the copy)."""

    def __init__(self, params, segments, world_size: int):
        self.n = len(params)
        self.world_size = world_size
        self._pd = _param_array(params)
        self._seg = _segment_array(segments)

    def _ptrs(self, shards):
        return (C.c_void_p * self.world_size)(*[_ptr(t) for t in shards])

    def pack(self, canonical, shards, workspace, stream=None) -> None:
        _check("mfsdp_pack_owner_shards",
               _lib.load().mfsdp_pack_owner_shards(
                   self._pd, self.n, self._seg, self.world_size, canonical.element_size(),
                   _ptr(canonical), self._ptrs(shards), _ptr(workspace), workspace.numel(),
                   _stream(stream)))

    def unpack(self, shards, canonical, workspace, stream=None) -> None:
        _check("mfsdp_unpack_owner_shards",
               _lib.load().mfsdp_unpack_owner_shards(
                   self._pd, self.n, self._seg, self.world_size, canonical.element_size(),
                   self._ptrs(shards), _ptr(canonical), _ptr(workspace), workspace.numel(),
                   _stream(stream)))


def mfsdp_pack_owner_shards(params, segments, world_size: int, canonical, shards, workspace,
                            stream=None) -> None:
    """Canonical tensor -> owner shard tensors (``shards[r]`` may be None to skip rank r).
    All tensors share one element size; ``workspace`` is a uint8 device tensor."""
    eb = canonical.element_size()
    ptrs = (C.c_void_p * world_size)(*[_ptr(t) for t in shards])
    _check("mfsdp_pack_owner_shards",
           _lib.load().mfsdp_pack_owner_shards(_param_array(params), len(params),
                                               _segment_array(segments), world_size, eb,
                                               _ptr(canonical), ptrs, _ptr(workspace),
                                               workspace.numel(), _stream(stream)))


def mfsdp_unpack_owner_shards(params, segments, world_size: int, shards, canonical, workspace,
                              stream=None) -> None:
    """Owner shard tensors (None entries skipped) -> canonical tensor."""
    eb = canonical.element_size()
    ptrs = (C.c_void_p * world_size)(*[_ptr(t) for t in shards])
    _check("mfsdp_unpack_owner_shards",
           _lib.load().mfsdp_unpack_owner_shards(_param_array(params), len(params),
                                                 _segment_array(segments), world_size, eb, ptrs,
                                                 _ptr(canonical), _ptr(workspace),
                                                 workspace.numel(), _stream(stream)))


# ------------------------------------------------------------------------------- Shampoo
SHAMPOO_FP32 = 0
SHAMPOO_SPLIT_BF16 = 1

class ShampooSet:
    """Handle of ``mfsdp_shampoo_set``: the owned matrices of an owner Shampoo step."""

    def __init__(self, mats: Sequence[Tuple[int, int, int]]):
        lib = _lib.load()
        n = len(mats)
        arr = (Matrix * max(n, 1))()
        for i, (r, c, off) in enumerate(mats):
            arr[i] = Matrix(r, c, off)
        h = C.c_void_p()
        _check("mfsdp_shampoo_set_create", lib.mfsdp_shampoo_set_create(arr, n, C.byref(h)))
        self._h = h
        ws, ln, rn = C.c_size_t(0), C.c_int64(0), C.c_int64(0)
        _check("mfsdp_shampoo_set_sizes",
               lib.mfsdp_shampoo_set_sizes(h, C.byref(ws), C.byref(ln), C.byref(rn)))
        self.workspace_bytes, self.l_numel, self.r_numel = ws.value, ln.value, rn.value

    def close(self) -> None:
        if self._h:
            _lib.load().mfsdp_shampoo_set_destroy(self._h)
            self._h = None

    __del__ = close

    def init_state(self, eps: float, l, r, workspace, stream=None) -> None:
        _check("mfsdp_shampoo_init_state",
               _lib.load().mfsdp_shampoo_init_state(self._h, eps, _ptr(l), _ptr(r),
                                                    _ptr(workspace), workspace.numel(),
                                                    _stream(stream)))

    def step(self, grad, l, r, weights, lr: float, weight_decay: float, root_iters: int,
             workspace, stream=None, precision: int = 0) -> None:
        """``precision``: SHAMPOO_FP32 (CUDA-core fp32 products) or SHAMPOO_SPLIT_BF16 (root
        iteration and preconditioning on the tensor cores, split-bf16 operands)."""
        _check("mfsdp_shampoo_step",
               _lib.load().mfsdp_shampoo_step(self._h, _ptr(grad), _ptr(l), _ptr(r),
                                              _ptr(weights), lr, weight_decay, root_iters,
                                              precision, _ptr(workspace), workspace.numel(),
                                              _stream(stream)))


# ------------------------------------------------------------------------------- SOAP
class SoapSet:
    """Handle of ``mfsdp_soap_set``: the owned matrices of an owner SOAP step.  ``state``
    arguments are dicts of fp32 device tensors with the keys of ``SOAP_STATE_KEYS``."""

    SOAP_STATE_KEYS = ("l", "r", "q_l", "q_r", "eig_l", "eig_r", "exp_avg", "exp_avg_sq")

    def __init__(self, mats: Sequence[Tuple[int, int, int]]):
        lib = _lib.load()
        n = len(mats)
        arr = (Matrix * max(n, 1))()
        for i, (r, c, off) in enumerate(mats):
            arr[i] = Matrix(r, c, off)
        h = C.c_void_p()
        _check("mfsdp_soap_set_create", lib.mfsdp_soap_set_create(arr, n, C.byref(h)))
        self._h = h
        ws, ln, rn, el, er = (C.c_size_t(0), C.c_int64(0), C.c_int64(0), C.c_int64(0),
                              C.c_int64(0))
        _check("mfsdp_soap_set_sizes",
               lib.mfsdp_soap_set_sizes(h, C.byref(ws), C.byref(ln), C.byref(rn), C.byref(el),
                                        C.byref(er)))
        self.workspace_bytes = ws.value
        self.l_numel, self.r_numel = ln.value, rn.value
        self.eig_l_numel, self.eig_r_numel = el.value, er.value
        self.n_mats = n

    def close(self) -> None:
        if self._h:
            _lib.load().mfsdp_soap_set_destroy(self._h)
            self._h = None

    __del__ = close

    def state_sizes(self, numel: int):
        """numel of every state buffer for owner buffers of ``numel`` elements."""
        return {"l": self.l_numel, "r": self.r_numel, "q_l": self.l_numel,
                "q_r": self.r_numel, "eig_l": self.eig_l_numel, "eig_r": self.eig_r_numel,
                "exp_avg": numel, "exp_avg_sq": numel}

    @staticmethod
    def _state(state) -> "_lib.SoapState":
        return _lib.SoapState(*[_ptr(state[k]) for k in SoapSet.SOAP_STATE_KEYS])

    def init_state(self, state, workspace, stream=None) -> None:
        st = self._state(state)
        _check("mfsdp_soap_init_state",
               _lib.load().mfsdp_soap_init_state(self._h, C.byref(st), _ptr(workspace),
                                                 workspace.numel(), _stream(stream)))

    def step(self, grad, weights, state, t: int, *, lr: float, beta1: float, beta2: float,
             beta_stats: float, eps: float, weight_decay: float, max_sweeps: int, workspace,
             info=None, stream=None, jacobi_tol: float = 0.0, refresh: bool = True) -> None:
        """``refresh`` false keeps the state's eigenbases for this step (SOAP refreshes them
        every f steps)."""
        st = self._state(state)
        hy = _lib.SoapHyper(lr, beta1, beta2, beta_stats, eps, weight_decay, max_sweeps,
                            jacobi_tol, 1 if refresh else 0)
        _check("mfsdp_soap_step",
               _lib.load().mfsdp_soap_step(self._h, _ptr(grad), _ptr(weights), C.byref(st), t,
                                           C.byref(hy), _ptr(info) if info is not None else None,
                                           _ptr(workspace), workspace.numel(),
                                           _stream(stream)))


# ------------------------------------------------------------------------------- owner set
class OwnerSet:
    """Handle of ``mfsdp_owner_set``: create, query workspace, bind, destroy."""

    def __init__(self, mats: Sequence[Tuple[int, int, int]], split_max_numel: int = 0):
        lib = _lib.load()
        n = len(mats)
        arr = (Matrix * max(n, 1))()
        for i, (r, c, off) in enumerate(mats):
            arr[i] = Matrix(r, c, off)
        h = C.c_void_p()
        _check("mfsdp_owner_set_create",
               lib.mfsdp_owner_set_create(arr, n, split_max_numel, C.byref(h)))
        self.handle = h
        self.n_mats = n
        self._bound = ()

    def workspace_bytes(self) -> int:
        b = C.c_size_t(0)
        _check("mfsdp_owner_set_workspace_bytes",
               _lib.load().mfsdp_owner_set_workspace_bytes(self.handle, C.byref(b)))
        return b.value

    def split_count(self) -> int:
        k = C.c_int32(0)
        _check("mfsdp_owner_set_split_count",
               _lib.load().mfsdp_owner_set_split_count(self.handle, C.byref(k)))
        return k.value

    def bind(self, workspace, ns_input, ns_input_lo, ortho_out, ortho_lo, stream=None) -> None:
        _check("mfsdp_owner_set_bind", _lib.load().mfsdp_owner_set_bind(
            self.handle, _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(ns_input), _ptr(ns_input_lo), _ptr(ortho_out), _ptr(ortho_lo), _stream(stream)))
        self._bound = (workspace, ns_input, ns_input_lo, ortho_out, ortho_lo)  # keep alive

    def close(self) -> None:
        if self.handle:
            _lib.load().mfsdp_owner_set_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------------------- step calls
def mfsdp_owner_reduce_momentum(oset: OwnerSet, contrib: Sequence, grad_scale: float,
                                momentum: float, nesterov: bool, momentum_buf, ns_input,
                                ns_input_lo, reduced_grad_out, norm_out, stream=None) -> None:
    ptrs = _ptr_array(contrib)
    _check("mfsdp_owner_reduce_momentum", _lib.load().mfsdp_owner_reduce_momentum(
        oset.handle, ptrs, len(contrib), _dtype_code(contrib[0]), grad_scale, momentum,
        1 if nesterov else 0, _ptr(momentum_buf), _ptr(ns_input), _ptr(ns_input_lo),
        _ptr(reduced_grad_out), _ptr(norm_out), _stream(stream)))


def mfsdp_newton_schulz(oset: OwnerSet, ns_input, ns_input_lo, norm, steps: int, a: float,
                        b: float, c: float, eps: float, ortho_out, ortho_lo, stream=None) -> None:
    _check("mfsdp_newton_schulz", _lib.load().mfsdp_newton_schulz(
        oset.handle, _ptr(ns_input), _ptr(ns_input_lo), _ptr(norm), steps, a, b, c, eps,
        _ptr(ortho_out), _ptr(ortho_lo), _stream(stream)))


def mfsdp_apply_update(oset: OwnerSet, weights, ortho, ortho_lo, lr: float, weight_decay: float,
                       lr_adjust: int = LR_ORIGINAL, stream=None) -> None:
    _check("mfsdp_apply_update", _lib.load().mfsdp_apply_update(
        oset.handle, _ptr(weights), _ptr(ortho), _ptr(ortho_lo), lr, weight_decay, lr_adjust,
        _stream(stream)))


def mfsdp_adamw_tail(contrib: Sequence, grad_scale: float, param, exp_avg, exp_avg_sq, step: int,
                     lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
                     stream=None) -> None:
    ptrs = _ptr_array(contrib)
    _check("mfsdp_adamw_tail", _lib.load().mfsdp_adamw_tail(
        ptrs, len(contrib), _dtype_code(contrib[0]), grad_scale, param.numel(), _ptr(param),
        _ptr(exp_avg), _ptr(exp_avg_sq), step, lr, beta1, beta2, eps, weight_decay,
        _stream(stream)))


def mfsdp_query_status(stream=None) -> int:
    out = C.c_int32(0)
    _check("mfsdp_query_status", _lib.load().mfsdp_query_status(_stream(stream), C.byref(out)))
    return out.value


def mfsdp_set_wait_limit_ns(limit_ns: int) -> None:
    _check("mfsdp_set_wait_limit_ns", _lib.load().mfsdp_set_wait_limit_ns(limit_ns))


def mfsdp_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check("mfsdp_selftest_wait_timeout",
           _lib.load().mfsdp_selftest_wait_timeout(limit_ns, _stream(stream)))


# ------------------------------------------------------------------------------- fp32 GEMM
def mfsdp_gemm_f32_batched(problems, trans_a: bool = False, trans_b: bool = False,
                           workspace=None, stream=None) -> None:
    """C_i = alpha_i op(A_i) op(B_i) + beta_i C_i for every (A, B, C, alpha, beta) in
    ``problems`` (fp32 2D tensors on the current device, row-major with unit column stride);
    op = transpose where ``trans_a`` / ``trans_b``.  ``workspace`` (uint8 tensor) defaults
    to a fresh one of mfsdp_gemm_f32_workspace_bytes(len(problems)) bytes."""
    import torch
    lib = _lib.load()
    n = len(problems)
    tab = (GemmProblem * max(n, 1))()
    for i, (a, b, c, alpha, beta) in enumerate(problems):
        for t in (a, b, c):
            if t.dtype != torch.float32 or t.dim() != 2 or t.stride(1) != 1:
                raise TypeError("fp32 2D row-major tensors expected")
        m, k = (a.shape[1], a.shape[0]) if trans_a else (a.shape[0], a.shape[1])
        nn = b.shape[0] if trans_b else b.shape[1]
        tab[i] = GemmProblem(a.data_ptr(), b.data_ptr(), c.data_ptr(), m, nn, k, a.stride(0),
                             b.stride(0), c.stride(0), alpha, beta)
    if workspace is None:
        workspace = torch.empty(max(lib.mfsdp_gemm_f32_workspace_bytes(n), 1), dtype=torch.uint8,
                                device=problems[0][2].device if n else None)
    _check("mfsdp_gemm_f32_batched",
           lib.mfsdp_gemm_f32_batched(tab, n, 1 if trans_a else 0, 1 if trans_b else 0,
                                      _ptr(workspace), workspace.numel(), _stream(stream)))

