"""ctypes loader for ``libmfsdp.so`` and the C signatures of ``include/mfsdp.h``.

The library is built in-tree (``matrix_optimizer_owner_gb300/lib/libmfsdp.so``, see
``build.py``).  There is no fallback: if it is missing, importing the binding raises.
"""

from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmfsdp.so")

MFSDP_OK = 0
STATUS_NAMES = {
    0: "MFSDP_OK", -1: "MFSDP_EINVAL", -2: "MFSDP_ESHAPE", -3: "MFSDP_EALIGN",
    -4: "MFSDP_ENOTCONTIG", -5: "MFSDP_EWORKSPACE", -6: "MFSDP_ECUDA", -7: "MFSDP_ETIMEOUT",
    -8: "MFSDP_ENONFINITE", -9: "MFSDP_ENODEVICE",
}


class ParamDesc(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("block", C.c_int32),
                ("is_matrix", C.c_int32)]


class Segment(C.Structure):
    _fields_ = [("owner", C.c_int32), ("role", C.c_int32), ("local_offset", C.c_int64),
                ("rank_offset", C.c_int64), ("numel", C.c_int64)]


class Matrix(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("offset", C.c_int64)]


class SoapState(C.Structure):
    _fields_ = [(name, C.c_void_p) for name in
                ("l", "r", "q_l", "q_r", "eig_l", "eig_r", "exp_avg", "exp_avg_sq")]


class SoapHyper(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("beta_stats", C.c_float), ("eps", C.c_float), ("weight_decay", C.c_float),
                ("max_sweeps", C.c_int32), ("jacobi_tol", C.c_float), ("refresh", C.c_int32)]


class GemmProblem(C.Structure):
    _fields_ = [("a", C.c_void_p), ("b", C.c_void_p), ("c", C.c_void_p), ("m", C.c_int32),
                ("n", C.c_int32), ("k", C.c_int32), ("lda", C.c_int32), ("ldb", C.c_int32),
                ("ldc", C.c_int32), ("alpha", C.c_float), ("beta", C.c_float)]


class CostModel(C.Structure):
    _fields_ = [("param_bytes", C.c_int32), ("grad_bytes", C.c_int32),
                ("state_bytes", C.c_int32), ("ns_steps", C.c_int32)]


class RankResources(C.Structure):
    _fields_ = [("param_bytes", C.c_int64), ("grad_bytes", C.c_int64),
                ("state_bytes", C.c_int64), ("comm_bytes", C.c_int64),
                ("workspace_bytes", C.c_int64), ("optimizer_flops", C.c_double)]


_vp = C.c_void_p
_i32, _i64, _f32, _u64 = C.c_int32, C.c_int64, C.c_float, C.c_uint64

SIGNATURES = {
    "mfsdp_plan_owner_set": (C.c_int, [C.POINTER(ParamDesc), _i64, _i32, _i32,
                                       C.POINTER(Segment), C.POINTER(_i64), C.POINTER(_i64)]),
    "mfsdp_score_plan": (C.c_int, [C.POINTER(ParamDesc), _i64, _i32, C.POINTER(Segment),
                                   C.POINTER(CostModel), C.POINTER(RankResources),
                                   C.POINTER(C.c_double), C.POINTER(_i64)]),
    "mfsdp_plan_cost_aware": (C.c_int, [C.POINTER(ParamDesc), _i64, _i32, C.POINTER(CostModel),
                                        _i64, C.POINTER(Segment), C.POINTER(_i32)]),
    "mfsdp_repack_workspace_bytes": (C.c_int, [_i64, C.POINTER(C.c_size_t)]),
    "mfsdp_pack_owner_shards": (C.c_int, [C.POINTER(ParamDesc), _i64, C.POINTER(Segment), _i32,
                                          _i32, _vp, C.POINTER(_vp), _vp, C.c_size_t, _vp]),
    "mfsdp_unpack_owner_shards": (C.c_int, [C.POINTER(ParamDesc), _i64, C.POINTER(Segment),
                                            _i32, _i32, C.POINTER(_vp), _vp, _vp, C.c_size_t,
                                            _vp]),
    "mfsdp_shampoo_set_create": (C.c_int, [C.POINTER(Matrix), _i32, C.POINTER(_vp)]),
    "mfsdp_shampoo_set_destroy": (C.c_int, [_vp]),
    "mfsdp_shampoo_set_sizes": (C.c_int, [_vp, C.POINTER(C.c_size_t), C.POINTER(_i64),
                                          C.POINTER(_i64)]),
    "mfsdp_shampoo_init_state": (C.c_int, [_vp, _f32, _vp, _vp, _vp, C.c_size_t, _vp]),
    "mfsdp_shampoo_step": (C.c_int, [_vp, _vp, _vp, _vp, _vp, _f32, _f32, _i32, _i32, _vp,
                                     C.c_size_t, _vp]),
    "mfsdp_gemm_f32_workspace_bytes": (C.c_size_t, [_i32]),
    "mfsdp_gemm_f32_batched": (C.c_int, [C.POINTER(GemmProblem), _i32, _i32, _i32, _vp,
                                         C.c_size_t, _vp]),
    "mfsdp_soap_set_create": (C.c_int, [C.POINTER(Matrix), _i32, C.POINTER(_vp)]),
    "mfsdp_soap_set_destroy": (C.c_int, [_vp]),
    "mfsdp_soap_set_sizes": (C.c_int, [_vp, C.POINTER(C.c_size_t), C.POINTER(_i64),
                                       C.POINTER(_i64), C.POINTER(_i64), C.POINTER(_i64)]),
    "mfsdp_soap_init_state": (C.c_int, [_vp, C.POINTER(SoapState), _vp, C.c_size_t, _vp]),
    "mfsdp_soap_step": (C.c_int, [_vp, _vp, _vp, C.POINTER(SoapState), _i64,
                                  C.POINTER(SoapHyper), _vp, _vp, C.c_size_t, _vp]),
    "mfsdp_owner_set_create": (C.c_int, [C.POINTER(Matrix), _i32, _i64, C.POINTER(_vp)]),
    "mfsdp_owner_set_destroy": (C.c_int, [_vp]),
    "mfsdp_owner_set_workspace_bytes": (C.c_int, [_vp, C.POINTER(C.c_size_t)]),
    "mfsdp_owner_set_split_count": (C.c_int, [_vp, C.POINTER(_i32)]),
    "mfsdp_owner_set_bind": (C.c_int, [_vp, _vp, C.c_size_t, _vp, _vp, _vp, _vp, _vp]),
    "mfsdp_owner_reduce_momentum": (C.c_int, [_vp, C.POINTER(_vp), _i32, _i32, _f32, _f32, _i32,
                                              _vp, _vp, _vp, _vp, _vp, _vp]),
    "mfsdp_newton_schulz": (C.c_int, [_vp, _vp, _vp, _vp, _i32, _f32, _f32, _f32, _f32, _vp, _vp,
                                      _vp]),
    "mfsdp_apply_update": (C.c_int, [_vp, _vp, _vp, _vp, _f32, _f32, _i32, _vp]),
    "mfsdp_adamw_tail": (C.c_int, [C.POINTER(_vp), _i32, _i32, _f32, _i64, _vp, _vp, _vp, _i64,
                                   _f32, _f32, _f32, _f32, _f32, _vp]),
    "mfsdp_owner_reduce_momentum_noalloc": (C.c_int, [C.POINTER(Matrix), _i32, _i64,
                                                      C.POINTER(_vp), _i32, _i32, _f32, _f32,
                                                      _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mfsdp_query_status": (C.c_int, [_vp, C.POINTER(_i32)]),
    "mfsdp_status_string": (C.c_char_p, [C.c_int]),
    "mfsdp_set_wait_limit_ns": (C.c_int, [_u64]),
    "mfsdp_selftest_wait_timeout": (C.c_int, [_u64, _vp]),
    "mfsdp_version": (C.c_int, []),
}

_LIB = None


def load() -> C.CDLL:
    """Load the library once; raise if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m matrix_optimizer_owner_gb300.build`")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB
