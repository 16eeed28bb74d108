"""ctypes declarations of the C ABI in include/fadam.h.

Argument marshalling only: every step of the update runs in libfadam.so.
Loading fails loudly when the library has not been built; there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
# FADAM_LIBRARY selects another build of the library (e.g. one compiled with
# different tuning defines by build.build(defines=..., lib=...))
LIB_PATH = os.environ.get("FADAM_LIBRARY") or os.path.join(_PKG, "_build", "libfadam.so")

# status codes
OK, EINVAL, EDTYPE, EALIGN, ECUDA, ETIMEOUT, ELIMIT = 0, 1, 2, 3, 4, 5, 6
# modes
MODE_L2, MODE_ADAMW = 0, 1
# dtypes
DT_NONE, DT_F32, DT_BF16, DT_F16 = 0, 1, 2, 3
# plan flags
CAPTURABLE, REMAINDERS, CHECK_FINITE, STEP_PREADVANCED = 1, 2, 4, 8
SCALED_STATES = 16
MOMENTS_BF16, MOMENTS_F16 = 32, 64
RECIP_BC = 128  # 16-bit state forms: multiply by 1/bc1, 1/bc2 instead of dividing
TEST_BARRIER_TIMEOUT = 0x80000000  # diagnostic: the screen's grid barrier runs out
EXCHANGE_AVERAGE, EXCHANGE_ACCUMULATE = 1, 2  # reduce_flags of fadam_plan_set_exchange
MAX_GROUPS = 32
MAX_SOURCES = 16
MAX_DESTS = 16


class Tensor(ctypes.Structure):
    """fadam_tensor."""
    _fields_ = [("p", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("g", ctypes.c_void_p), ("p_out", ctypes.c_void_p), ("rem", ctypes.c_void_p),
                ("numel", ctypes.c_int64), ("group", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class Group(ctypes.Structure):
    """fadam_group."""
    _fields_ = [("mode", ctypes.c_int32), ("bias_correction", ctypes.c_int32),
                ("beta1", ctypes.c_float), ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("lr", ctypes.c_float),
                ("grad_scale", ctypes.c_float), ("step", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("lr_dev", ctypes.c_void_p),
                ("grad_scale_dev", ctypes.c_void_p), ("step_dev", ctypes.c_void_p)]


class PlanInfo(ctypes.Structure):
    """fadam_plan_info."""
    _fields_ = [("n_tensors", ctypes.c_int64), ("n_elements", ctypes.c_int64),
                ("n_items", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
                ("grid", ctypes.c_int32), ("block", ctypes.c_int32),
                ("blocks_per_sm", ctypes.c_int32), ("sm_count", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("device", ctypes.c_int32),
                ("bytes_per_step", ctypes.c_double), ("check_bytes_per_step", ctypes.c_double)]


class PackItem(ctypes.Structure):
    """fadam_pack_item."""
    _fields_ = [("tensor", ctypes.c_int64), ("offset", ctypes.c_int64), ("n", ctypes.c_int32),
                ("vec", ctypes.c_int32)]


# (name, restype, argtypes) for every function the header declares
_vp, _i32, _i64, _u32, _f32 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                               ctypes.c_float)
SIGNATURES = [
    ("fadam_plan_create", _i32, [ctypes.POINTER(Tensor), _i64, ctypes.POINTER(Group), _i32, _i32,
                                 _i32, _i32, _u32, ctypes.POINTER(_vp)]),
    ("fadam_plan_set_groups", _i32, [_vp, ctypes.POINTER(Group), _i32]),
    ("fadam_step", _i32, [_vp, _vp, _vp]),
    ("fadam_step_host_grads", _i32, [_vp, ctypes.POINTER(_vp), _vp, ctypes.POINTER(_i32), _vp]),
    ("fadam_plan_status", _i32, [_vp, ctypes.POINTER(_i32)]),
    ("fadam_plan_get_info", _i32, [_vp, ctypes.POINTER(PlanInfo)]),
    ("fadam_plan_destroy", _i32, [_vp]),
    ("fadam_step_once", _i32, [ctypes.POINTER(Tensor), _i64, _i32, _i32, _f32, _f32, _f32, _f32,
                               _f32, _vp, _i32, _vp, _f32, _vp, _vp, _i32, _i32, _vp]),
    ("fadam_pack_dry", _i32, [ctypes.POINTER(Tensor), _i64, _i32, _i32, _i32, _i32, _u32, _i32,
                              ctypes.POINTER(PackItem), _i64, ctypes.POINTER(_i32),
                              ctypes.POINTER(_i64)]),
    ("fadam_chunk_dry", _i32, [ctypes.POINTER(Tensor), _i64, _i32, _i32, _i32, _i32, _u32, _i32,
                               _i64, ctypes.POINTER(_i32), _i64, ctypes.POINTER(_i64)]),
    ("fadam_step_noalloc", _i32, [ctypes.POINTER(Tensor), _i64, ctypes.POINTER(Group), _i32, _i32,
                                  _i32, _i32, _u32, _vp, _vp]),
    ("fadam_grad_sumsq", _i32, [_vp, _vp, _vp]),
    ("fadam_clip_apply", _i32, [_vp, _vp, _f32, _vp, _vp, _vp, _vp]),
    ("fadam_plan_set_exchange", _i32, [_vp, _vp, ctypes.POINTER(_vp), _i32, _i32, _vp,
                                       ctypes.POINTER(_vp), _i32]),
    ("fadam_grad_reduce", _i32, [_vp, _vp]),
    ("fadam_step_reduce", _i32, [_vp, _vp, _vp]),
    ("fadam_plan_set_state_scales", _i32, [_vp, _vp]),
    ("fadam_status_string", ctypes.c_char_p, [_i32]),
    ("fadam_last_error", ctypes.c_char_p, []),
    ("fadam_version", _i32, []),
]

_LIB = None


class FadamError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: status {status} ({_status_name(status)}): {detail}")
        self.status = status


def _status_name(status: int) -> str:
    names = {OK: "ok", EINVAL: "invalid argument", EDTYPE: "unsupported dtype",
             EALIGN: "misaligned pointer", ECUDA: "CUDA error", ETIMEOUT: "device wait timed out",
             ELIMIT: "size beyond maximum"}
    return names.get(status, "unknown")


def lib() -> ctypes.CDLL:
    """Load libfadam.so; raises when it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no fallback path exists)")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(status: int, where: str) -> None:
    if status != OK:
        raise FadamError(status, where, lib().fadam_last_error().decode())
