"""CPU oracle for the fused Adam/AdamW shard step.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the library under
``adamw_optimizer_step_persistent_gb300`` never does, and it shares no code
with it.  The per-element arithmetic is plain C (``fadam_oracle.c``); this
module only marshals numpy arrays and carries the per-step bookkeeping:

* the step counters: every group advances, empty or not ("[PyTorch] Advance
  FusedAdam step counter for empty param groups", Fix section);
* the regular path advances each counter by one before the update
  (distributed_fused_adam.py, ``step``), the capturable path by
  ``noop != 1`` (same function, capturable branch), and with a set noop flag
  nothing changes at all (DistAdamCapturableFunctor, early return);
* an optional inf/nan screen of the scaled gradients that sets the noop flag
  before any state is touched.

Around the step, the one-GPU stand-in for the data-parallel exchange (the
reduce-scatter that fills this rank's gradient shard, the all-gather of the
param-out shard) is plain numpy float32 arithmetic in this module.

Arrays: fp32 data are ``np.float32``; bf16 and fp16 data are ``np.uint16``
bit patterns; remainders are ``np.int16``.  Every function is pinned by
``tests/test_oracle_pins.py``; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

from .build import build as _build
from .build import build_timed as _build_timed

DT_NONE, DT_F32, DT_BF16, DT_F16 = 0, 1, 2, 3
MODE_L2, MODE_ADAMW = 0, 1

_LIB = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_vp = ctypes.c_void_p
L_F32_ARGS = [_i64, ctypes.c_int, ctypes.c_int, _i32, _f32, _f32, _f32, _f32, _f32, _f32, _vp,
              _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_int]
L_REM_ARGS = [_i64, ctypes.c_int, ctypes.c_int, _i32, _f32, _f32, _f32, _f32, _f32, _f32, _vp,
              _vp, _vp, _vp, _vp, ctypes.c_int, _vp]


def lib():
    """Load (building first if needed) the oracle's C library."""
    global _LIB
    if _LIB is None:
        L = ctypes.CDLL(_build())
        L.oracle_bias_correction.restype = _f32
        L.oracle_bias_correction.argtypes = [_f32, _i32]
        L.oracle_adam_f32.restype = None
        L.oracle_adam_f32.argtypes = L_F32_ARGS
        L.oracle_adam_rem.restype = None
        L.oracle_adam_rem.argtypes = L_REM_ARGS
        L.oracle_adam_state.restype = None
        L.oracle_adam_state.argtypes = [_i64, ctypes.c_int, ctypes.c_int, _i32, _f32, _f32,
                                        _f32, _f32, _f32, _f32, _vp, _vp, _vp, ctypes.c_int,
                                        _vp, ctypes.c_int, _vp, ctypes.c_int]
        L.oracle_adam_moments.restype = None
        L.oracle_adam_moments.argtypes = [_i64, ctypes.c_int, ctypes.c_int, _i32, _f32, _f32,
                                          _f32, _f32, _f32, _f32, _vp, _vp, _vp, ctypes.c_int,
                                          _vp, ctypes.c_int, _vp, ctypes.c_int]
        L.oracle_adam_f64.restype = None
        L.oracle_adam_f64.argtypes = [_i64, ctypes.c_int, ctypes.c_int, _i32, _f32, _f32,
                                      _f32, _f32, _f32, _f32, _vp, _vp, _vp, _vp]
        L.oracle_sumsq.restype = ctypes.c_double
        L.oracle_sumsq.argtypes = [_i64, _vp, ctypes.c_int]
        L.oracle_any_nonfinite.restype = ctypes.c_int
        L.oracle_any_nonfinite.argtypes = [_i64, _vp, ctypes.c_int, _f32]
        L.oracle_rem_pack_n.restype = None
        L.oracle_rem_pack_n.argtypes = [_i64, _vp, _vp, _vp]
        L.oracle_rem_split_n.restype = None
        L.oracle_rem_split_n.argtypes = [_i64, _vp, _vp, _vp]
        for name in ("oracle_f32_to_bf16_n", "oracle_f32_to_f16_n", "oracle_bf16_to_f32_n",
                     "oracle_f16_to_f32_n"):
            getattr(L, name).restype = None
            getattr(L, name).argtypes = [_i64, _vp, _vp]
        _LIB = L
    return _LIB


_TIMED = None


def timed_lib():
    """The timed-only build (-O3 -fopenmp, the same source plus an OpenMP
    driver that splits each tensor across the threads): for the benchmark's
    CPU baseline only; the tests use ``lib()``."""
    global _TIMED
    if _TIMED is None:
        L = ctypes.CDLL(_build_timed())
        L.oracle_omp_threads.restype = ctypes.c_int
        L.oracle_omp_threads.argtypes = []
        L.oracle_omp_adam_f32.restype = None
        L.oracle_omp_adam_f32.argtypes = L_F32_ARGS
        L.oracle_omp_adam_rem.restype = None
        L.oracle_omp_adam_rem.argtypes = L_REM_ARGS
        _TIMED = L
    return _TIMED


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _check(a: np.ndarray, dtype, n: int, what: str):
    assert a.dtype == dtype, f"{what}: expected {np.dtype(dtype)}, got {a.dtype}"
    assert a.size == n, f"{what}: expected {n} elements, got {a.size}"


_G_NP = {DT_F32: np.float32, DT_BF16: np.uint16, DT_F16: np.uint16}


# ---- scalar helpers ---------------------------------------------------------

def bias_correction(beta: float, step: int) -> np.float32:
    """1 - beta^step with beta a float, pow in double, rounded once to float."""
    return np.float32(lib().oracle_bias_correction(float(np.float32(beta)), int(step)))


def _map_n(fn, x, out_dtype):
    x = np.ascontiguousarray(x)
    out = np.empty(x.shape, dtype=out_dtype)
    fn(x.size, _ptr(x), _ptr(out))
    return out


def f32_to_bf16(x) -> np.ndarray:
    return _map_n(lib().oracle_f32_to_bf16_n, np.asarray(x, dtype=np.float32), np.uint16)


def f32_to_f16(x) -> np.ndarray:
    return _map_n(lib().oracle_f32_to_f16_n, np.asarray(x, dtype=np.float32), np.uint16)


def bf16_to_f32(h) -> np.ndarray:
    return _map_n(lib().oracle_bf16_to_f32_n, np.asarray(h, dtype=np.uint16), np.float32)


def f16_to_f32(h) -> np.ndarray:
    return _map_n(lib().oracle_f16_to_f32_n, np.asarray(h, dtype=np.uint16), np.float32)


def rem_pack(hi, rem) -> np.ndarray:
    """(bf16 high half, int16 remainder) -> fp32 bit patterns (uint32)."""
    hi = np.ascontiguousarray(hi, dtype=np.uint16)
    rem = np.ascontiguousarray(rem, dtype=np.int16)
    out = np.empty(hi.shape, dtype=np.uint32)
    lib().oracle_rem_pack_n(hi.size, _ptr(hi), _ptr(rem), _ptr(out))
    return out


def rem_split(bits):
    """fp32 bit patterns (uint32) -> (bf16 high half, int16 remainder)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint32)
    hi = np.empty(bits.shape, dtype=np.uint16)
    rem = np.empty(bits.shape, dtype=np.int16)
    lib().oracle_rem_split_n(bits.size, _ptr(bits), _ptr(hi), _ptr(rem))
    return hi, rem


# ---- per-tensor update ------------------------------------------------------

@dataclass
class Group:
    """Hyper-parameters of one param group (the functor's arguments)."""
    mode: int = MODE_ADAMW
    bias_correction: int = 1
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    lr: float = 1e-3
    grad_scale: float = 1.0


def adam_f32(group: Group, step: int, p, m, v, g, g_dtype=DT_F32, p_out=None,
             out_dtype=DT_NONE, timed: bool = False) -> None:
    """Update one tensor with an fp32 master in place (p, m, v, p_out).
    ``timed``: run it through the timed OpenMP build instead (the CPU
    baseline)."""
    n = p.size
    _check(p, np.float32, n, "p")
    _check(m, np.float32, n, "m")
    _check(v, np.float32, n, "v")
    _check(g, _G_NP[g_dtype], n, "g")
    if out_dtype != DT_NONE:
        _check(p_out, np.float32 if out_dtype == DT_F32 else np.uint16, n, "p_out")
    fn = timed_lib().oracle_omp_adam_f32 if timed else lib().oracle_adam_f32
    fn(n, group.mode, group.bias_correction, step, group.beta1, group.beta2, group.eps,
       group.weight_decay, group.lr, group.grad_scale, _ptr(p), _ptr(m), _ptr(v), _ptr(g),
       g_dtype, _ptr(p_out) if out_dtype != DT_NONE else None, out_dtype)


_S_NP = {DT_F32: np.float32, DT_BF16: np.uint16, DT_F16: np.uint16}


def adam_state(group: Group, step: int, p, m, v, state_dtype, g, g_dtype=DT_F32, p_out=None,
               out_dtype=DT_NONE) -> None:
    """Update one tensor whose p, m, v all have `state_dtype` (in place)."""
    n = p.size
    for a, w in ((p, "p"), (m, "m"), (v, "v")):
        _check(a, _S_NP[state_dtype], n, w)
    _check(g, _G_NP[g_dtype], n, "g")
    if out_dtype != DT_NONE:
        _check(p_out, np.float32 if out_dtype == DT_F32 else np.uint16, n, "p_out")
    lib().oracle_adam_state(n, group.mode, group.bias_correction, step, group.beta1,
                            group.beta2, group.eps, group.weight_decay, group.lr,
                            group.grad_scale, _ptr(p), _ptr(m), _ptr(v), state_dtype, _ptr(g),
                            g_dtype, _ptr(p_out) if out_dtype != DT_NONE else None, out_dtype)


def adam_moments(group: Group, step: int, p, m, v, moment_dtype, g, g_dtype=DT_F32, p_out=None,
                 out_dtype=DT_NONE) -> None:
    """Update one tensor with an fp32 master p and 16-bit moments m, v of
    `moment_dtype` (uint16 bits), in place."""
    n = p.size
    _check(p, np.float32, n, "p")
    for a, w in ((m, "m"), (v, "v")):
        _check(a, np.uint16, n, w)
    _check(g, _G_NP[g_dtype], n, "g")
    if out_dtype != DT_NONE:
        _check(p_out, np.float32 if out_dtype == DT_F32 else np.uint16, n, "p_out")
    lib().oracle_adam_moments(n, group.mode, group.bias_correction, step, group.beta1,
                              group.beta2, group.eps, group.weight_decay, group.lr,
                              group.grad_scale, _ptr(p), _ptr(m), _ptr(v), moment_dtype, _ptr(g),
                              g_dtype, _ptr(p_out) if out_dtype != DT_NONE else None, out_dtype)


def adam_rem(group: Group, step: int, p_hi, rem, m, v, g, g_dtype, p_out,
             timed: bool = False) -> None:
    """Update one tensor whose master is bf16 high half + int16 remainder
    (``timed``: through the timed OpenMP build)."""
    n = p_hi.size
    _check(p_hi, np.uint16, n, "p_hi")
    _check(rem, np.int16, n, "rem")
    _check(m, np.float32, n, "m")
    _check(v, np.float32, n, "v")
    _check(g, _G_NP[g_dtype], n, "g")
    _check(p_out, np.uint16, n, "p_out")
    fn = timed_lib().oracle_omp_adam_rem if timed else lib().oracle_adam_rem
    fn(n, group.mode, group.bias_correction, step, group.beta1, group.beta2, group.eps,
       group.weight_decay, group.lr, group.grad_scale, _ptr(p_hi), _ptr(rem), _ptr(m), _ptr(v),
       _ptr(g), g_dtype, _ptr(p_out))


def adam_f64(group: Group, step: int, p, m, v, g) -> None:
    """Double-precision evaluation (error analysis only); arrays are float64."""
    n = p.size
    for a, w in ((p, "p"), (m, "m"), (v, "v"), (g, "g")):
        _check(a, np.float64, n, w)
    lib().oracle_adam_f64(n, group.mode, group.bias_correction, step, group.beta1,
                          group.beta2, group.eps, group.weight_decay, group.lr,
                          group.grad_scale, _ptr(p), _ptr(m), _ptr(v), _ptr(g))


def sumsq(g, g_dtype) -> float:
    """Sum of squares of one gradient tensor, in double."""
    g = np.ascontiguousarray(g)
    return float(lib().oracle_sumsq(g.size, _ptr(g), g_dtype))


def any_nonfinite(g, g_dtype, grad_scale) -> bool:
    g = np.ascontiguousarray(g)
    return bool(lib().oracle_any_nonfinite(g.size, _ptr(g), g_dtype, float(grad_scale)))


# ---- whole shard step -------------------------------------------------------

@dataclass
class Tensor:
    """One tensor of the shard, as numpy arrays updated in place.

    For an fp32 master set ``p``; for 16-bit state set ``p``, ``m``, ``v`` as
    uint16 bits and ``state_dtype``; for an fp32 master with 16-bit moments
    set ``m``, ``v`` as uint16 bits and ``moment_dtype``; for the remainder form set ``p_hi``
    (bf16 bits) and ``rem`` and give ``p_out`` (bf16 bits, may be ``p_hi``).
    """
    group: int
    m: np.ndarray
    v: np.ndarray
    g: np.ndarray
    g_dtype: int = DT_F32
    p: Optional[np.ndarray] = None
    p_hi: Optional[np.ndarray] = None
    rem: Optional[np.ndarray] = None
    p_out: Optional[np.ndarray] = None
    out_dtype: int = DT_NONE
    state_dtype: int = DT_F32  # dtype of p, m and v (fp32 master form)
    moment_dtype: int = DT_NONE  # bf16 or fp16: m, v in it, fp32 p (else the state dtype)
    scales: Optional[np.ndarray] = None  # scaled 16-bit state: float32[3] (p, m, v)


@dataclass
class Shard:
    """A shard: param groups, tensors and the step counters.

    ``step_slot[i]`` names the counter group i uses; groups may share one
    counter (one optimizer-wide step) or own one each (one per group).
    """
    groups: List[Group]
    tensors: List[Tensor]
    steps: List[int] = field(default_factory=list)
    step_slot: List[int] = field(default_factory=list)

    def __post_init__(self):
        if not self.step_slot:
            self.step_slot = list(range(len(self.groups)))
        if not self.steps:
            self.steps = [0] * (max(self.step_slot) + 1 if self.step_slot else 0)


def shard_step(shard: Shard, *, capturable: bool, noop: bool = False,
               check_finite: bool = False, step_preadvanced: bool = False) -> bool:
    """Apply one optimizer step to every tensor of the shard.

    Returns the noop flag as it stands after the step (it can only go from
    0 to 1, through the inf/nan screen).  With the flag set nothing changes:
    neither the tensors nor, on either path, the step counters.
    """
    if check_finite and not noop:
        for t in shard.tensors:
            if any_nonfinite(t.g, t.g_dtype, shard.groups[t.group].grad_scale):
                noop = True
                break
    if noop:
        return True
    if not (capturable and step_preadvanced):
        for slot in sorted(set(shard.step_slot)):
            shard.steps[slot] += 1
    for t in shard.tensors:
        grp = shard.groups[t.group]
        step = shard.steps[shard.step_slot[t.group]]
        if t.rem is not None:
            adam_rem(grp, step, t.p_hi, t.rem, t.m, t.v, t.g, t.g_dtype, t.p_out)
        elif t.scales is not None:
            adam_scaled(grp, step, t.p, t.m, t.v, t.scales, t.state_dtype, t.g, t.g_dtype,
                        t.p_out, t.out_dtype)
        elif t.moment_dtype != DT_NONE:
            adam_moments(grp, step, t.p, t.m, t.v, t.moment_dtype, t.g, t.g_dtype, t.p_out,
                         t.out_dtype)
        elif t.state_dtype != DT_F32:
            adam_state(grp, step, t.p, t.m, t.v, t.state_dtype, t.g, t.g_dtype, t.p_out,
                       t.out_dtype)
        else:
            adam_f32(grp, step, t.p, t.m, t.v, t.g, t.g_dtype, t.p_out, t.out_dtype)
    return False


def group_steps(shard: Shard) -> List[int]:
    """The step each group reports (its counter's value)."""
    return [shard.steps[s] for s in shard.step_slot]


# ---- gradient norm and clipping ---------------------------------------------
#
# "apex/contrib/optimizers/distributed_fused_adam.py": _local_grad_norm (sum
# of squares of the local gradient shard), grad_norm (all-reduced, square
# root, times the grad scale), clip_grad_norm (clip_coef = max_norm /
# (total_norm + 1e-6), clamped to at most 1, multiplied into the grad
# scale) and step() (found_inf = not isfinite(grad norm), copied into the
# noop flag).  Readings: with one grad scale per group the squared norm is
# sum_g scale_g^2 * sum_{i in g} g_i^2, accumulated in double (the norm of
# the scaled gradient; with one scale for all groups this is the page's
# norm times scale); the norm is that square root rounded once to float;
# the clip arithmetic is in float, one IEEE operation at a time.


def shard_sumsq(shard: "Shard") -> float:
    """Squared norm of the scaled gradient of the shard (before any
    all-reduce across ranks)."""
    per_group = [0.0] * len(shard.groups)
    for t in shard.tensors:
        per_group[t.group] += sumsq(t.g, t.g_dtype)
    total = 0.0
    for grp, s in zip(shard.groups, per_group):
        gs = float(np.float32(grp.grad_scale))
        total += gs * gs * s
    return total


def clip_from_sumsq(total_sumsq: float, max_norm: float, grad_scale: float):
    """(norm, found_inf, clip coefficient, new grad scale) from the squared
    norm summed over all ranks; max_norm <= 0 means no clipping."""
    import math
    with np.errstate(over="ignore", invalid="ignore"):
        norm = np.float32(math.sqrt(total_sumsq))  # inf and NaN propagate
        found_inf = not np.isfinite(norm)
        if max_norm <= 0:
            return norm, found_inf, np.float32(1.0), np.float32(grad_scale)
        coef = np.float32(max_norm) / (norm + np.float32(1e-6))
        coef = min(coef, np.float32(1.0))
        return norm, found_inf, np.float32(coef), np.float32(grad_scale) * np.float32(coef)


# ---- the data-parallel exchange around the step (one-GPU stand-in) ------------
#
# "apex/contrib/optimizers/distributed_fused_adam.py": _start_bucket_grad_sync
# (each rank's gradient bucket is reduce-scattered into this rank's shard
# buffer, which has the grad sync dtype; ReduceOp.AVG when average_grad_sync,
# SUM otherwise), _finish_bucket_grad_sync (the synced shard becomes the
# gradient shard the local step reads) and _start_bucket_param_sync (every
# rank's param shard is all-gathered into each rank's param bucket).
# Readings: this rank's shard receives, element by element, the R ranks'
# values widened to float and added in rank order 0, 1, ..., R-1, one IEEE
# float addition at a time; the average divides that sum by R (one IEEE float
# division); the result is rounded once to the grad dtype (nearest-even),
# which is what the shard buffer holds.  The exchange runs whether or not the
# step is then skipped.  The all-gather puts this rank's param-out shard,
# byte for byte, at this rank's place in every rank's param bucket.

def _widen(x, dtype) -> np.ndarray:
    if dtype == DT_F32:
        return np.asarray(x, dtype=np.float32)
    return bf16_to_f32(x) if dtype == DT_BF16 else f16_to_f32(x)


def _narrow(x, dtype) -> np.ndarray:
    if dtype == DT_F32:
        return np.asarray(x, dtype=np.float32).copy()
    return f32_to_bf16(x) if dtype == DT_BF16 else f32_to_f16(x)


def reduce_sources(sources, g_dtype: int, average: bool) -> np.ndarray:
    """This rank's gradient shard from the R ranks' contributions to it
    (``sources[r]``: rank r's values for this shard, in the grad dtype)."""
    if len(sources) < 1:
        raise ValueError("at least one source")
    with np.errstate(over="ignore", invalid="ignore"):
        acc = _widen(sources[0], g_dtype).copy()
        for s in sources[1:]:
            acc = acc + _widen(s, g_dtype)  # float32 + float32: one IEEE addition
        if average:
            acc = acc / np.float32(len(sources))
    return _narrow(acc, g_dtype)


def accumulate_grad(g_shard, synced, g_dtype: int) -> np.ndarray:
    """Gradient accumulation across reduce-scatters (_finish_bucket_grad_sync:
    after the first, each synced shard is added to the gradient shard with
    ``grads_shard.add_(sync_grads_shard)``).  Reading: both are in the grad
    dtype; the sum is taken in float (one IEEE addition of the widened
    values) and rounded once to the grad dtype."""
    with np.errstate(over="ignore", invalid="ignore"):
        acc = _widen(g_shard, g_dtype) + _widen(synced, g_dtype)
    return _narrow(acc, g_dtype)


def reduce_into(g_shard, sources, g_dtype: int, average: bool, accumulate: bool) -> np.ndarray:
    """This rank's gradient shard after one reduce-scatter: the reduced
    contributions, or (accumulating) the old shard plus them."""
    synced = reduce_sources(sources, g_dtype, average)
    return accumulate_grad(g_shard, synced, g_dtype) if accumulate else synced


def exchange_step(shard: Shard, sources, *, average: bool, capturable: bool,
                  noop: bool = False, check_finite: bool = False,
                  step_preadvanced: bool = False, accumulate: bool = False) -> bool:
    """Reduce-scatter stand-in, then the shard step.  ``sources[i]`` lists the
    R contributions for tensor i; each tensor's ``g`` becomes the reduced
    shard, or with ``accumulate`` its old value plus the reduced shard (the
    exchange happens even if the step is then skipped).  Returns the noop
    flag after the step; the all-gather side is ``gather_param_out``."""
    for t, src in zip(shard.tensors, sources):
        t.g[...] = reduce_into(t.g, src, t.g_dtype, average, accumulate)
    return shard_step(shard, capturable=capturable, noop=noop, check_finite=check_finite,
                      step_preadvanced=step_preadvanced)


def gather_param_out(p_out_shard, n_ranks: int, rank: int) -> np.ndarray:
    """Every rank's bucket receives this rank's param-out shard at offset
    rank * shard size; returns what this rank contributes to one bucket of
    R shards (other ranks' places left zero)."""
    shard = np.asarray(p_out_shard)
    out = np.zeros(shard.size * n_ranks, dtype=shard.dtype)
    out[rank * shard.size:(rank + 1) * shard.size] = shard
    return out


# ---- scaled optimizer state -----------------------------------------------------
#
# "apex/contrib/optimizers/distributed_fused_adam.py": _local_step_with_scaled_states
# (per fragment: the fp16/bf16 param, exp_avg and exp_avg_sq are copied to
# fp32 and multiplied by their scales, the Adam step runs on the fp32
# buffers with the param buffer as its own param-out, the param-out of the
# param sync dtype is the cast of the new fp32 param, then every buffer is
# rescaled and copied back) and _apply_state_scale (absmax = max(-min, max)
# of the buffer; scale = absmax / (finfo(dtype).max / 2); rscale = 1 / scale
# where scale > 0, else 0; buffer *= rscale).  Readings: every product,
# quotient and reciprocal is one IEEE float operation; absmax is the largest
# magnitude as a float (+0 when every value is a zero of either sign; NaN
# when any value is NaN, as aminmax propagates it); the copies to the state
# dtype round to nearest even; empty tensors are skipped (the page skips
# fragments with no local elements).

def max_scaled_state(state_dtype: int) -> np.float32:
    """finfo(dtype).max / 2 for the 16-bit state dtype, as a float."""
    if state_dtype == DT_BF16:
        return np.float32(bf16_to_f32(np.array([0x7F7F], np.uint16))[0]) / np.float32(2)
    if state_dtype == DT_F16:
        return np.float32(65504.0) / np.float32(2)
    raise ValueError("scaled states need a 16-bit state dtype")


def state_scale(buf, state_dtype: int):
    """(scale, rscale) of an fp32 buffer, as _apply_state_scale computes them."""
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        a = np.abs(np.asarray(buf, np.float32))
        absmax = np.float32(np.max(a)) if a.size else np.float32(0)  # NaN propagates
        scale = absmax / max_scaled_state(state_dtype)
        rscale = np.float32(1) / scale if scale > 0 else np.float32(0)
    return np.float32(scale), np.float32(rscale)


def adam_scaled(group: Group, step: int, p16, m16, v16, scales, state_dtype: int, g,
                g_dtype=DT_F32, p_out=None, out_dtype=DT_NONE) -> None:
    """One step of a tensor in scaled 16-bit state.  ``p16, m16, v16``: uint16
    bits of the state dtype, updated in place; ``scales``: float32[3] (param,
    exp_avg, exp_avg_sq), updated in place."""
    if np.asarray(p16).size == 0:
        return
    with np.errstate(invalid="ignore", over="ignore"):
        bufs = [_widen(x, state_dtype) * np.float32(s) for x, s in zip((p16, m16, v16), scales)]
    p, m, v = (np.ascontiguousarray(b, np.float32) for b in bufs)
    adam_f32(group, step, p, m, v, g, g_dtype, p_out, out_dtype)
    for k, (buf, dst) in enumerate(((p, p16), (m, m16), (v, v16))):
        scale, rscale = state_scale(buf, state_dtype)
        with np.errstate(invalid="ignore", over="ignore"):
            dst[...] = _narrow(buf * rscale, state_dtype)
        scales[k] = scale


def scale_state(x, state_dtype: int):
    """A new scaled state from fp32 values (how the page stores the params
    at construction): (16-bit bits, scale)."""
    buf = np.asarray(x, np.float32)
    scale, rscale = state_scale(buf, state_dtype)
    with np.errstate(invalid="ignore", over="ignore"):
        return _narrow(buf * rscale, state_dtype), scale
