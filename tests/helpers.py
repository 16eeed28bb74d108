"""Test helpers: hand the same seeded inputs to the oracle, and compare.

Tolerances (GPU vs oracle):
  fp32 p, m, v:        |d| <= 2e-6 * |x| + 1e-9   (x the oracle value)
  bf16/fp16 param-out, and p, m, v kept in a 16-bit state dtype: at most
                       1 unit in the last place
  noop, step counters, remainder round trip: bit-exact
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np
import torch

import oracle
import workloads

RTOL, ATOL = 2e-6, 1e-9

_ODT = {torch.float32: oracle.DT_F32, torch.bfloat16: oracle.DT_BF16, torch.float16: oracle.DT_F16}


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.int16:
        return t.numpy().copy()
    raise TypeError(t.dtype)


def oracle_groups(spec: workloads.ShardSpec) -> List[oracle.Group]:
    out = []
    for g in spec.groups:
        out.append(oracle.Group(mode=oracle.MODE_ADAMW if g.adam_w_mode else oracle.MODE_L2,
                                bias_correction=1 if g.bias_correction else 0,
                                beta1=g.betas[0], beta2=g.betas[1], eps=g.eps,
                                weight_decay=g.weight_decay, lr=g.lr,
                                grad_scale=spec.grad_scale))
    return out


def _selector(elems, i: int, device):
    """Element selection of tensor i: everything, a contiguous range (a
    slice) or gathered indices."""
    if elems is None:
        return lambda t: t
    e = elems[i]
    if isinstance(e, slice):
        return lambda t: t[e]
    e = torch.as_tensor(e, device=device)
    return lambda t: t[e]


def oracle_shard(shard: workloads.Shard, idx: List[int] = None, elems: Dict[int, np.ndarray] = None,
                 step_slot=None, scales: torch.Tensor = None) -> oracle.Shard:
    """Snapshot of the shard (or of sampled elements of it) as oracle arrays.

    `idx` is the tensor order; `elems[i]`, when given, selects elements of
    tensor i, as an index array or a slice (the oracle then runs on the
    selected elements only, which is exact because every element updates
    independently).
    """
    spec = shard.spec
    idx = shard.plan_order() if idx is None else idx
    g_dt = _ODT[spec.g_dtype]
    tensors = []
    for i in idx:
        sel = _selector(elems, i, shard.params[i].device)
        t = oracle.Tensor(group=spec.group_of[i], m=to_np(sel(shard.exp_avgs[i])),
                          v=to_np(sel(shard.exp_avg_sqs[i])), g=to_np(sel(shard.grads[i])),
                          g_dtype=g_dt)
        if spec.remainders:
            t.p_hi = to_np(sel(shard.params[i]))
            t.rem = to_np(sel(shard.remainders[i]))
            t.p_out = t.p_hi  # the new high half replaces the param in place
            t.out_dtype = oracle.DT_BF16
        else:
            t.p = to_np(sel(shard.params[i]))
            t.state_dtype = _ODT[spec.state_dtype]
            if spec.moment_dtype is not None:
                t.moment_dtype = _ODT[spec.moment_dtype]
            if scales is not None:  # [n, 3] in the order of idx
                t.scales = to_np(scales[len(tensors)]).copy()
            if spec.out_dtype is not None:
                t.p_out = to_np(sel(shard.params_out[i]))
                t.out_dtype = _ODT[spec.out_dtype]
        tensors.append(t)
    return oracle.Shard(groups=oracle_groups(spec), tensors=tensors,
                        step_slot=list(step_slot) if step_slot else [])


def refresh_grads(osh: oracle.Shard, shard: workloads.Shard, idx=None, elems=None) -> None:
    idx = shard.plan_order() if idx is None else idx
    for t, i in zip(osh.tensors, idx):
        t.g = to_np(_selector(elems, i, shard.grads[i].device)(shard.grads[i]))


def put(dst: Optional[torch.Tensor], arr: Optional[np.ndarray]) -> None:
    """Write an oracle array (fp32 values, 16-bit bit patterns or int16)
    into a device tensor of the same size."""
    if dst is None or arr is None:
        return
    if dst.dtype == torch.float32:
        dst.copy_(torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)))
    else:
        dst.view(torch.int16).copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)))


def load_oracle_state(shard: workloads.Shard, osh: oracle.Shard, idx=None,
                      scales: torch.Tensor = None) -> None:
    """Make the oracle's current state the GPU shard's (p, m, v, the
    remainders, and the scaled state's scales in the order of idx), so that
    the next step starts both from the same values."""
    idx = shard.plan_order() if idx is None else idx
    for k, (t, i) in enumerate(zip(osh.tensors, idx)):
        put(shard.exp_avgs[i], t.m)
        put(shard.exp_avg_sqs[i], t.v)
        if t.rem is not None:
            put(shard.params[i], t.p_hi)
            put(shard.remainders[i], t.rem)
        else:
            put(shard.params[i], t.p)
        if scales is not None and t.scales is not None:
            scales[k].copy_(torch.from_numpy(np.ascontiguousarray(t.scales, dtype=np.float32)))


def widen16(bits: np.ndarray, dtype) -> np.ndarray:
    """16-bit bit patterns of `dtype` as float64 values."""
    if dtype == torch.bfloat16:
        return oracle.bf16_to_f32(bits).astype(np.float64)
    return oracle.f16_to_f32(bits).astype(np.float64)


def ulp16(values: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the 16-bit dtype at each (finite) value."""
    mant, emin = (7, -133) if dtype == torch.bfloat16 else (10, -24)
    a = np.abs(values)
    _, e = np.frexp(np.where(a > 0, a, 1.0))  # a = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, np.maximum(e - 1 - mant, emin))


def check_recip_p16(got_bits, want_bits, dtype, x_before, what, report,
                    got_scale=1.0, want_scale=1.0):
    """A 16-bit p (or param-out) of a step with reciprocal bias corrections:
    the value (times its scale, for a scaled state) within one ulp of its
    dtype plus 2e-6 * max(|p before the step|, |p'|) + 1e-9.  The
    reciprocal's extra rounding is relative to lr*u <= |p| + |p'|, which can
    exceed |p'| many times where the step nearly cancels p, so a small p'
    may land several of its own ulps away; m and v need no such allowance."""
    g = widen16(got_bits, dtype) * np.float64(got_scale)
    w = widen16(want_bits, dtype) * np.float64(want_scale)
    x = np.abs(np.asarray(x_before, np.float64))
    both_nan = np.isnan(g) & np.isnan(w)
    same = (g == w) | both_nan
    # a value that is infinite or NaN on either side must be the same on
    # the other (the bound's terms are infinite there)
    nonfinite = ~np.isfinite(g) | ~np.isfinite(w)
    with np.errstate(invalid="ignore", over="ignore"):
        lim = (ulp16(widen16(want_bits, dtype), dtype) * abs(np.float64(want_scale))
               + 2e-6 * np.maximum(x, np.abs(w)) + 1e-9)
        bad = ~same & (nonfinite | ~(np.abs(g - w) <= lim))
    if bad.any():
        k = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {g.size} outside the bound; first at "
                             f"{k}: got {g[k]!r} want {w[k]!r} p before {x[k]!r}")
    report.n += g.size
    report.exact += int(np.sum(np.asarray(got_bits) == np.asarray(want_bits)))


def compare_recip(shard: workloads.Shard, osh: oracle.Shard, x_before, report: Report,
                  idx=None, elems=None, got_scales: np.ndarray = None) -> Report:
    """GPU vs oracle after one step of a 16-bit state with reciprocal bias
    corrections (FADAM_RECIP_BC): m and v within one ulp of their dtype, p
    and a 16-bit param-out under check_recip_p16, an fp32 param-out within
    2e-6 * max(|p before|, |p'|) + 1e-9.  x_before[k]: tensor k's fp32
    master before the step (for a scaled state, unscaled); got_scales[k]:
    the GPU's new scales of tensor k (scaled state)."""
    spec = shard.spec
    sdt = spec.state_dtype
    idx = shard.plan_order() if idx is None else idx
    for k, (t, i, x0) in enumerate(zip(osh.tensors, idx, x_before)):
        sel = _selector(elems, i, shard.params[i].device)
        report.ulp16(to_np(sel(shard.exp_avgs[i])), t.m, f"tensor {i} m", sdt)
        report.ulp16(to_np(sel(shard.exp_avg_sqs[i])), t.v, f"tensor {i} v", sdt)
        gs = 1.0 if got_scales is None else got_scales[k][0]
        ws = 1.0 if t.scales is None else t.scales[0]
        check_recip_p16(to_np(sel(shard.params[i])), t.p, sdt, x0, f"tensor {i} p", report, gs, ws)
        if spec.out_dtype == torch.float32:
            got = to_np(sel(shard.params_out[i])).astype(np.float64)
            want = t.p_out.astype(np.float64)
            lim = 2e-6 * np.maximum(np.abs(want), np.abs(np.asarray(x0, np.float64))) + 1e-9
            nonfinite = ~np.isfinite(got) | ~np.isfinite(want)  # must be the same there
            with np.errstate(invalid="ignore"):
                bad = ((nonfinite | ~(np.abs(got - want) <= lim))
                       & ~(np.isnan(got) & np.isnan(want)) & (got != want))
            assert not bad.any(), f"tensor {i} p_out: {int(bad.sum())} outside; first at {int(np.argmax(bad))}"
            report.n += got.size
            report.exact += int(np.sum(got == want))
        elif spec.out_dtype is not None:
            check_recip_p16(to_np(sel(shard.params_out[i])), t.p_out, spec.out_dtype, x0,
                            f"tensor {i} p_out", report)
    return report


def unscaled_p(osh: oracle.Shard, state_dtype) -> List[np.ndarray]:
    """Each oracle tensor's master p as float64 values (times its p scale for
    a scaled state): the state a step starts from."""
    out = []
    for t in osh.tensors:
        x = widen16(t.p, state_dtype)
        if t.scales is not None:
            x = x * np.float64(t.scales[0])
        out.append(x)
    return out


def _ordered16(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def _is_inf_or_nan16(bits: np.ndarray, dtype) -> np.ndarray:
    b = bits.astype(np.int32)
    e = 0x7F80 if dtype == torch.bfloat16 else 0x7C00
    return (b & e) == e


def _is_nan16(bits: np.ndarray, dtype) -> np.ndarray:
    b = bits.astype(np.int32)
    if dtype == torch.bfloat16:
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return ((b & 0x7C00) == 0x7C00) & ((b & 0x3FF) != 0)


class Report:
    """Collects the worst deviations and the share of bit-identical values."""

    def __init__(self):
        self.n = 0
        self.exact = 0
        self.worst = 0.0

    def _same_bytes(self, got: np.ndarray, want: np.ndarray) -> bool:
        """Equal bit patterns (the common case): counted as exact, with no
        need for the tolerance arithmetic."""
        if got.shape != want.shape or got.dtype.itemsize != want.dtype.itemsize:
            return False
        u = {2: np.uint16, 4: np.uint32}.get(got.dtype.itemsize)
        if u is None or not np.array_equal(np.ascontiguousarray(got).view(u),
                                           np.ascontiguousarray(want).view(u)):
            return False
        self.n += got.size
        self.exact += got.size
        return True

    def merge(self, other: "Report") -> None:
        self.n += other.n
        self.exact += other.exact
        self.worst = max(self.worst, other.worst)

    def f32(self, got: np.ndarray, want: np.ndarray, what: str) -> None:
        if self._same_bytes(got, want):
            return
        got = got.astype(np.float64)
        want = want.astype(np.float64)
        both_nan = np.isnan(got) & np.isnan(want)
        same = (got == want) | both_nan  # equal infinities included
        with np.errstate(invalid="ignore"):
            d = np.where(same, 0.0, np.abs(got - want))
            # a non-finite expected value must be matched exactly
            lim = np.where(same | ~np.isfinite(want), 0.0, RTOL * np.abs(want) + ATOL)
        bad = ~(d <= lim)
        if bad.any():
            k = int(np.argmax(bad))
            raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} outside tolerance; "
                                 f"first at {k}: got {got[k]!r} want {want[k]!r}")
        self.n += got.size
        self.exact += int(np.sum((got == want) | both_nan))
        with np.errstate(invalid="ignore", divide="ignore"):
            rel = np.where(d > 0, d / np.maximum(lim, 1e-300), 0.0)
        if rel.size:
            self.worst = max(self.worst, float(rel.max()))

    def ulp16(self, got: np.ndarray, want: np.ndarray, what: str, dtype=None) -> None:
        if self._same_bytes(got, want):
            return
        d = np.abs(_ordered16(got) - _ordered16(want))
        if dtype is not None:
            # an infinity sits one step from the largest finite value in this
            # order: a value that is infinite or NaN on either side must be
            # the same on the other; two NaNs match whatever their payloads
            both_nan = _is_nan16(got, dtype) & _is_nan16(want, dtype)
            nonfinite = _is_inf_or_nan16(got, dtype) | _is_inf_or_nan16(want, dtype)
            d = np.where(nonfinite & (np.asarray(got) != np.asarray(want)), 1 << 20, d)
            d = np.where(both_nan, 0, d)
        if (d > 1).any():
            k = int(np.argmax(d > 1))
            raise AssertionError(f"{what}: {int((d > 1).sum())} values beyond 1 ulp; first at "
                                 f"{k}: got 0x{int(got[k]):04X} want 0x{int(want[k]):04X}")
        self.n += got.size
        self.exact += int(np.sum(d == 0))

    @property
    def exact_fraction(self) -> float:
        return self.exact / max(1, self.n)


def compare(shard: workloads.Shard, osh: oracle.Shard, idx=None, elems=None,
            report: Report = None) -> Report:
    """GPU shard vs oracle shard, element by element (or on the samples)."""
    report = report or Report()
    spec = shard.spec
    idx = shard.plan_order() if idx is None else idx
    state16 = not spec.remainders and spec.state_dtype != torch.float32
    for t, i in zip(osh.tensors, idx):
        sel = _selector(elems, i, shard.params[i].device)
        if state16:  # 16-bit p, m, v: within one unit in the last place
            sdt = spec.state_dtype
            report.ulp16(to_np(sel(shard.exp_avgs[i])), t.m, f"tensor {i} m", sdt)
            report.ulp16(to_np(sel(shard.exp_avg_sqs[i])), t.v, f"tensor {i} v", sdt)
            report.ulp16(to_np(sel(shard.params[i])), t.p, f"tensor {i} p", sdt)
            if spec.out_dtype == torch.float32:
                report.f32(to_np(sel(shard.params_out[i])), t.p_out, f"tensor {i} p_out")
            elif spec.out_dtype is not None:
                report.ulp16(to_np(sel(shard.params_out[i])), t.p_out, f"tensor {i} p_out",
                             spec.out_dtype)
            continue
        if spec.moment_dtype is not None:  # 16-bit moments under an fp32 master
            mdt = spec.moment_dtype
            report.ulp16(to_np(sel(shard.exp_avgs[i])), t.m, f"tensor {i} m", mdt)
            report.ulp16(to_np(sel(shard.exp_avg_sqs[i])), t.v, f"tensor {i} v", mdt)
        else:
            report.f32(to_np(sel(shard.exp_avgs[i])), t.m, f"tensor {i} m")
            report.f32(to_np(sel(shard.exp_avg_sqs[i])), t.v, f"tensor {i} v")
        if spec.remainders:
            hi = to_np(sel(shard.params[i]))
            rem = to_np(sel(shard.remainders[i]))
            got = oracle.rem_pack(hi, rem).view(np.float32)
            want = oracle.rem_pack(t.p_hi, t.rem).view(np.float32)
            report.f32(got, want, f"tensor {i} fp32 master (bf16 + remainder)")
            # a NaN master has no one encoding: its payload depends on where
            # the NaN arose, and the split maps payloads to different (high
            # half, remainder) pairs that all pack back to a NaN, which the
            # master comparison above checks; the halves are compared
            # wherever the master is a number
            both_nan = np.isnan(got) & np.isnan(want)
            report.ulp16(np.where(both_nan, t.p_hi, hi), t.p_hi, f"tensor {i} bf16 high half",
                         torch.bfloat16)
        else:
            report.f32(to_np(sel(shard.params[i])), t.p, f"tensor {i} p")
            if spec.out_dtype == torch.float32:
                report.f32(to_np(sel(shard.params_out[i])), t.p_out, f"tensor {i} p_out")
            elif spec.out_dtype is not None:
                report.ulp16(to_np(sel(shard.params_out[i])), t.p_out, f"tensor {i} p_out",
                             spec.out_dtype)
    return report


def sample_elements(spec: workloads.ShardSpec, per_tensor: int, seed: int) -> Dict[int, np.ndarray]:
    """Seeded element samples per tensor (every element of small tensors),
    always including each tensor's first and last element."""
    rng = np.random.default_rng(seed)
    out = {}
    for i, n in enumerate(spec.sizes):
        if n <= per_tensor:
            out[i] = np.arange(n, dtype=np.int64)
        else:
            e = rng.choice(n, size=per_tensor - 2, replace=False)
            out[i] = np.unique(np.concatenate([e, [0, n - 1]])).astype(np.int64)
    return out


def snapshot(shard: workloads.Shard) -> List[torch.Tensor]:
    """Clones of every state tensor of the shard (on its device)."""
    ts = []
    for lst in (shard.params, shard.exp_avgs, shard.exp_avg_sqs, shard.params_out,
                shard.remainders):
        for t in lst:
            if t is not None:
                ts.append(t.clone())
    return ts


def state_equal(shard: workloads.Shard, snap: List[torch.Tensor]) -> bool:
    k = 0
    for lst in (shard.params, shard.exp_avgs, shard.exp_avg_sqs, shard.params_out,
                shard.remainders):
        for t in lst:
            if t is not None:
                a = t.view(torch.int16) if t.dtype != torch.int16 and t.element_size() == 2 else t
                b = snap[k].view(torch.int16) if snap[k].element_size() == 2 and snap[k].dtype != torch.int16 else snap[k]
                if t.dtype == torch.float32:
                    a, b = t.view(torch.int32), snap[k].view(torch.int32)
                if not torch.equal(a, b):
                    return False
                k += 1
    return True
