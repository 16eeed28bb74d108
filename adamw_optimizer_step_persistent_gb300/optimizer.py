"""Python face of the library: a shard optimizer over the C ABI.

``FusedAdamShard`` holds one data-parallel rank's optimizer shard as lists
of tensors per param group (the lists p, m, v, g, p_out of
distributed_fused_adam.py's ``_local_step``), builds one plan for all of
them and runs each step as a single persistent-grid launch.  It only
marshals pointers and scalars; PyTorch supplies device memory and streams.

Step counters ("[PyTorch] Advance FusedAdam step counter for empty param
groups"): every group, empty or not, has one and it advances every applied
step.  Regular shards keep them on the host and advance them before the
launch, as ``step()`` of distributed_fused_adam.py does; capturable shards
keep int32 device counters that the kernel advances by (noop != 1), so a
captured step replays correctly.
"""
from __future__ import annotations

import ctypes
from typing import Dict, List, Optional, Sequence

import torch

from . import _abi

_DT = {torch.float32: _abi.DT_F32, torch.bfloat16: _abi.DT_BF16, torch.float16: _abi.DT_F16}


def dtype_code(dt: Optional[torch.dtype]) -> int:
    if dt is None:
        return _abi.DT_NONE
    if dt not in _DT:
        raise TypeError(f"unsupported dtype {dt}")
    return _DT[dt]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class FusedAdamShard:
    """Fused Adam/AdamW over one shard: one kernel launch per step.

    ``param_groups`` is a list of dicts with keys
      params, exp_avgs, exp_avg_sqs, grads      lists of equal length
      params_out (optional), remainders (remainder mode only)
      lr, betas, eps, weight_decay, bias_correction, adam_w_mode
    A group with empty lists is allowed; its step counter still advances.
    ``params`` are the masters and set the state dtype: fp32, bf16 or fp16,
    with ``exp_avgs`` and ``exp_avg_sqs`` of the same dtype (updated in
    float, rounded back on store), or, under an fp32 master, both bf16 or
    both fp16 (TransformerEngine's exp_avg_dtype and exp_avg_sq_dtype).  In
    remainder mode ``params`` are the bf16 high halves (``remainders`` then
    holds the int16 low halves, the moments are fp32, and ``params_out`` the
    bf16 tensors that receive the new high halves; they may be ``params``).
    ``recip_bc`` (16-bit state only) multiplies the moments by reciprocal
    bias corrections instead of dividing them (FADAM_RECIP_BC): faster for
    those issue-bound forms, within a derived bound rather than bit-identical.
    """

    def __init__(self, param_groups: Sequence[Dict], *, capturable: bool = False,
                 check_finite: bool = False, remainders: bool = False,
                 shared_step: bool = False, step_preadvanced: bool = False,
                 grad_scale: float = 1.0, device=None, extra_flags: int = 0,
                 state_scales: Optional[torch.Tensor] = None, recip_bc: bool = False):
        if check_finite and not capturable:
            raise ValueError("check_finite needs capturable=True (the counters live on the device)")
        self.capturable = capturable
        self.device = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        self.groups = [dict(g) for g in param_groups]
        if not 1 <= len(self.groups) <= _abi.MAX_GROUPS:
            raise ValueError(f"1..{_abi.MAX_GROUPS} param groups supported")
        self._keep: List[torch.Tensor] = []  # tensors the plan points into
        flags = (_abi.CAPTURABLE if capturable else 0) | (_abi.REMAINDERS if remainders else 0)
        flags |= (_abi.CHECK_FINITE if check_finite else 0)
        flags |= (_abi.STEP_PREADVANCED if step_preadvanced else 0)
        flags |= (_abi.SCALED_STATES if state_scales is not None else 0)
        flags |= (_abi.RECIP_BC if recip_bc else 0)
        flags |= int(extra_flags)
        self.flags = flags

        descs = []
        g_dtype = out_dtype = None
        p_dtype = torch.bfloat16 if remainders else None
        mv_dtype = None
        for gi, g in enumerate(self.groups):
            ps, ms, vs, gs = g["params"], g["exp_avgs"], g["exp_avg_sqs"], g["grads"]
            outs = g.get("params_out") or [None] * len(ps)
            rems = g.get("remainders") or [None] * len(ps)
            if not (len(ps) == len(ms) == len(vs) == len(gs) == len(outs) == len(rems)):
                raise ValueError(f"group {gi}: tensor lists differ in length")
            for p, m, v, gr, o, r in zip(ps, ms, vs, gs, outs, rems):
                for t in (p, m, v, gr, o, r):
                    if t is not None and (not t.is_contiguous() or t.device != self.device):
                        raise ValueError("tensors must be contiguous and on the shard's device")
                p_dtype = p_dtype or p.dtype
                # m and v: the state dtype, fp32 in remainder mode, or one
                # 16-bit dtype under an fp32 master (exp_avg_dtype =
                # exp_avg_sq_dtype)
                if mv_dtype is None:
                    mv_dtype = torch.float32 if remainders else (
                        m.dtype if p_dtype == torch.float32 else p_dtype)
                if p.dtype != p_dtype or m.dtype != mv_dtype or v.dtype != mv_dtype:
                    raise TypeError(f"group {gi}: p must be {p_dtype}, m and v {mv_dtype}")
                g_dtype = g_dtype or gr.dtype
                if gr.dtype != g_dtype:
                    raise TypeError("every grad must have the same dtype")
                if o is not None:
                    out_dtype = out_dtype or o.dtype
                    if o.dtype != out_dtype:
                        raise TypeError("every param-out tensor must have the same dtype")
                if not (p.numel() == m.numel() == v.numel() == gr.numel()):
                    raise ValueError("p, m, v, g sizes differ")
                descs.append(_abi.Tensor(p=_ptr(p), m=_ptr(m), v=_ptr(v), g=_ptr(gr),
                                         p_out=_ptr(o), rem=_ptr(r), numel=p.numel(), group=gi))
                self._keep += [t for t in (p, m, v, gr, o, r) if t is not None]
        self.n_tensors = len(descs)
        p_dtype = p_dtype or torch.float32
        self.state_dtype = p_dtype
        self.moment_dtype = None
        if not remainders and p_dtype == torch.float32 and mv_dtype not in (None, torch.float32):
            if mv_dtype not in (torch.bfloat16, torch.float16):
                raise TypeError(f"moments of dtype {mv_dtype} under an fp32 master")
            self.moment_dtype = mv_dtype
            flags |= _abi.MOMENTS_BF16 if mv_dtype == torch.bfloat16 else _abi.MOMENTS_F16
            self.flags = flags
        self.g_dtype = g_dtype or torch.float32
        self.out_dtype = out_dtype

        n = len(self.groups)
        self.host_steps = [0] * n
        self.host_lr = [float(g.get("lr", 1e-3)) for g in self.groups]
        self.host_grad_scale = float(grad_scale)
        if capturable:
            dev = self.device
            self.lr_dev = [torch.tensor([lr], dtype=torch.float32, device=dev) for lr in self.host_lr]
            self.grad_scale_dev = torch.tensor([grad_scale], dtype=torch.float32, device=dev)
            if shared_step:
                one = torch.zeros(1, dtype=torch.int32, device=dev)
                self.step_dev = [one] * n
            else:
                self.step_dev = [torch.zeros(1, dtype=torch.int32, device=dev) for _ in range(n)]
            self.noop = torch.zeros(1, dtype=torch.int32, device=dev)
        self._groups_c = (_abi.Group * n)()
        self._fill_groups()

        arr = (_abi.Tensor * max(1, len(descs)))(*descs)
        plan = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _abi.check(_abi.lib().fadam_plan_create(
                arr, len(descs), self._groups_c, n, dtype_code(p_dtype), dtype_code(self.g_dtype),
                dtype_code(out_dtype), flags, ctypes.byref(plan)), "fadam_plan_create")
        self._plan = plan
        self.state_scales = None
        if state_scales is not None:
            # scaled 16-bit state: one fp32 scale per tensor for p, m and v,
            # in the order the tensors were given ([n_tensors, 3])
            if (state_scales.dtype != torch.float32 or state_scales.device != self.device
                    or not state_scales.is_contiguous()
                    or tuple(state_scales.shape) != (self.n_tensors, 3)):
                raise ValueError("state_scales must be a contiguous fp32 [n_tensors, 3] "
                                 "tensor on the shard's device")
            _abi.check(_abi.lib().fadam_plan_set_state_scales(self._plan, state_scales.data_ptr()),
                       "fadam_plan_set_state_scales")
            self.state_scales = state_scales

    # ---- scalars ---------------------------------------------------------------

    def _fill_groups(self) -> None:
        for i, g in enumerate(self.groups):
            b1, b2 = g.get("betas", (0.9, 0.999))
            c = self._groups_c[i]
            c.mode = _abi.MODE_ADAMW if g.get("adam_w_mode", True) else _abi.MODE_L2
            c.bias_correction = 1 if g.get("bias_correction", True) else 0
            c.beta1, c.beta2 = float(b1), float(b2)
            c.eps = float(g.get("eps", 1e-8))
            c.weight_decay = float(g.get("weight_decay", 0.0))
            c.lr = self.host_lr[i]
            c.grad_scale = self.host_grad_scale
            c.step = self.host_steps[i]
            if self.capturable:
                c.lr_dev = self.lr_dev[i].data_ptr()
                c.grad_scale_dev = self.grad_scale_dev.data_ptr()
                c.step_dev = self.step_dev[i].data_ptr()

    def set_lr(self, group: int, lr: float) -> None:
        """New learning rate for a group (a device write when capturable)."""
        self.host_lr[group] = float(lr)
        if self.capturable:
            self.lr_dev[group].fill_(float(lr))

    def set_grad_scale(self, scale: float) -> None:
        self.host_grad_scale = float(scale)
        if self.capturable:
            self.grad_scale_dev.fill_(float(scale))

    # ---- stepping ----------------------------------------------------------------

    def step(self, found_inf: bool = False) -> None:
        """One optimizer step on the current stream.

        Regular shards: ``found_inf`` (a host bool, as the page's regular
        path reads it) skips the step entirely; otherwise every group's
        counter advances and one launch runs.  Capturable shards: one launch
        that honours ``self.noop`` on the device; nothing here syncs, so the
        call can be captured in a CUDA graph.
        """
        lib = _abi.lib()
        if self.capturable:
            _abi.check(lib.fadam_step(self._plan, self.noop.data_ptr(),
                                      _stream_handle(self.device)), "fadam_step")
            return
        if found_inf:
            return
        self.host_steps = [s + 1 for s in self.host_steps]
        self._fill_groups()
        _abi.check(lib.fadam_plan_set_groups(self._plan, self._groups_c, len(self.groups)),
                   "fadam_plan_set_groups")
        _abi.check(lib.fadam_step(self._plan, None, _stream_handle(self.device)), "fadam_step")

    def step_from_host(self, grads_host: Sequence[torch.Tensor]) -> List[int]:
        """Copy host gradients (one per tensor, plan order) in, step, and
        return the group step counters; waits for the stream."""
        lib = _abi.lib()
        if len(grads_host) != self.n_tensors:
            raise ValueError("one host gradient per tensor")
        ptrs = (ctypes.c_void_p * max(1, self.n_tensors))(*[g.data_ptr() for g in grads_host])
        steps = (ctypes.c_int32 * len(self.groups))()
        if not self.capturable:
            self.host_steps = [s + 1 for s in self.host_steps]
            self._fill_groups()
            _abi.check(lib.fadam_plan_set_groups(self._plan, self._groups_c, len(self.groups)),
                       "fadam_plan_set_groups")
        noop = self.noop.data_ptr() if self.capturable else None
        _abi.check(lib.fadam_step_host_grads(self._plan, ptrs, noop, steps,
                                             _stream_handle(self.device)), "fadam_step_host_grads")
        return list(steps)

    # ---- gradient norm and clipping ------------------------------------------

    def grad_norm_sq(self) -> torch.Tensor:
        """Squared L2 norm of this shard's scaled gradient, as a float64
        device tensor (all-reduce it across data-parallel ranks before
        clip_apply).  One launch, no sync."""
        if not hasattr(self, "_sumsq"):
            self._sumsq = torch.zeros(1, dtype=torch.float64, device=self.device)
        if not self.capturable:  # the plan reads the current host grad_scale
            self._fill_groups()
            _abi.check(_abi.lib().fadam_plan_set_groups(self._plan, self._groups_c,
                                                        len(self.groups)), "fadam_plan_set_groups")
        _abi.check(_abi.lib().fadam_grad_sumsq(self._plan, self._sumsq.data_ptr(),
                                               _stream_handle(self.device)), "fadam_grad_sumsq")
        return self._sumsq

    def clip_apply(self, sumsq: torch.Tensor, max_norm: float) -> torch.Tensor:
        """Norm from the (all-reduced) squared norm; found_inf into the noop
        flag; the clip coefficient multiplied into the grad scale by the
        same launch: on the device for capturable shards, and for regular
        shards into a device copy of each group's host grad scale, which is
        read back (one sync, as the page's .item() path).  Returns the norm
        as a float32 device tensor."""
        if not hasattr(self, "_norm"):
            self._norm = torch.zeros(1, dtype=torch.float32, device=self.device)
            self._scales_out = torch.zeros(len(self.groups), dtype=torch.float32,
                                           device=self.device)
        noop = self.noop.data_ptr() if self.capturable else None
        scales_out = None
        if not self.capturable:
            self._fill_groups()  # the plan scales the current host grad scale
            _abi.check(_abi.lib().fadam_plan_set_groups(self._plan, self._groups_c,
                                                        len(self.groups)), "fadam_plan_set_groups")
            scales_out = self._scales_out.data_ptr()
        _abi.check(_abi.lib().fadam_clip_apply(self._plan, sumsq.data_ptr(), float(max_norm),
                                               self._norm.data_ptr(), noop, scales_out,
                                               _stream_handle(self.device)), "fadam_clip_apply")
        if not self.capturable:
            # every group shares the binding's one host grad scale
            self.host_grad_scale = float(self._scales_out[0].item())
        return self._norm

    def clip_grad_norm(self, max_norm: float) -> torch.Tensor:
        """Single-rank clip: grad_norm_sq then clip_apply."""
        return self.clip_apply(self.grad_norm_sq(), max_norm)

    # ---- the data-parallel exchange (one-GPU stand-in) ----------------------------

    def set_exchange(self, g_shard: torch.Tensor, sources: Sequence[torch.Tensor], *,
                     average: bool = True, out_shard: Optional[torch.Tensor] = None,
                     dests: Sequence[torch.Tensor] = (), accumulate: bool = False) -> None:
        """Register the reduce-scatter sources and the param all-gather
        destinations (fadam_plan_set_exchange).  Every tensor's gradient is
        a view of ``g_shard`` and each source is laid out like it (same
        dtype, at least as many elements); every param-out copy is a view of
        ``out_shard`` and each destination is laid out like it.
        ``accumulate``: each reduction adds to the shard's gradient instead
        of replacing it (gradient accumulation: the second and later
        reduce-scatters of a step; see ``set_accumulate``)."""
        for s in sources:
            if s.dtype != g_shard.dtype or s.numel() < g_shard.numel() or s.device != g_shard.device:
                raise ValueError("each source needs g_shard's dtype, device and at least its size")
        if dests and out_shard is None:
            raise ValueError("destinations need out_shard")
        for d in dests:
            if d.dtype != out_shard.dtype or d.numel() < out_shard.numel() or d.device != out_shard.device:
                raise ValueError("each destination needs out_shard's dtype, device and at least its size")
        src = (ctypes.c_void_p * max(1, len(sources)))(*[s.data_ptr() for s in sources])
        dst = (ctypes.c_void_p * max(1, len(dests)))(*[d.data_ptr() for d in dests])
        flags = ((_abi.EXCHANGE_AVERAGE if average else 0)
                 | (_abi.EXCHANGE_ACCUMULATE if accumulate else 0))
        _abi.check(_abi.lib().fadam_plan_set_exchange(
            self._plan, g_shard.data_ptr() if sources else None, src, len(sources), flags,
            out_shard.data_ptr() if dests else None, dst, len(dests)), "fadam_plan_set_exchange")
        # the plan holds raw pointers: keep the buffers alive with it
        self._exchange = (g_shard, list(sources), out_shard, list(dests), bool(average))

    def set_accumulate(self, accumulate: bool) -> None:
        """Switch gradient accumulation of the registered exchange on (the
        second and later reduce-scatters of a step) or off (a step's first).
        Host only: may be called between captured launches."""
        g_shard, sources, out_shard, dests, average = self._exchange
        self.set_exchange(g_shard, sources, average=average, out_shard=out_shard, dests=dests,
                          accumulate=accumulate)

    def grad_reduce(self) -> None:
        """The reduce-scatter stand-in alone: every tensor's gradient from the
        sources.  One launch, no sync."""
        _abi.check(_abi.lib().fadam_grad_reduce(self._plan, _stream_handle(self.device)),
                   "fadam_grad_reduce")

    def step_reduce(self, found_inf: bool = False) -> None:
        """The reduce-scatter stand-in fused with the step (one launch).  The
        gradient shard is written even when the step is skipped: regular
        shards with ``found_inf`` run the reduction alone."""
        lib = _abi.lib()
        if self.capturable:
            _abi.check(lib.fadam_step_reduce(self._plan, self.noop.data_ptr(),
                                             _stream_handle(self.device)), "fadam_step_reduce")
            return
        if found_inf:
            self.grad_reduce()
            return
        self.host_steps = [s + 1 for s in self.host_steps]
        self._fill_groups()
        _abi.check(lib.fadam_plan_set_groups(self._plan, self._groups_c, len(self.groups)),
                   "fadam_plan_set_groups")
        _abi.check(lib.fadam_step_reduce(self._plan, None, _stream_handle(self.device)),
                   "fadam_step_reduce")

    # ---- state -------------------------------------------------------------------

    def set_group_steps(self, steps: Sequence[int]) -> None:
        """Set each group's counter to the steps already taken, as when a
        shard resumes from a checkpoint: the next step of group i is
        ``steps[i] + 1`` (with ``step_preadvanced`` the counter is what the
        next launch uses, as always).  Capturable shards get a device write
        on the current stream; a shared counter takes one value for all
        groups."""
        steps = [int(s) for s in steps]
        if len(steps) != len(self.groups) or any(s < 0 or s >= 2**31 - 1 for s in steps):
            raise ValueError("one step count in [0, 2^31 - 1) per group")
        if self.capturable:
            if len({t.data_ptr() for t in self.step_dev}) == 1 and len(set(steps)) > 1:
                raise ValueError("the groups share one step counter")
            for t, s in zip(self.step_dev, steps):
                t.fill_(s)
        self.host_steps = steps
        self._fill_groups()
        _abi.check(_abi.lib().fadam_plan_set_groups(self._plan, self._groups_c, len(self.groups)),
                   "fadam_plan_set_groups")

    def state_dict(self) -> Dict:
        """The shard's scalar state for a checkpoint: an int step counter for
        every group, empty groups included ("[PyTorch] Advance FusedAdam step
        counter for empty param groups": a checkpoint whose empty group holds
        no step resumes wrongly), each group's learning rate and the grad
        scale.  Reads the device when capturable.  The tensors (p, m, v,
        remainders, state scales) belong to the caller, who saves them."""
        if self.capturable:
            lr = [float(t.item()) for t in self.lr_dev]
            grad_scale = float(self.grad_scale_dev.item())
        else:
            lr, grad_scale = list(self.host_lr), self.host_grad_scale
        return {"step": self.group_steps(), "lr": lr, "grad_scale": grad_scale}

    def load_state_dict(self, state: Dict) -> None:
        """Restore what ``state_dict`` returned (the same number of groups)."""
        steps, lr = list(state["step"]), list(state["lr"])
        if len(steps) != len(self.groups) or len(lr) != len(self.groups):
            raise ValueError("the checkpoint has a different number of param groups")
        if any(s is None for s in steps):
            raise ValueError("the checkpoint lacks the step counter of a group")
        self.set_group_steps(steps)
        for i, x in enumerate(lr):
            self.set_lr(i, x)
        self.set_grad_scale(state["grad_scale"])
        if not self.capturable:
            self._fill_groups()
            _abi.check(_abi.lib().fadam_plan_set_groups(self._plan, self._groups_c,
                                                        len(self.groups)),
                       "fadam_plan_set_groups")

    def group_steps(self) -> List[int]:
        """Each group's step counter (reads the device when capturable)."""
        if self.capturable:
            return [int(s.item()) for s in self.step_dev]
        return list(self.host_steps)

    def info(self) -> Dict[str, float]:
        info = _abi.PlanInfo()
        _abi.check(_abi.lib().fadam_plan_get_info(self._plan, ctypes.byref(info)),
                   "fadam_plan_get_info")
        return {name: getattr(info, name) for name, _ in _abi.PlanInfo._fields_}

    def device_status(self) -> int:
        st = ctypes.c_int32()
        _abi.check(_abi.lib().fadam_plan_status(self._plan, ctypes.byref(st)), "fadam_plan_status")
        return st.value

    def close(self) -> None:
        if getattr(self, "_plan", None):
            _abi.lib().fadam_plan_destroy(self._plan)
            self._plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def step_once(params, exp_avgs, exp_avg_sqs, grads, *, lr, betas, eps, weight_decay,
              step, adam_w_mode=True, bias_correction=True, grad_scale=1.0, params_out=None,
              lr_dev=None, step_dev=None, grad_scale_dev=None, noop=None) -> None:
    """One-shot step through ``fadam_step_once`` (all tensors in one group)."""
    descs = []
    outs = params_out or [None] * len(params)
    g_dtype = grads[0].dtype if grads else torch.float32
    out_dtype = outs[0].dtype if outs and outs[0] is not None else None
    for p, m, v, g, o in zip(params, exp_avgs, exp_avg_sqs, grads, outs):
        descs.append(_abi.Tensor(p=_ptr(p), m=_ptr(m), v=_ptr(v), g=_ptr(g), p_out=_ptr(o),
                                 rem=None, numel=p.numel(), group=0))
    arr = (_abi.Tensor * max(1, len(descs)))(*descs)
    dev = params[0].device if params else torch.device("cuda", torch.cuda.current_device())
    b1, b2 = betas
    _abi.check(_abi.lib().fadam_step_once(
        arr, len(descs), _abi.MODE_ADAMW if adam_w_mode else _abi.MODE_L2,
        1 if bias_correction else 0, float(b1), float(b2), float(eps), float(weight_decay),
        float(lr), _ptr(lr_dev), int(step), _ptr(step_dev), float(grad_scale),
        _ptr(grad_scale_dev), _ptr(noop), dtype_code(g_dtype), dtype_code(out_dtype),
        _stream_handle(dev)), "fadam_step_once")
