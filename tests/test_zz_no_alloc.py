"""The allocation-free entry point, fadam_step_noalloc.

Some callers of this library cannot allocate device memory themselves: code
that runs while a framework's caching allocator holds nearly all of the
GPU's memory, hooks inside other libraries that may only use memory handed
to them, and loops that cannot afford a cudaMalloc/cudaFree that may
synchronise the device.  fadam_step_noalloc serves them from a static device
array instead of allocated scratch.  These tests call it through the C ABI:

* twice in a row, capturable (with and without the inf/nan screen), each
  result against two steps of the fadam_plan_create/fadam_step path on the
  same inputs, with the tolerance the parity tests use;
* twice in a row with host scalars (regular), each result against the
  oracle directly;
* with the noop flag set (nothing written, no counter moved), then clear;
* with a bf16 state and reciprocal bias corrections, against the plan path
  with the same flag;
* on two shards with different betas at the same step indices, in turn,
  and with a counter moved by the caller: the bias-correction memo in the
  shared array must never serve an entry made for other betas or another
  step, so every result is bit-identical to the plan path's;
* on a stream that is capturing (refused before any device work), and with
  a shard too large for the array (refused before any device work).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import copy

import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard, _abi
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _c_args(shard, lr_dev=None, gs_dev=None, step_dev=None, host_steps=None):
    """Descriptors of `shard` in plan order; groups read device scalars when
    `lr_dev` is given (capturable), else the host lr, grad scale and the
    step of this update from `host_steps` (regular)."""
    spec = shard.spec
    order = shard.plan_order()
    descs = [_abi.Tensor(p=shard.params[i].data_ptr(), m=shard.exp_avgs[i].data_ptr(),
                         v=shard.exp_avg_sqs[i].data_ptr(), g=shard.grads[i].data_ptr(),
                         p_out=None, rem=None, numel=shard.params[i].numel(),
                         group=spec.group_of[i]) for i in order]
    groups = (_abi.Group * len(spec.groups))()
    for gi, g in enumerate(spec.groups):
        c = groups[gi]
        c.mode = _abi.MODE_ADAMW if g.adam_w_mode else _abi.MODE_L2
        c.bias_correction = 1 if g.bias_correction else 0
        c.beta1, c.beta2 = g.betas
        c.eps, c.weight_decay = g.eps, g.weight_decay
        if lr_dev is not None:
            c.lr_dev = lr_dev[gi].data_ptr()
            c.grad_scale_dev = gs_dev.data_ptr()
            c.step_dev = step_dev[gi].data_ptr()
        else:
            c.lr, c.grad_scale, c.step = g.lr, spec.grad_scale, host_steps[gi]
    return (_abi.Tensor * len(descs))(*descs), len(descs), groups


class _DeviceScalars:
    """Device lr per group, one grad scale and a step counter per group."""

    def __init__(self, spec):
        self.lr = [torch.tensor([g.lr], dtype=torch.float32, device=DEV) for g in spec.groups]
        self.gs = torch.tensor([spec.grad_scale], dtype=torch.float32, device=DEV)
        self.step = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in spec.groups]

    def steps(self):
        return [int(s.item()) for s in self.step]


def _noalloc(shard, args, flags, noop=None):
    arr, n, groups = args
    L = _abi.lib()
    st = L.fadam_step_noalloc(arr, n, groups, len(shard.spec.groups), _abi.DT_F32, _abi.DT_F32,
                              _abi.DT_NONE, flags, None if noop is None else noop.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    return st


def _bit_equal(a, b):
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        if not torch.equal(x.view(torch.int32), y.view(torch.int32)):
            return False
    return True


@pytest.mark.parametrize("check_finite", [False, True], ids=["capturable", "capturable+screen"])
def test_noalloc_matches_plan_path_on_two_calls(check_finite):
    spec = workloads.small_versions()["many_small"]
    ref = workloads.materialize(spec, DEV)
    out = workloads.materialize(spec, DEV)
    plan_opt = FusedAdamShard(ref.param_groups(), capturable=True, check_finite=check_finite)
    ds = _DeviceScalars(spec)
    noop = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = _c_args(out, ds.lr, ds.gs, ds.step)
    flags = _abi.CAPTURABLE | (_abi.CHECK_FINITE if check_finite else 0)
    L = _abi.lib()

    for call in (1, 2):
        plan_opt.step()
        st = _noalloc(out, args, flags, noop)
        assert st == _abi.OK, L.fadam_last_error()
        torch.cuda.synchronize()
        rep = helpers.Report()
        for i in ref.plan_order():
            rep.f32(helpers.to_np(out.params[i]), helpers.to_np(ref.params[i]), f"call {call} p")
            rep.f32(helpers.to_np(out.exp_avgs[i]), helpers.to_np(ref.exp_avgs[i]), f"call {call} m")
            rep.f32(helpers.to_np(out.exp_avg_sqs[i]), helpers.to_np(ref.exp_avg_sqs[i]),
                    f"call {call} v")
        assert ds.steps() == plan_opt.group_steps() == [call] * 3
        assert noop.item() == 0
    plan_opt.close()


def test_noalloc_regular_host_scalars_match_oracle():
    """Two regular calls (host lr, grad scale and step, fresh gradients for
    the second) against the oracle itself, element by element."""
    spec = workloads.small_versions()["many_small"]
    out = workloads.materialize(spec, DEV)
    osh = helpers.oracle_shard(out)
    L = _abi.lib()
    for call in (1, 2):
        if call > 1:
            workloads.fresh_grads(out, call)
            helpers.refresh_grads(osh, out)
        args = _c_args(out, host_steps=[call] * len(spec.groups))
        assert _noalloc(out, args, 0) == _abi.OK, L.fadam_last_error()
        oracle.shard_step(osh, capturable=False)
        torch.cuda.synchronize()
        rep = helpers.compare(out, osh)
        assert rep.n == 3 * sum(spec.sizes)
    assert oracle.group_steps(osh) == [2, 2, 2]


def test_noalloc_noop_flag_leaves_everything():
    """A set noop flag: p, m, v and the device counters stay bit-identical,
    on the capturable and on the regular form; after the flag is cleared the
    next call is the oracle's first step."""
    spec = workloads.small_versions()["many_small"]
    out = workloads.materialize(spec, DEV)
    osh = helpers.oracle_shard(out)
    ds = _DeviceScalars(spec)
    noop = torch.ones(1, dtype=torch.int32, device=DEV)
    snap = helpers.snapshot(out)
    L = _abi.lib()
    cap_args = _c_args(out, ds.lr, ds.gs, ds.step)
    assert _noalloc(out, cap_args, _abi.CAPTURABLE, noop) == _abi.OK, L.fadam_last_error()
    reg_args = _c_args(out, host_steps=[1] * len(spec.groups))
    assert _noalloc(out, reg_args, 0, noop) == _abi.OK, L.fadam_last_error()
    oracle.shard_step(osh, capturable=True, noop=True)
    torch.cuda.synchronize()
    assert helpers.state_equal(out, snap)
    assert ds.steps() == oracle.group_steps(osh) == [0, 0, 0] and noop.item() == 1
    noop.zero_()
    assert _noalloc(out, cap_args, _abi.CAPTURABLE, noop) == _abi.OK, L.fadam_last_error()
    oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    helpers.compare(out, osh)
    assert ds.steps() == oracle.group_steps(osh) == [1, 1, 1] and noop.item() == 0


def test_noalloc_memo_serves_only_matching_betas_and_steps():
    """Shard A (betas (0.9, 0.999)) and shard B (betas (0.8, 0.95), its own
    counters) alternate at the same step indices, then A's counters are
    moved by the caller: every call's state is bit-identical to the plan
    path's on a copy of the same shard (each plan has a memo of its own)."""
    spec_a = workloads.small_versions()["many_small"]
    spec_b = copy.deepcopy(workloads.small_versions()["large_uniform"])
    spec_b.seed += 11
    for g in spec_b.groups:
        g.betas = (0.8, 0.95)
    shards, refs, plans, scal, args = {}, {}, {}, {}, {}
    for key, spec in (("A", spec_a), ("B", spec_b)):
        shards[key] = workloads.materialize(spec, DEV)
        refs[key] = workloads.materialize(spec, DEV)
        plans[key] = FusedAdamShard(refs[key].param_groups(), capturable=True)
        scal[key] = _DeviceScalars(spec)
        args[key] = _c_args(shards[key], scal[key].lr, scal[key].gs, scal[key].step)
    noop = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = _abi.lib()

    def both(key):
        plans[key].step()
        assert _noalloc(shards[key], args[key], _abi.CAPTURABLE, noop) == _abi.OK, \
            L.fadam_last_error()
        torch.cuda.synchronize()
        assert _bit_equal(shards[key], refs[key]), f"shard {key} differs from the plan path"
        assert scal[key].steps() == plans[key].group_steps()

    for key in ("A", "B", "A", "B", "A"):
        both(key)
    assert scal["A"].steps() == [3, 3, 3] and scal["B"].steps() == [2]
    # the caller moves A's counters to 5: the next call applies step 6, of
    # the same parity as the entry A's last call left behind (step 4), which
    # must not serve
    moved = [5, 5, 5]
    plans["A"].set_group_steps(moved)
    for s, v in zip(scal["A"].step, moved):
        s.fill_(v)
    both("A")
    both("B")
    assert scal["A"].steps() == [6, 6, 6] and scal["B"].steps() == [3]
    for p in plans.values():
        p.close()


def test_noalloc_16bit_state_with_reciprocal_corrections():
    """A bf16 state with FADAM_RECIP_BC (its own kernel instances): two
    capturable calls bit-identical to the plan path with the same flag."""
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=torch.bfloat16,
                                   g_dtype=torch.bfloat16)
    spec.sizes = [40_003, 7, 131_072 + 5]
    ref = workloads.materialize(spec, DEV)
    out = workloads.materialize(spec, DEV)
    plan_opt = FusedAdamShard(ref.param_groups(), capturable=True, recip_bc=True)
    ds = _DeviceScalars(spec)
    noop = torch.zeros(1, dtype=torch.int32, device=DEV)
    arr, n, groups = _c_args(out, ds.lr, ds.gs, ds.step)
    L = _abi.lib()
    for call in (1, 2):
        plan_opt.step()
        st = L.fadam_step_noalloc(arr, n, groups, len(spec.groups), _abi.DT_BF16, _abi.DT_BF16,
                                  _abi.DT_NONE, _abi.CAPTURABLE | _abi.RECIP_BC, noop.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
        assert st == _abi.OK, L.fadam_last_error()
        torch.cuda.synchronize()
        for x, y in zip(helpers.snapshot(out), helpers.snapshot(ref)):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"call {call}"
        assert ds.steps() == plan_opt.group_steps() == [call]
    plan_opt.close()


# the refused call launches nothing, so the captured graph is empty
@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_noalloc_refuses_a_capturing_stream():
    """Each call uploads its work list from host memory that is freed when
    it returns, so a call on a capturing stream is refused before any device
    work: nothing is captured and nothing runs."""
    spec = workloads.small_versions()["tiny_adamw"]
    out = workloads.materialize(spec, DEV)
    ds = _DeviceScalars(spec)
    noop = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = _c_args(out, ds.lr, ds.gs, ds.step)
    L = _abi.lib()
    assert _noalloc(out, args, _abi.CAPTURABLE, noop) == _abi.OK, L.fadam_last_error()
    torch.cuda.synchronize()
    snap = helpers.snapshot(out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        graph.capture_begin()
        st = _noalloc(out, args, _abi.CAPTURABLE, noop)
        msg = L.fadam_last_error()
        graph.capture_end()
    torch.cuda.current_stream().wait_stream(side)
    assert st == _abi.EINVAL and b"capture" in msg
    torch.cuda.synchronize()
    assert helpers.state_equal(out, snap) and ds.steps() == [1, 1]
    # the stream works as before once the capture has ended
    assert _noalloc(out, args, _abi.CAPTURABLE, noop) == _abi.OK, L.fadam_last_error()
    torch.cuda.synchronize()
    assert ds.steps() == [2, 2]


def test_noalloc_refuses_a_shard_beyond_its_array():
    # 5000 one-element tensors pack into 5000 work items, more than the 4096
    # the static array holds; the call must refuse before any device work
    buf = torch.zeros(4 * 5000, dtype=torch.float32, device=DEV)
    base = buf.data_ptr()
    descs = [_abi.Tensor(p=base + 4 * i, m=base + 4 * (5000 + i), v=base + 4 * (10000 + i),
                         g=base + 4 * (15000 + i), numel=1, group=0) for i in range(5000)]
    arr = (_abi.Tensor * 5000)(*descs)
    grp = (_abi.Group * 1)(_abi.Group(mode=1, bias_correction=1, beta1=0.9, beta2=0.999, eps=1e-8,
                                      weight_decay=0.0, lr=1e-3, grad_scale=1.0, step=1))
    L = _abi.lib()
    st = L.fadam_step_noalloc(arr, 5000, grp, 1, _abi.DT_F32, _abi.DT_F32, _abi.DT_NONE, 0, None,
                              torch.cuda.current_stream().cuda_stream)
    assert st == _abi.ELIMIT
    assert b"4096" in L.fadam_last_error()
    torch.cuda.synchronize()
    assert not buf.any()
