"""The allocation-free entry point, fadam_step_noalloc, against the plan path.

Some callers of this library cannot allocate device memory themselves: code
that runs while a framework's caching allocator holds nearly all of the
GPU's memory, hooks inside other libraries that may only use memory handed
to them, and loops that cannot afford a cudaMalloc/cudaFree that may
synchronise the device.  fadam_step_noalloc serves them from a static device
array instead of allocated scratch.  These tests call it through the C ABI
twice in a row and check each result against two steps of the existing
fadam_plan_create/fadam_step path on the same inputs, with the tolerance the
parity tests use; they also check that a shard too large for the array is
refused before any device work.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard, _abi
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _c_args(shard, lr_dev, gs_dev, step_dev):
    """Descriptors of `shard` in plan order, groups reading device scalars."""
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
        c.lr_dev = lr_dev[gi].data_ptr()
        c.grad_scale_dev = gs_dev.data_ptr()
        c.step_dev = step_dev[gi].data_ptr()
    return (_abi.Tensor * len(descs))(*descs), len(descs), groups


@pytest.mark.parametrize("check_finite", [False, True], ids=["capturable", "capturable+screen"])
def test_noalloc_matches_plan_path_on_two_calls(check_finite):
    spec = workloads.small_versions()["many_small"]
    ref = workloads.materialize(spec, DEV)
    out = workloads.materialize(spec, DEV)
    plan_opt = FusedAdamShard(ref.param_groups(), capturable=True, check_finite=check_finite)

    lr_dev = [torch.tensor([g.lr], dtype=torch.float32, device=DEV) for g in spec.groups]
    gs_dev = torch.tensor([spec.grad_scale], dtype=torch.float32, device=DEV)
    step_dev = [torch.zeros(1, dtype=torch.int32, device=DEV) for _ in spec.groups]
    noop = torch.zeros(1, dtype=torch.int32, device=DEV)
    arr, n, groups = _c_args(out, lr_dev, gs_dev, step_dev)
    flags = _abi.CAPTURABLE | (_abi.CHECK_FINITE if check_finite else 0)
    L = _abi.lib()
    stream = torch.cuda.current_stream().cuda_stream

    for call in (1, 2):
        plan_opt.step()
        st = L.fadam_step_noalloc(arr, n, groups, len(spec.groups), _abi.DT_F32, _abi.DT_F32,
                                  _abi.DT_NONE, flags, noop.data_ptr(), stream)
        assert st == _abi.OK, L.fadam_last_error()
        torch.cuda.synchronize()
        rep = helpers.Report()
        for i in ref.plan_order():
            rep.f32(helpers.to_np(out.params[i]), helpers.to_np(ref.params[i]), f"call {call} p")
            rep.f32(helpers.to_np(out.exp_avgs[i]), helpers.to_np(ref.exp_avgs[i]), f"call {call} m")
            rep.f32(helpers.to_np(out.exp_avg_sqs[i]), helpers.to_np(ref.exp_avg_sqs[i]),
                    f"call {call} v")
        assert [int(s.item()) for s in step_dev] == plan_opt.group_steps() == [call] * 3
        assert noop.item() == 0
    plan_opt.close()


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
