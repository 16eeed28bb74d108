"""Checkpoint and resume of a shard's scalar state.

"[PyTorch] Advance FusedAdam step counter for empty param groups": every
group, empty or not, carries a step counter, and a checkpoint that stores no
step for an empty group resumes with the wrong bias correction.  Here a
shard with an empty group runs two steps, its state_dict (an int step for
every group, learning rates, grad scale) goes into a fresh optimizer over
copies of the tensors, and both run two more steps on the same gradients:
the resumed run must equal the uninterrupted one bit for bit, step counters
included.
"""
import pytest
import torch

import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _clone_groups(groups):
    out = []
    for g in groups:
        c = dict(g)
        for k in ("params", "exp_avgs", "exp_avg_sqs", "params_out", "remainders"):
            if k in c and c[k] is not None:
                c[k] = [t.clone() for t in c[k]]
        out.append(c)
    return out


def _state_tensors(groups):
    return [t for g in groups for k in ("params", "exp_avgs", "exp_avg_sqs", "params_out",
                                        "remainders") for t in (g.get(k) or [])]


@pytest.mark.parametrize("capturable", [False, True])
def test_resume_from_state_dict_is_bit_identical(capturable):
    spec = workloads.small_versions()["many_small"]
    assert any(k not in spec.group_of for k in range(len(spec.groups)))  # an empty group
    shard = workloads.materialize(spec, DEV)
    groups = shard.param_groups()
    opt = FusedAdamShard(groups, capturable=capturable, grad_scale=spec.grad_scale)
    for k in (1, 2):
        if k > 1:
            workloads.fresh_grads(shard, k)
        opt.step()
    opt.set_lr(0, 7e-4)
    sd = opt.state_dict()
    assert sd["step"] == [2] * len(spec.groups)
    assert all(isinstance(s, int) for s in sd["step"])
    assert sd["lr"][0] == pytest.approx(7e-4)

    resumed_groups = _clone_groups(groups)  # the checkpointed tensors
    fresh = FusedAdamShard(resumed_groups, capturable=capturable, grad_scale=1.0)
    fresh.set_lr(0, 1.0)  # overwritten by the checkpoint
    fresh.load_state_dict(sd)
    assert fresh.state_dict() == sd
    for k in (3, 4):
        workloads.fresh_grads(shard, k)  # the grads tensors are shared by both
        opt.step()
        fresh.step()
    torch.cuda.synchronize()
    for a, b in zip(_state_tensors(groups), _state_tensors(resumed_groups)):
        assert torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a,
                           b.view(torch.int32) if b.dtype == torch.float32 else b)
    assert opt.group_steps() == fresh.group_steps() == [4] * len(spec.groups)
    opt.close()
    fresh.close()


@pytest.mark.parametrize("capturable", [False, True])
def test_empty_group_step_in_state_dict_after_three_steps(capturable):
    """The check the TransformerEngine fix describes: one populated group
    and one empty group, three steps, both groups at step 3 in the state
    dict (before the fix the empty group had no step)."""
    p = torch.randn(1000, device=DEV)
    groups = [{"params": [p], "exp_avgs": [torch.zeros_like(p)],
               "exp_avg_sqs": [torch.zeros_like(p)], "grads": [torch.randn_like(p) * 1e-3],
               "lr": 1e-3},
              {"params": [], "exp_avgs": [], "exp_avg_sqs": [], "grads": [], "lr": 1e-3}]
    opt = FusedAdamShard(groups, capturable=capturable)
    for _ in range(3):
        opt.step()
    sd = opt.state_dict()
    assert sd["step"] == [3, 3]
    assert opt.group_steps() == [3, 3]
    opt.close()


def test_load_state_dict_refuses_a_missing_step():
    spec = workloads.small_versions()["tiny_adamw"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups())
    sd = opt.state_dict()
    bad = dict(sd, step=[None] + sd["step"][1:])
    with pytest.raises(ValueError):
        opt.load_state_dict(bad)
    with pytest.raises(ValueError):
        opt.load_state_dict(dict(sd, step=sd["step"][:-1]))
    opt.close()
