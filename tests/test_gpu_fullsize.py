"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses (default plan: persistent grid sized to the device).

The oracle cannot redo 1-4e9 elements per step in seconds, so each test
samples elements (every tensor's first and last element included), gathers
their inputs before the steps, and lets the oracle run the same steps on the
samples only; every element updates independently, so this is exact.  The
noop step of the capturable L2 shard is checked bit-exactly over the whole
state, and the step counters over every group.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _sampled_run(spec, steps, per_tensor, tensor_subset=None, inf_step=None, capturable=None):
    if capturable is not None:
        spec.capturable = capturable
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=spec.capturable,
                         remainders=spec.remainders, grad_scale=spec.grad_scale)
    order = shard.plan_order()
    idx = order if tensor_subset is None else [i for i in order if i in tensor_subset]
    elems = helpers.sample_elements(spec, per_tensor, seed=spec.seed + 5)
    osh = helpers.oracle_shard(shard, idx=idx, elems=elems)
    t_inf, e_inf = workloads.inf_position(spec) if inf_step else (None, None)
    for k in range(1, steps + 1):
        noop = k == inf_step
        if noop:
            saved = shard.grads[t_inf][e_inf].clone()
            shard.grads[t_inf][e_inf] = float("inf")
            before = helpers.snapshot(shard)
            opt.noop.copy_(torch.isinf(shard.grads[t_inf]).any().to(torch.int32).view(1))
        opt.step()
        if noop:
            torch.cuda.synchronize()
            assert opt.noop.item() == 1
            assert helpers.state_equal(shard, before), "a noop step changed the state"
            del before
            shard.grads[t_inf][e_inf] = saved
            opt.noop.zero_()
        oracle.shard_step(osh, capturable=spec.capturable, noop=noop)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh, idx=idx, elems=elems)
    steps_dev = opt.group_steps()
    opt.close()
    del shard, opt
    _free()
    return rep, steps_dev, oracle.group_steps(osh)


def test_large_uniform_full_size():
    spec = workloads.large_uniform()
    # the benchmark's headline path: capturable, device scalars
    rep, steps, want = _sampled_run(spec, 2, per_tensor=4096, capturable=True)
    assert steps == want == [2]
    print(f"large_uniform: {rep.n} sampled values, {rep.exact_fraction:.6f} bit-identical")


def test_large_uniform_bf16_moments_full_size():
    # the 201-tensor shard with an fp32 master and bf16 moments, capturable
    spec = workloads.large_uniform(moment_dtype=torch.bfloat16)
    rep, steps, want = _sampled_run(spec, 2, per_tensor=2048, capturable=True)
    assert steps == want == [2]
    assert rep.exact_fraction == 1.0


def test_capturable_l2_full_size_with_inf_step():
    spec = workloads.capturable_l2()
    rep, steps, want = _sampled_run(spec, 5, per_tensor=4096, inf_step=spec.inf_at_step)
    assert steps == want == [4]
    print(f"capturable_l2: {rep.n} sampled values, {rep.exact_fraction:.6f} bit-identical")


def test_remainder_shard_full_size():
    spec = workloads.remainder_shard()
    rep, steps, want = _sampled_run(spec, 3, per_tensor=2048)
    assert steps == want == [3]
    print(f"remainder_shard: {rep.n} sampled values, {rep.exact_fraction:.6f} bit-identical")


def test_many_small_full_size():
    spec = workloads.many_small()
    rng = np.random.default_rng(3)
    subset = set(rng.choice(len(spec.sizes), size=1500, replace=False).tolist())
    subset |= {0, len(spec.sizes) - 1}
    rep, steps, want = _sampled_run(spec, 5, per_tensor=256, tensor_subset=subset)
    assert steps == want == [5, 5, 5]
    print(f"many_small: {rep.n} sampled values, {rep.exact_fraction:.6f} bit-identical")


def test_tensor_beyond_2_pow_31_elements():
    n = (1 << 31) + 4099
    spec = workloads.large_uniform(n_tensors=1, numel=n)
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=False)
    e = np.unique(np.concatenate([np.arange(0, 64), np.arange(n - 4200, n),
                                  (1 << 31) + np.arange(-64, 64),
                                  np.random.default_rng(1).choice(n, 100_000, replace=False)]))
    elems = {0: e.astype(np.int64)}
    osh = helpers.oracle_shard(shard, elems=elems)
    opt.step()
    oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    helpers.compare(shard, osh, elems=elems)
    info = opt.info()
    assert info["n_elements"] == n and info["n_items"] >= 32
    opt.close()
    del shard, opt
    _free()


def test_large_uniform_norm_full_size():
    """Squared norm of the 201 x 20,971,520 shard against the oracle run
    tensor by tensor on the host."""
    spec = workloads.large_uniform()
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    got = opt.grad_norm_sq().item()
    want = sum(oracle.sumsq(helpers.to_np(g), oracle.DT_F32) for g in shard.grads)
    assert got == pytest.approx(want, rel=2e-6)
    opt.close()
    del shard, opt
    _free()


def test_exchange_shard_full_size():
    """Eight ranks' bf16 gradients averaged into the 1.2e9-element shard and
    stepped in one launch, param-out to the seven other ranks' places, for
    two steps; sampled elements against the oracle (the reduced gradient
    bit for bit), destinations byte-equal over the whole shard."""
    spec = workloads.exchange_versions(full=True)["exchange_shard"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    opt.set_exchange(shard.buckets["g"], list(shard.sources), average=True,
                     out_shard=shard.buckets["p_out"], dests=list(shard.dests))
    order = shard.plan_order()
    elems = helpers.sample_elements(spec, 4096, seed=spec.seed + 5)
    osh = helpers.oracle_shard(shard, elems=elems)
    src = []
    for i in order:
        e = torch.as_tensor(elems[i], device=DEV) + shard.offsets[i]
        src.append([helpers.to_np(shard.sources[r][e]) for r in range(spec.exchange_ranks)])
    for _ in range(2):
        opt.step_reduce()
        oracle.exchange_step(osh, src, average=True, capturable=True)
    torch.cuda.synchronize()
    for t, i in zip(osh.tensors, order):
        got = helpers.to_np(shard.grads[i][torch.as_tensor(elems[i], device=DEV)])
        assert got.tobytes() == t.g.tobytes(), f"tensor {i}: reduced gradient differs"
    rep = helpers.compare(shard, osh, elems=elems)
    assert rep.exact_fraction == 1.0
    out = shard.buckets["p_out"].view(torch.int16)
    for d in range(spec.exchange_dests):
        assert torch.equal(shard.dests[d].view(torch.int16), out), f"destination {d}"
    assert opt.group_steps() == [2]
    opt.close()
    del shard, opt
    _free()


def test_scaled_state_full_size():
    """The 1.2e9-element fp16 scaled-state shard, two regular steps.  The
    rescale depends on every element of a tensor, so the oracle runs whole
    tensors: the first layer's 4096x4096 and 4096x11008 matrices and both
    norm vectors, against every one of their elements and their scales."""
    spec = workloads.scaled_versions(full=True)["scaled_state_shard"]
    shard = workloads.materialize(spec, DEV)
    order = shard.plan_order()
    scales = shard.state_scales[order].contiguous()
    opt = FusedAdamShard(shard.param_groups(), state_scales=scales)
    pos = [0, 1, 4, 5]
    idx = [order[k] for k in pos]
    osh = helpers.oracle_shard(shard, idx=idx, scales=scales[pos])
    for k in (1, 2):
        if k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard, idx=idx)
        opt.step()
        oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh, idx=idx)
    assert rep.exact_fraction == 1.0
    got = helpers.to_np(scales)
    for k, t in zip(pos, osh.tensors):
        assert got[k].tobytes() == t.scales.tobytes(), k
    assert opt.group_steps() == [2]
    opt.close()
    del shard, opt
    _free()
