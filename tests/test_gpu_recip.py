"""GPU parity of the reciprocal bias corrections (FADAM_RECIP_BC) against
the oracle.

With the flag, the 16-bit state forms multiply the moments by 1/bc1 and
1/bc2 (one IEEE reciprocal per group and CTA) instead of dividing every
element: each bias-corrected moment carries one more rounding, so the
update u moves by a few float ulps.  m and v are computed before any
division and do not move.  p' = p - lr*u moves by a few ulps of lr*u, and
lr*u <= |p| + |p'|: where the step nearly cancels p, that is many ulps of a
small p', so p (and a param-out copy) is held to one ulp of its dtype plus
2e-6 * max(|p|, |p'|) + 1e-9 (helpers.check_recip_p16), values compared
after the scale for a scaled state, whose new scales must be within 2e-6
relative.  That bound holds for one step from a given state; over many
free-running steps the two paths may drift apart the way two 16-bit
trajectories do, so each step here starts from the oracle's state, written
into the GPU tensors.  Ten steps each, at the start of training and across
the steps where a correction becomes 1, regular and capturable.
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


def _state_spec(state_dtype, g_dtype, out_dtype):
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=state_dtype,
                                   g_dtype=g_dtype)
    spec.sizes = [40_003, 7, 131_072 + 5]
    spec.group_of = [0, 1, 1]
    spec.groups = [spec.groups[0], workloads.GroupSpec(adam_w_mode=False, weight_decay=0.05,
                                                       betas=(0.9, 0.999))]
    spec.out_dtype = out_dtype
    return spec


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("out_dtype", [None, torch.float32, torch.bfloat16])
@pytest.mark.parametrize("start", [0, 160, 20000])
def test_recip_16bit_state_each_step_within_one_ulp(state_dtype, g_dtype, out_dtype, start):
    spec = _state_spec(state_dtype, g_dtype, out_dtype)
    for capturable in (False, True):
        shard = workloads.materialize(spec, DEV)
        opt = FusedAdamShard(shard.param_groups(), capturable=capturable, recip_bc=True)
        osh = helpers.oracle_shard(shard)
        if start:
            opt.set_group_steps([start] * len(spec.groups))
            osh.steps = [start] * len(osh.steps)
        rep = helpers.Report()
        for k in range(1, 11):
            if k > 1:
                workloads.fresh_grads(shard, k)
                helpers.refresh_grads(osh, shard)
                helpers.load_oracle_state(shard, osh)
            p_before = helpers.unscaled_p(osh, state_dtype)
            opt.step()
            oracle.shard_step(osh, capturable=capturable)
            torch.cuda.synchronize()
            helpers.compare_recip(shard, osh, p_before, rep)
        assert opt.group_steps() == oracle.group_steps(osh) == [start + 10] * 2
        if start == 20000:
            # both corrections are 1 in float: the instance without any
            # division by them runs, bit for bit
            assert rep.exact_fraction == 1.0
        elif start == 0 and out_dtype == torch.float32:
            # the products by reciprocals do run: the fp32 param-out (p' as
            # computed, before any 16-bit rounding) differs from the
            # division's in a few float ulps for some of the 1.7 million
            # values (a 16-bit value only where p' falls within such a
            # distance of a rounding boundary, far rarer)
            assert rep.exact < rep.n
        print(f"{state_dtype} g {g_dtype} out {out_dtype} start {start} capturable {capturable}: "
              f"{rep.n} values, {rep.exact_fraction:.6f} bit-identical")
        opt.close()


@pytest.mark.parametrize("name", ["scaled_state_shard", "scaled_bf16"])
@pytest.mark.parametrize("capturable", [False, True])
def test_recip_scaled_state_each_step(name, capturable):
    spec = workloads.scaled_versions()[name]
    shard = workloads.materialize(spec, DEV)
    order = shard.plan_order()
    scales = shard.state_scales[order].contiguous()
    opt = FusedAdamShard(shard.param_groups(), capturable=capturable, state_scales=scales,
                         recip_bc=True)
    osh = helpers.oracle_shard(shard, scales=scales)
    rep = helpers.Report()
    for k in range(1, 11):
        if k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard)
            helpers.load_oracle_state(shard, osh, scales=scales)
        p_before = helpers.unscaled_p(osh, spec.state_dtype)
        opt.step()
        oracle.shard_step(osh, capturable=capturable)
        torch.cuda.synchronize()
        helpers.compare_recip(shard, osh, p_before, rep, got_scales=helpers.to_np(scales))
        got = helpers.to_np(scales).astype(np.float64)
        for j, t in enumerate(osh.tensors):
            want = t.scales.astype(np.float64)
            assert np.all(np.abs(got[j] - want) <= 2e-6 * np.abs(want)), (k, j, got[j], want)
    assert opt.group_steps() == [10]
    print(f"{name} capturable {capturable}: {rep.n} values, "
          f"{rep.exact_fraction:.6f} bit-identical")
    opt.close()


@pytest.mark.parametrize("start", [0, 160])
def test_recip_special_values(start):
    """Infinities, NaNs, signed zeros, subnormals and values near overflow in
    p, m, v and g of a bf16 state with fp16 gradients and an fp16 param-out,
    with FADAM_RECIP_BC, one step from the same state on both sides: m and v
    bit-identical to the oracle (no division precedes them), every p or
    param-out value that is infinite or NaN on either side the same on the
    other (NaN where the oracle gives NaN, the same infinity), and the
    finite ones within the derived bound."""
    from tests.test_gpu_parity import _sprinkle
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=torch.bfloat16,
                                   g_dtype=torch.float16)
    spec.out_dtype = torch.float16
    shard = workloads.materialize(spec, DEV)
    gen = np.random.default_rng(16)
    for i in range(len(shard.params)):
        shard.exp_avgs[i].copy_(torch.randn_like(shard.exp_avgs[i]) * 1e-2)
        shard.exp_avg_sqs[i].copy_(torch.rand_like(shard.exp_avg_sqs[i]) * 1e-4)
        for t, every in ((shard.params[i], 7), (shard.exp_avgs[i], 11),
                         (shard.exp_avg_sqs[i], 13), (shard.grads[i], 5)):
            _sprinkle(t, gen, every)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, recip_bc=True)
    osh = helpers.oracle_shard(shard)
    if start:
        opt.set_group_steps([start] * len(spec.groups))
        osh.steps = [start] * len(osh.steps)
    p_before = helpers.unscaled_p(osh, spec.state_dtype)
    opt.step()
    oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    rep = helpers.Report()
    n_nonfinite = 0
    for t, i, x0 in zip(osh.tensors, shard.plan_order(), p_before):
        for got_t, want, what in ((shard.exp_avgs[i], t.m, "m"), (shard.exp_avg_sqs[i], t.v, "v")):
            got = helpers.to_np(got_t)
            nan = np.isnan(helpers.widen16(got, spec.state_dtype))
            want_nan = np.isnan(helpers.widen16(want, spec.state_dtype))
            # the same bits, any two NaNs alike (payloads are not compared)
            assert ((got == want) | (nan & want_nan)).all(), f"tensor {i} {what}"
        for got_t, want, dt, what in ((shard.params[i], t.p, spec.state_dtype, "p"),
                                      (shard.params_out[i], t.p_out, spec.out_dtype, "p_out")):
            got = helpers.to_np(got_t)
            g = helpers.widen16(got, dt)
            w = helpers.widen16(want, dt)
            special = ~np.isfinite(g) | ~np.isfinite(w) | ~np.isfinite(x0)
            same = (g == w) | (np.isnan(g) & np.isnan(w))
            assert same[~np.isfinite(g) | ~np.isfinite(w)].all(), f"tensor {i} {what}: non-finite"
            n_nonfinite += int(special.sum())
            helpers.check_recip_p16(got[~special], want[~special], dt, x0[~special],
                                    f"tensor {i} {what}", rep)
    assert n_nonfinite > 0 and rep.n > 0
    print(f"start {start}: {n_nonfinite} non-finite values matched, {rep.n} finite within the bound, "
          f"{rep.exact_fraction:.6f} of those bit-identical")
