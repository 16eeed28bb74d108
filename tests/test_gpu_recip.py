"""GPU parity of the reciprocal bias corrections (FADAM_RECIP_BC) against
the oracle.

With the flag, the 16-bit state forms multiply the moments by 1/bc1 and
1/bc2 (one IEEE reciprocal per group and CTA) instead of dividing every
element: each bias-corrected moment carries one more rounding, so the
update u moves by a few float ulps and a value stored in 16 bits by at most
one unit in its last place.  That bound holds for one step from a given
state; over many free-running steps the two paths may drift apart the way
two 16-bit trajectories do, so each step here starts from the oracle's
state, written into the GPU tensors, and the step's results are compared:
p, m, v and a 16-bit param-out within one 16-bit ulp (m and v come out
exact, being computed before any division), and the scaled state's new
scales within 2e-6 relative.

An fp32 param-out is p' = p - lr*u unrounded.  The reciprocal's extra
rounding is relative to lr*u, which exceeds |p'| when the two terms nearly
cancel (a 16-bit v that underflowed can leave u well above 1), so the
error bound follows the larger of the terms: |d| <= 2e-6 * max(|p|, |p'|)
+ 1e-9, the fp32 tolerance's relative form taken against the step's input
as well as its result (a few float ulps of lr*u <= |p| + |p'| stay far
inside it).  Ten steps each, at the start of training and across the
steps where a correction becomes 1, regular and capturable.
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


def _widen16(bits, dtype):
    return oracle.bf16_to_f32(bits) if dtype == torch.bfloat16 else oracle.f16_to_f32(bits)


def _compare_recip(shard, osh, p_before, rep):
    """16-bit p, m, v and param-out within one ulp; an fp32 param-out within
    2e-6 * max(|p before the step|, |p'|) + 1e-9."""
    spec = shard.spec
    sdt = spec.state_dtype
    for t, i, x0 in zip(osh.tensors, shard.plan_order(), p_before):
        rep.ulp16(helpers.to_np(shard.exp_avgs[i]), t.m, f"tensor {i} m", sdt)
        rep.ulp16(helpers.to_np(shard.exp_avg_sqs[i]), t.v, f"tensor {i} v", sdt)
        rep.ulp16(helpers.to_np(shard.params[i]), t.p, f"tensor {i} p", sdt)
        if spec.out_dtype == torch.float32:
            got = helpers.to_np(shard.params_out[i]).astype(np.float64)
            want = t.p_out.astype(np.float64)
            lim = 2e-6 * np.maximum(np.abs(want), np.abs(x0.astype(np.float64))) + 1e-9
            d = np.abs(got - want)
            bad = ~(d <= lim)
            assert not bad.any(), (f"tensor {i} p_out: {int(bad.sum())} outside; first at "
                                   f"{int(np.argmax(bad))}")
            rep.n += got.size
            rep.exact += int(np.sum(got == want))
        elif spec.out_dtype is not None:
            rep.ulp16(helpers.to_np(shard.params_out[i]), t.p_out, f"tensor {i} p_out",
                      spec.out_dtype)


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
            p_before = [_widen16(t.p, state_dtype) for t in osh.tensors]
            opt.step()
            oracle.shard_step(osh, capturable=capturable)
            torch.cuda.synchronize()
            _compare_recip(shard, osh, p_before, rep)
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
        opt.step()
        oracle.shard_step(osh, capturable=capturable)
        torch.cuda.synchronize()
        helpers.compare(shard, osh, report=rep)
        got = helpers.to_np(scales).astype(np.float64)
        for j, t in enumerate(osh.tensors):
            want = t.scales.astype(np.float64)
            assert np.all(np.abs(got[j] - want) <= 2e-6 * np.abs(want)), (k, j, got[j], want)
    assert opt.group_steps() == [10]
    print(f"{name} capturable {capturable}: {rep.n} values, "
          f"{rep.exact_fraction:.6f} bit-identical")
    opt.close()
