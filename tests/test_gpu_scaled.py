"""GPU parity of the scaled 16-bit optimizer state (FADAM_SCALED_STATES)
against the oracle: p, m, v bits, the new scales and the param-out copy
over several steps (fp16, and bf16 in the range where its scale target
keeps reciprocals finite), bf16's overflowing reciprocals reproduced NaN for
NaN, an empty tensor keeping its scales, a set noop flag, the inf/nan
screen, graph replay, the exchange stand-in in front of it, and the checks
on plans and dtypes."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard, _abi
from adamw_optimizer_step_persistent_gb300._abi import FadamError
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _make(name, capturable=False, **kw):
    spec = workloads.scaled_versions()[name]
    shard = workloads.materialize(spec, DEV)
    order = shard.plan_order()
    scales = shard.state_scales[order].contiguous()
    opt = FusedAdamShard(shard.param_groups(), capturable=capturable, state_scales=scales, **kw)
    osh = helpers.oracle_shard(shard, scales=scales)
    return spec, shard, opt, osh, scales


def _check_scales(opt, osh, nan_ok=False):
    got = helpers.to_np(opt.state_scales)
    for k, t in enumerate(osh.tensors):
        if nan_ok:
            assert np.array_equal(np.isnan(got[k]), np.isnan(t.scales)), k
            ok = ~np.isnan(t.scales)
            assert got[k][ok].tobytes() == t.scales[ok].tobytes(), (k, got[k], t.scales)
        else:
            assert got[k].tobytes() == t.scales.tobytes(), (k, got[k], t.scales)


@pytest.mark.parametrize("capturable", [False, True])
@pytest.mark.parametrize("name", ["scaled_state_shard", "scaled_bf16"])
def test_scaled_steps_match_oracle(name, capturable):
    spec, shard, opt, osh, _ = _make(name, capturable=capturable)
    rep = helpers.Report()
    for k in range(1, 4):
        if k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard)
        opt.step()
        oracle.shard_step(osh, capturable=capturable)
        torch.cuda.synchronize()
        helpers.compare(shard, osh, report=rep)
        _check_scales(opt, osh)
    assert rep.exact_fraction == 1.0, rep.exact_fraction
    assert opt.group_steps() == [3]
    # the empty tensor kept the scales it was given
    empty = [k for k, i in enumerate(shard.plan_order()) if spec.sizes[i] == 0]
    for k in empty:
        assert helpers.to_np(opt.state_scales[k]).tolist() == pytest.approx(list(spec.scale_of))
    opt.close()


@pytest.mark.parametrize("start", [163, 20000])
def test_scaled_late_steps_match_oracle(start):
    """The scaled passes at steps where the bias corrections round to 1
    (their tile instances leave those divisions out): bits and scales equal
    the oracle's across the switch at step 165 and far beyond it."""
    spec, shard, opt, osh, _ = _make("scaled_state_shard", capturable=True)
    opt.set_group_steps([start])
    osh.steps = [start] * len(osh.steps)
    rep = helpers.Report()
    for k in range(1, 4):
        if k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard)
        opt.step()
        oracle.shard_step(osh, capturable=True)
        torch.cuda.synchronize()
        helpers.compare(shard, osh, report=rep)
        _check_scales(opt, osh)
    assert rep.exact_fraction == 1.0, rep.exact_fraction
    assert opt.group_steps() == [start + 3]
    opt.close()


def test_bf16_overflowing_reciprocals_as_the_oracle():
    spec, shard, opt, osh, _ = _make("scaled_bf16_small_moments")
    opt.step()
    oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)  # NaN matches NaN whatever the payload
    _check_scales(opt, osh, nan_ok=True)
    # the moments' reciprocals overflowed: their stored values are infinite
    m = helpers.to_np(shard.exp_avgs[shard.plan_order()[0]])
    assert np.all(~np.isfinite(oracle.bf16_to_f32(m)))
    assert rep.exact_fraction == 1.0
    opt.close()


def test_noop_leaves_state_and_scales():
    spec, shard, opt, osh, scales = _make("scaled_state_shard", capturable=True)
    snap = helpers.snapshot(shard)
    before = scales.clone()
    opt.noop.fill_(1)
    opt.step()
    torch.cuda.synchronize()
    assert helpers.state_equal(shard, snap)
    assert torch.equal(before, opt.state_scales) and opt.group_steps() == [0]
    opt.close()


def test_screen_skips_a_scaled_step():
    spec, shard, opt, osh, scales = _make("scaled_state_shard", capturable=True, check_finite=True)
    opt.step()
    oracle.shard_step(osh, capturable=True)
    snap = helpers.snapshot(shard)
    before = opt.state_scales.clone()
    shard.grads[shard.plan_order()[2]][7] = float("nan")
    opt.step()
    torch.cuda.synchronize()
    assert opt.noop.item() == 1 and opt.group_steps() == [1]
    assert helpers.state_equal(shard, snap) and torch.equal(before, opt.state_scales)
    helpers.compare(shard, osh)
    opt.close()


def test_scaled_plan_recovers_from_a_wait_that_gave_up():
    """The first step's screen barrier runs out (diagnostic flag): nothing is
    written, scales included.  The next steps on the same plan, its status
    left unread, store the rescaled state and replace the scales as the
    oracle does (a timeout of an earlier launch does not hold the new scales
    back)."""
    spec, shard, opt, osh, scales = _make("scaled_state_shard", capturable=True, check_finite=True,
                                          extra_flags=_abi.TEST_BARRIER_TIMEOUT)
    snap = helpers.snapshot(shard)
    before = scales.clone()
    opt.step()
    torch.cuda.synchronize()
    assert helpers.state_equal(shard, snap) and torch.equal(before, opt.state_scales)
    assert opt.group_steps() == [0] and opt.noop.item() == 0
    rep = helpers.Report()
    for k in (2, 3):
        workloads.fresh_grads(shard, k)
        helpers.refresh_grads(osh, shard)
        opt.step()
        oracle.shard_step(osh, capturable=True)
        torch.cuda.synchronize()
        helpers.compare(shard, osh, report=rep)
        _check_scales(opt, osh)
    assert rep.exact_fraction == 1.0
    assert opt.group_steps() == [2]
    assert opt.device_status() == _abi.ETIMEOUT and opt.device_status() == _abi.OK
    opt.close()


def test_scaled_barrier_runs_out_then_the_next_step_is_exact():
    """The first step's wait between the two scaled passes runs out in every
    CTA (diagnostic flag, a plan without the screen): p, m, v, the scales and
    the counter stay as they were.  The absmax slots the first pass filled
    are cleared all the same, so the next step, on fresh gradients, gets
    exactly the oracle's state and new scales (stale maxima would show in
    the scales)."""
    spec, shard, opt, osh, scales = _make("scaled_state_shard", capturable=True,
                                          extra_flags=_abi.TEST_BARRIER_TIMEOUT)
    order = shard.plan_order()
    state = [t.clone() for lst in (shard.params, shard.exp_avgs, shard.exp_avg_sqs)
             for t in (lst[i] for i in order)]
    before = scales.clone()
    opt.step()
    torch.cuda.synchronize()
    after = [t for lst in (shard.params, shard.exp_avgs, shard.exp_avg_sqs)
             for t in (lst[i] for i in order)]
    assert all(torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(after, state))
    assert torch.equal(before, opt.state_scales) and opt.group_steps() == [0]
    assert opt.device_status() == _abi.ETIMEOUT
    workloads.fresh_grads(shard, 2)
    helpers.refresh_grads(osh, shard)
    opt.step()
    oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)
    _check_scales(opt, osh)
    assert rep.exact_fraction == 1.0 and opt.group_steps() == [1]
    assert opt.device_status() == _abi.OK
    opt.close()


def test_graph_replay_equals_eager():
    _, a, oa, _, _ = _make("scaled_state_shard", capturable=True)
    _, b, ob, _, _ = _make("scaled_state_shard", capturable=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ob.step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ob.step()
    for _ in range(3):
        oa.step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x.view(torch.int8), y.view(torch.int8))
    assert torch.equal(oa.state_scales, ob.state_scales)
    oa.close()
    ob.close()


def test_exchange_then_scaled_step():
    """Three ranks' gradients averaged into the shard, then the scaled step,
    in one launch (reduce pass, barrier, absmax pass, barrier, rescale)."""
    spec, shard, opt, osh, _ = _make("scaled_state_shard")
    order = shard.plan_order()
    sizes = [spec.sizes[i] for i in order]
    offs = workloads.exchange_offsets(sizes)
    total = offs[-1] + sizes[-1]
    g_shard = torch.zeros(total, dtype=torch.bfloat16, device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(77)
    padded = (total + 63) // 64 * 64  # rows 128-byte apart
    src = (torch.randn(3, padded, generator=gen, device=DEV) * 1e-2).to(torch.bfloat16)[:, :total]
    groups = shard.param_groups()
    groups[0]["grads"] = [g_shard[o:o + n] for o, n in zip(offs, sizes)]
    scales = shard.state_scales[order].contiguous()
    opt2 = FusedAdamShard(groups, state_scales=scales)
    opt2.set_exchange(g_shard, list(src), average=True)
    opt2.step_reduce()
    osrc = [[helpers.to_np(src[r, o:o + n]) for r in range(3)] for o, n in zip(offs, sizes)]
    for t in osh.tensors:
        t.g = np.zeros(t.p.size, np.uint16)
    oracle.exchange_step(osh, osrc, average=True, capturable=False)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)
    _check_scales(opt2, osh)
    assert rep.exact_fraction == 1.0
    opt2.close()
    opt.close()


def test_scaled_plan_checks():
    # fp32 state cannot be scaled
    spec = workloads.large_uniform(n_tensors=1, numel=4096)
    sh = workloads.materialize(spec, DEV)
    with pytest.raises(FadamError):
        FusedAdamShard(sh.param_groups(), state_scales=torch.ones(1, 3, device=DEV))
    # a scaled plan without its scales refuses to step
    spec2, shard, opt, osh, _ = _make("scaled_bf16")
    bare = FusedAdamShard(shard.param_groups(), extra_flags=_abi.SCALED_STATES)
    with pytest.raises(FadamError):
        bare.step()
    with pytest.raises(ValueError):  # wrong shape
        FusedAdamShard(shard.param_groups(), state_scales=torch.ones(2, 3, device=DEV))
    bare.close()
    opt.close()
