"""GPU parity at the full workload sizes, in the launch configuration the
benchmark uses (default plan: persistent grid sized to the device), over
every element.

The state each tensor starts from is cloned on the device before the GPU
runs all the steps of a workload (gradients that do not change between
steps are only read, so the shard's own serve).  The oracle then replays
the same steps tensor by tensor, each tensor cut into contiguous ranges of
elements (exact, because every element updates independently; the scaled
state, whose rescale needs every new value of a tensor, replays whole
tensors), on a pool of one thread per host core, and every value the GPU
wrote is compared with the oracle's under the parity tolerances (equal
bytes are counted without the tolerance arithmetic).  Each test prints how
many values it compared against how many the shard holds.  The noop step
of the capturable L2 shard is also checked bit-exactly over the whole state
on the GPU, and the step counters over every group.
"""
import os
from concurrent.futures import ThreadPoolExecutor
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"

THREADS = max(1, len(os.sched_getaffinity(0)))
RANGE = 1 << 22  # elements per oracle work unit


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _clone(lst):
    return [None if t is None else t.clone() for t in lst]


def _inputs(shard, grads=None):
    """The state every tensor starts from, as device clones, in the shape
    helpers.oracle_shard reads (param-out is only written, so the shard's
    own buffers serve)."""
    return SimpleNamespace(spec=shard.spec, params=_clone(shard.params),
                           exp_avgs=_clone(shard.exp_avgs), exp_avg_sqs=_clone(shard.exp_avg_sqs),
                           remainders=_clone(shard.remainders), params_out=shard.params_out,
                           grads=shard.grads if grads is None else grads)


def _units(spec, order, whole=False):
    """(tensor, element range) work units: every non-empty tensor in ranges
    of RANGE elements, or whole."""
    out = []
    for i in order:
        n = spec.sizes[i]
        if n == 0:
            continue
        if whole:
            out.append((i, None))
        else:
            out += [(i, slice(a, min(n, a + RANGE))) for a in range(0, n, RANGE)]
    return out


def _replay(shard, init, unit, schedule, capturable):
    """The oracle's steps on one unit, then the comparison with the GPU."""
    i, sl = unit
    elems = None if sl is None else {i: sl}
    osh = helpers.oracle_shard(init, idx=[i], elems=elems)
    for noop in schedule:
        oracle.shard_step(osh, capturable=capturable, noop=noop)
    return helpers.compare(shard, osh, idx=[i], elems=elems)


def _pool_map(fn, units):
    rep = helpers.Report()
    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        for r in ex.map(fn, units):
            rep.merge(r)
    return rep


def _values_per_element(spec):
    """Values the comparison reads per element: p (or the packed master and
    its high half), m, v, and param-out when it is a separate buffer."""
    if spec.remainders:
        return 4
    return 3 + (1 if spec.out_dtype is not None else 0)


def _full_run(spec, steps, inf_step=None, capturable=None, recip_bc=False):
    if capturable is not None:
        spec.capturable = capturable
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=spec.capturable,
                         remainders=spec.remainders, grad_scale=spec.grad_scale, recip_bc=recip_bc)
    init = _inputs(shard)
    t_inf, e_inf = workloads.inf_position(spec) if inf_step else (None, None)
    schedule = []
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
        schedule.append(noop)
    torch.cuda.synchronize()
    steps_dev = opt.group_steps()
    opt.close()
    rep = _pool_map(lambda u: _replay(shard, init, u, schedule, spec.capturable),
                    _units(spec, shard.plan_order()))
    total = _values_per_element(spec) * sum(spec.sizes)
    want_steps = [sum(1 for n in schedule if not n)] * len(spec.groups)
    del shard, init
    _free()
    return rep, total, steps_dev, want_steps


def _report(name, rep, total):
    print(f"{name}: {rep.n} of {total} values compared, {rep.exact} bit-identical, "
          f"worst {rep.worst:.3g} of tolerance")
    assert rep.n == total


def test_large_uniform_full_size():
    # the benchmark's headline path: capturable, device scalars; two steps
    # over all 4,215,275,520 elements
    spec = workloads.large_uniform()
    rep, total, steps, want = _full_run(spec, 2, capturable=True)
    assert steps == want == [2]
    _report("large_uniform", rep, total)


def test_large_uniform_bf16_moments_full_size():
    # the 201-tensor shard with an fp32 master and bf16 moments, capturable
    spec = workloads.large_uniform(moment_dtype=torch.bfloat16)
    rep, total, steps, want = _full_run(spec, 2, capturable=True)
    assert steps == want == [2]
    _report("large_uniform_bf16_moments", rep, total)
    assert rep.exact_fraction == 1.0


def test_large_uniform_bf16_state_full_size():
    # the 201-tensor shard with p, m, v and g in bf16 (IEEE division): every
    # element of two capturable steps, bit for bit in bf16 units
    spec = workloads.large_uniform(state_dtype=torch.bfloat16, g_dtype=torch.bfloat16)
    rep, total, steps, want = _full_run(spec, 2, capturable=True)
    assert steps == want == [2]
    _report("large_uniform_bf16_state", rep, total)
    assert rep.exact_fraction == 1.0


def test_large_uniform_bf16_state_recip_full_size():
    # the benchmark's FADAM_RECIP_BC row: one step over all 4,215,275,520
    # elements, m and v within one bf16 ulp of the oracle's, p under the
    # reciprocal bound (helpers.check_recip_p16)
    spec = workloads.large_uniform(state_dtype=torch.bfloat16, g_dtype=torch.bfloat16)
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, recip_bc=True)
    init = _inputs(shard)
    opt.step()
    torch.cuda.synchronize()
    assert opt.group_steps() == [1]
    opt.close()

    def unit(u):
        i, sl = u
        osh = helpers.oracle_shard(init, idx=[i], elems={i: sl})
        x0 = helpers.unscaled_p(osh, spec.state_dtype)
        oracle.shard_step(osh, capturable=True)
        return helpers.compare_recip(shard, osh, x0, helpers.Report(), idx=[i], elems={i: sl})

    rep = _pool_map(unit, _units(spec, shard.plan_order()))
    _report("large_uniform_bf16_state, reciprocal corrections", rep, 3 * sum(spec.sizes))
    del shard, init
    _free()


def test_capturable_l2_full_size_with_inf_step():
    spec = workloads.capturable_l2()
    rep, total, steps, want = _full_run(spec, 10, inf_step=spec.inf_at_step)
    assert steps == want == [9]
    _report("capturable_l2", rep, total)


def test_remainder_shard_full_size():
    spec = workloads.remainder_shard()
    rep, total, steps, want = _full_run(spec, 10)
    assert steps == want == [10]
    _report("remainder_shard", rep, total)


def test_many_small_full_size():
    spec = workloads.many_small()
    rep, total, steps, want = _full_run(spec, 10)
    assert steps == want == [10, 10, 10]
    _report("many_small", rep, total)


def test_tensor_beyond_2_pow_31_elements():
    n = (1 << 31) + 4099
    spec = workloads.large_uniform(n_tensors=1, numel=n)
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=False)
    init = _inputs(shard)
    opt.step()
    torch.cuda.synchronize()
    info = opt.info()
    assert info["n_elements"] == n and info["n_items"] >= 32
    opt.close()
    rep = _pool_map(lambda u: _replay(shard, init, u, [False], False), _units(spec, [0]))
    _report("one tensor of 2^31 + 4099", rep, 3 * n)
    del shard, init
    _free()


def test_large_uniform_norm_full_size():
    """Squared norm of the 201 x 20,971,520 shard against the oracle run
    tensor by tensor on the host."""
    spec = workloads.large_uniform()
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    got = opt.grad_norm_sq().item()
    with ThreadPoolExecutor(max_workers=THREADS) as ex:
        parts = list(ex.map(lambda g: oracle.sumsq(helpers.to_np(g), oracle.DT_F32), shard.grads))
    assert got == pytest.approx(sum(parts), rel=2e-6)
    opt.close()
    del shard, opt
    _free()


def test_exchange_shard_full_size():
    """Eight ranks' bf16 gradients averaged into the 1.2e9-element shard,
    param-out to the seven other ranks' places, two steps of two
    micro-batches each: the first reduce-scatter writes the shard, the
    second (the ranks' buffers in another order) adds to it fused with the
    step.  Every element against the oracle (the reduced gradient bit for
    bit), destinations byte-equal over the whole shard."""
    spec = workloads.exchange_versions(full=True)["exchange_shard"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    R = spec.exchange_ranks
    srcs = list(shard.sources)

    def micro_batch(k, accumulate):
        opt.set_exchange(shard.buckets["g"], srcs[k:] + srcs[:k], average=True,
                         out_shard=shard.buckets["p_out"], dests=list(shard.dests),
                         accumulate=accumulate)

    init = _inputs(shard)
    for _ in range(2):
        micro_batch(0, False)
        opt.grad_reduce()
        micro_batch(1, True)
        opt.step_reduce()
    torch.cuda.synchronize()
    assert opt.group_steps() == [2]
    opt.close()

    def unit(u):
        i, sl = u
        a = shard.offsets[i] + sl.start
        b = shard.offsets[i] + sl.stop
        raw = [helpers.to_np(shard.sources[r][a:b]) for r in range(R)]
        src0, src1 = [raw], [raw[1:] + raw[:1]]
        osh = helpers.oracle_shard(init, idx=[i], elems={i: sl})
        t = osh.tensors[0]
        for _ in range(2):
            t.g[...] = oracle.reduce_into(t.g, src0[0], t.g_dtype, True, False)
            oracle.exchange_step(osh, src1, average=True, capturable=True, accumulate=True)
        got = helpers.to_np(shard.grads[i][sl])
        assert got.tobytes() == t.g.tobytes(), f"tensor {i}: reduced gradient differs"
        return helpers.compare(shard, osh, idx=[i], elems={i: sl})

    rep = _pool_map(unit, _units(spec, shard.plan_order()))
    _report("exchange_shard", rep, 4 * sum(spec.sizes))
    assert rep.exact_fraction == 1.0
    out = shard.buckets["p_out"].view(torch.int16)
    for d in range(spec.exchange_dests):
        assert torch.equal(shard.dests[d].view(torch.int16), out), f"destination {d}"
    del shard, init
    _free()


def test_scaled_state_recip_full_size():
    """The benchmark's scaled-state row with FADAM_RECIP_BC: one step, every
    element of every tensor: m and v within one fp16 ulp, p and the bf16
    param-out under the reciprocal bound (helpers.check_recip_p16, values
    after the scales), every scale within 2e-6 relative."""
    spec = workloads.scaled_versions(full=True)["scaled_state_shard"]
    shard = workloads.materialize(spec, DEV)
    order = shard.plan_order()
    scales = shard.state_scales[order].contiguous()
    scales0 = scales.clone()
    opt = FusedAdamShard(shard.param_groups(), state_scales=scales, recip_bc=True)
    init = _inputs(shard)
    opt.step()
    torch.cuda.synchronize()
    assert opt.group_steps() == [1]
    opt.close()
    got_scales = helpers.to_np(scales).astype(np.float64)
    pos = {i: k for k, i in enumerate(order)}

    def unit(u):
        i, _ = u
        k = pos[i]
        osh = helpers.oracle_shard(init, idx=[i], scales=scales0[k:k + 1])
        x0 = helpers.unscaled_p(osh, spec.state_dtype)
        oracle.shard_step(osh, capturable=False)
        want = osh.tensors[0].scales.astype(np.float64)
        assert np.all(np.abs(got_scales[k] - want) <= 2e-6 * np.abs(want)), (i, got_scales[k], want)
        return helpers.compare_recip(shard, osh, x0, helpers.Report(), idx=[i],
                                     got_scales=got_scales[k:k + 1])

    rep = _pool_map(unit, _units(spec, order, whole=True))
    _report("scaled_state_shard, reciprocal corrections", rep,
            _values_per_element(spec) * sum(spec.sizes))
    del shard, init
    _free()


def test_scaled_state_full_size():
    """The 1.2e9-element fp16 scaled-state shard, two regular steps with
    fresh gradients for the second.  The rescale depends on every element
    of a tensor, so the oracle replays whole tensors: every element of every
    tensor, and every tensor's scales, bit for bit."""
    spec = workloads.scaled_versions(full=True)["scaled_state_shard"]
    shard = workloads.materialize(spec, DEV)
    order = shard.plan_order()
    scales = shard.state_scales[order].contiguous()
    scales0 = scales.clone()
    opt = FusedAdamShard(shard.param_groups(), state_scales=scales)
    init = _inputs(shard, grads=_clone(shard.grads))
    opt.step()
    workloads.fresh_grads(shard, 2)
    opt.step()
    torch.cuda.synchronize()
    assert opt.group_steps() == [2]
    opt.close()
    got_scales = helpers.to_np(scales)
    pos = {i: k for k, i in enumerate(order)}

    def unit(u):
        i, _ = u
        k = pos[i]
        osh = helpers.oracle_shard(init, idx=[i], scales=scales0[k:k + 1])
        oracle.shard_step(osh, capturable=False)
        osh.tensors[0].g = helpers.to_np(shard.grads[i])
        oracle.shard_step(osh, capturable=False)
        assert got_scales[k].tobytes() == osh.tensors[0].scales.tobytes(), i
        return helpers.compare(shard, osh, idx=[i])

    rep = _pool_map(unit, _units(spec, order, whole=True))
    _report("scaled_state_shard", rep, _values_per_element(spec) * sum(spec.sizes))
    assert rep.exact_fraction == 1.0
    del shard, init
    _free()
