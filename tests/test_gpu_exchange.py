"""GPU parity of the data-parallel exchange stand-in (fadam_plan_set_exchange,
fadam_grad_reduce, fadam_step_reduce) against the oracle: the reduced
gradient shard bit for bit, the fused step element by element, the
param-out copies in every destination, a set noop flag, the inf/nan screen
of the reduced gradient, graph replay, the norm of the reduced shard, and the
argument checks."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard
from adamw_optimizer_step_persistent_gb300._abi import FadamError
from tests import helpers

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAMES = ["exchange_shard", "exchange_packed_sum"]


def _make(name, capturable=True, check_finite=False):
    spec = workloads.exchange_versions()[name]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=capturable, check_finite=check_finite)
    opt.set_exchange(shard.buckets["g"], list(shard.sources), average=spec.exchange_average,
                     out_shard=shard.buckets["p_out"], dests=list(shard.dests))
    return spec, shard, opt


def _oracle_sources(shard, idx=None):
    """Per tensor (plan order): the R ranks' contributions to its fragment."""
    idx = shard.plan_order() if idx is None else idx
    out = []
    for i in idx:
        o, n = shard.offsets[i], shard.spec.sizes[i]
        out.append([helpers.to_np(shard.sources[r, o:o + n]) for r in range(shard.sources.shape[0])])
    return out


def _check_reduced(shard, osh):
    """The reduced shard bit for bit (any two NaNs alike: their payloads
    are not compared)."""
    for t, i in zip(osh.tensors, shard.plan_order()):
        got = helpers.to_np(shard.grads[i])
        if got.tobytes() == t.g.tobytes():
            continue
        dt = shard.grads[i].dtype
        if dt == torch.float32:
            nan = np.isnan(got) & np.isnan(t.g)
        else:
            nan = np.isnan(helpers.widen16(got, dt)) & np.isnan(helpers.widen16(t.g, dt))
        assert ((got == t.g) | nan).all(), f"tensor {i}: reduced gradient differs"


def _check_dests(shard):
    o = shard.buckets["p_out"]
    for d in range(shard.dests.shape[0]):
        assert torch.equal(shard.dests[d].view(torch.int16), o.view(torch.int16)), f"destination {d}"


@pytest.mark.parametrize("capturable", [True, False])
@pytest.mark.parametrize("name", NAMES)
def test_step_reduce_matches_oracle(name, capturable):
    spec, shard, opt = _make(name, capturable=capturable)
    osh = helpers.oracle_shard(shard)
    src = _oracle_sources(shard)
    rep = helpers.Report()
    for k in range(3):
        opt.step_reduce()
        oracle.exchange_step(osh, src, average=spec.exchange_average, capturable=capturable)
        torch.cuda.synchronize()
        _check_reduced(shard, osh)
        helpers.compare(shard, osh, report=rep)
        _check_dests(shard)
        # the next step's contributions: rank r's buffer rolled by one rank
        shard.sources.copy_(torch.roll(shard.sources, 1, dims=0))
        src = _oracle_sources(shard)
    assert opt.group_steps() == [3]
    assert rep.exact_fraction == 1.0, rep.exact_fraction
    opt.close()


@pytest.mark.parametrize("name", NAMES)
def test_grad_reduce_alone_touches_only_g(name):
    spec, shard, opt = _make(name)
    snap = helpers.snapshot(shard)
    dests = shard.dests.clone()
    opt.grad_reduce()
    torch.cuda.synchronize()
    osh = helpers.oracle_shard(shard)
    for t, s in zip(osh.tensors, _oracle_sources(shard)):
        t.g[...] = oracle.reduce_sources(s, oracle.DT_BF16, spec.exchange_average)
    _check_reduced(shard, osh)
    assert helpers.state_equal(shard, snap)
    assert torch.equal(dests, shard.dests)
    assert opt.group_steps() == [0]
    opt.close()


def test_noop_still_reduces():
    spec, shard, opt = _make("exchange_shard")
    snap = helpers.snapshot(shard)
    opt.noop.fill_(1)
    opt.step_reduce()
    torch.cuda.synchronize()
    osh = helpers.oracle_shard(shard)
    assert oracle.exchange_step(osh, _oracle_sources(shard), average=True, capturable=True, noop=True)
    _check_reduced(shard, osh)
    assert helpers.state_equal(shard, snap)
    assert opt.group_steps() == [0]
    opt.close()


@pytest.mark.parametrize("name", NAMES)
def test_screen_of_the_reduced_gradient(name):
    spec, shard, opt = _make(name, check_finite=True)
    opt.step_reduce()  # finite: one step applied
    torch.cuda.synchronize()
    assert opt.noop.item() == 0 and opt.group_steps() == [1]
    snap = helpers.snapshot(shard)
    # an inf in one rank's contribution, in a fragment's tail element
    i = shard.plan_order()[-1]
    shard.sources[1, shard.offsets[i] + spec.sizes[i] - 1] = float("inf")
    opt.step_reduce()
    torch.cuda.synchronize()
    assert opt.noop.item() == 1 and opt.group_steps() == [1]
    assert helpers.state_equal(shard, snap)
    assert torch.isinf(shard.grads[i][-1].float())
    opt.close()


def test_graph_replay_equals_eager():
    spec, a, oa = _make("exchange_shard")
    _, b, ob = _make("exchange_shard")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ob.step_reduce()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ob.step_reduce()
    for _ in range(4):
        oa.step_reduce()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x.view(torch.int8), y.view(torch.int8))
    assert torch.equal(a.dests, b.dests) and oa.group_steps() == ob.group_steps() == [4]
    oa.close()
    ob.close()


def test_norm_of_the_reduced_shard():
    spec, shard, opt = _make("exchange_shard")
    opt.grad_reduce()
    got = opt.grad_norm_sq().item()
    osh = helpers.oracle_shard(shard)
    want = oracle.shard_sumsq(osh)
    assert got == pytest.approx(want, rel=2e-6)
    opt.close()


@pytest.mark.parametrize("case", ["inf", "nan", "overflow"])
def test_reduce_special_values(case):
    """An infinity or NaN in one rank's contribution, and contributions
    whose float sum overflows, reach the reduced shard as the oracle's
    reduction gives them (a NaN's payload aside: the GPU writes its own)."""
    spec, shard, opt = _make("exchange_shard")
    i = shard.plan_order()[2]
    o = shard.offsets[i]
    if case == "inf":
        shard.sources[2, o + 5] = float("inf")
    elif case == "nan":
        shard.sources[1, o + 77] = float("nan")
    else:
        shard.sources[:, o:o + 3000] = 2e38
    osh = helpers.oracle_shard(shard)
    for t, src in zip(osh.tensors, _oracle_sources(shard)):
        t.g[...] = oracle.reduce_into(t.g, src, t.g_dtype, spec.exchange_average, False)
    opt.grad_reduce()
    torch.cuda.synchronize()
    _check_reduced(shard, osh)
    g = shard.grads[i].float()
    if case == "nan":
        assert torch.isnan(g[77])
    else:
        assert torch.isinf(g[5] if case == "inf" else g[0])
    opt.close()


def test_plain_step_writes_destinations():
    spec, shard, opt = _make("exchange_packed_sum")
    opt.step()  # no reduction: g as it stands (zeros), param-out to every destination
    torch.cuda.synchronize()
    _check_dests(shard)
    assert shard.buckets["p_out"].abs().sum().item() > 0
    opt.close()


def test_exchange_argument_checks():
    spec, shard, opt = _make("exchange_shard")
    g = shard.buckets["g"]
    with pytest.raises(ValueError):  # a source smaller than the shard
        opt.set_exchange(g, [shard.sources[0, :10]])
    with pytest.raises(FadamError):  # 17 sources
        opt.set_exchange(g, [shard.sources[0]] * 17)
    with pytest.raises(FadamError):  # a source start 2 bytes off
        opt.set_exchange(g, [shard.sources.reshape(-1)[1:1 + g.numel()]])
    with pytest.raises(ValueError):
        opt.set_exchange(g, [shard.sources[0]], dests=[shard.dests[0]])  # dests without out_shard
    opt.set_exchange(g, [])  # no exchange: the reduce entry points refuse
    with pytest.raises(FadamError):
        opt.grad_reduce()
    with pytest.raises(FadamError):
        opt.step_reduce()
    opt.close()
    # destinations on a plan without a param-out copy
    lspec = workloads.large_uniform(n_tensors=1, numel=4096)
    lsh = workloads.materialize(lspec, DEV)
    lopt = FusedAdamShard(lsh.param_groups(), capturable=True)
    with pytest.raises(FadamError):
        out = torch.zeros(4096, dtype=torch.bfloat16, device=DEV)
        lopt.set_exchange(lsh.grads[0], [], out_shard=out, dests=[out.clone()])
    lopt.close()


@pytest.mark.parametrize("ranks,average", [(2, True), (4, False), (8, True), (7, True)])
def test_unrolled_and_generic_reduce_tiles(ranks, average):
    # 2, 4 and 8 sources take the reduce tiles unrolled for that count, 7 the
    # generic loop; each sums in rank order and gives the oracle's shard
    # bit for bit, and the fused step the oracle's state
    spec = workloads.exchange_shard(layers=1, hidden=256, ffn=688, ranks=ranks, dests=1)
    spec.exchange_average = average
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    opt.set_exchange(shard.buckets["g"], list(shard.sources), average=average,
                     out_shard=shard.buckets["p_out"], dests=list(shard.dests))
    osh = helpers.oracle_shard(shard)
    src = _oracle_sources(shard)
    for _ in range(2):
        opt.step_reduce()
        oracle.exchange_step(osh, src, average=average, capturable=True)
    torch.cuda.synchronize()
    _check_reduced(shard, osh)
    rep = helpers.compare(shard, osh)
    _check_dests(shard)
    assert rep.exact_fraction == 1.0
    opt.close()


@pytest.mark.parametrize("accumulate", [False, True])
def test_sixteen_sources_and_sixteen_destinations(accumulate):
    """The exchange at its limits (FADAM_MAX_SOURCES, FADAM_MAX_DESTS): 16
    ranks' slices through the generic reduce loop (17 slices per tile when
    the shard's old g is added to them), param-out written to 16
    destinations; the reduced shard bit for bit, the state and every
    destination against the oracle over two steps."""
    spec = workloads.exchange_shard(layers=1, hidden=256, ffn=688, ranks=16, dests=16)
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True)
    opt.set_exchange(shard.buckets["g"], list(shard.sources), average=spec.exchange_average,
                     out_shard=shard.buckets["p_out"], dests=list(shard.dests),
                     accumulate=accumulate)
    osh = helpers.oracle_shard(shard)
    src = _oracle_sources(shard)
    rep = helpers.Report()
    for _ in range(2):
        opt.step_reduce()
        oracle.exchange_step(osh, src, average=spec.exchange_average, capturable=True,
                             accumulate=accumulate)
        torch.cuda.synchronize()
        _check_reduced(shard, osh)
        helpers.compare(shard, osh, report=rep)
        _check_dests(shard)
    assert shard.dests.shape[0] == 16 and shard.sources.shape[0] == 16
    assert rep.exact_fraction == 1.0, rep.exact_fraction
    assert opt.group_steps() == [2]
    opt.close()


def _rotated(shard, k):
    """The ranks' buffers in rank order rotated by k: each micro-batch's
    contributions arrive in another order, so their sums differ."""
    src = list(shard.sources)
    k %= len(src)
    return src[k:] + src[:k]


def _set_micro_batch(opt, shard, spec, k, accumulate):
    opt.set_exchange(shard.buckets["g"], _rotated(shard, k), average=spec.exchange_average,
                     out_shard=shard.buckets["p_out"], dests=list(shard.dests),
                     accumulate=accumulate)


def _oracle_micro_batch(shard, k):
    """Per tensor: the rotated ranks' contributions to its fragment."""
    out = []
    R = shard.sources.shape[0]
    for i in shard.plan_order():
        o, n = shard.offsets[i], shard.spec.sizes[i]
        out.append([helpers.to_np(shard.sources[(r + k) % R, o:o + n]) for r in range(R)])
    return out


@pytest.mark.parametrize("name", NAMES)
def test_gradient_accumulation_over_three_micro_batches(name):
    """Two steps of three micro-batches each: the first reduce-scatter of a
    step writes the shard, the second adds to it (fadam_grad_reduce with
    FADAM_EXCHANGE_ACCUMULATE), the third adds to it fused with the step
    (fadam_step_reduce).  The shard's g bit for bit after every micro-batch,
    the state and every destination against the oracle after each step."""
    spec, shard, opt = _make(name)
    osh = helpers.oracle_shard(shard)
    rep = helpers.Report()
    k = 0
    for step in range(2):
        for mb in range(3):
            _set_micro_batch(opt, shard, spec, k, accumulate=mb > 0)
            src = _oracle_micro_batch(shard, k)
            if mb < 2:
                opt.grad_reduce()
                for t, s in zip(osh.tensors, src):
                    t.g[...] = oracle.reduce_into(t.g, s, t.g_dtype, spec.exchange_average, mb > 0)
            else:
                opt.step_reduce()
                oracle.exchange_step(osh, src, average=spec.exchange_average, capturable=True,
                                     accumulate=True)
            torch.cuda.synchronize()
            _check_reduced(shard, osh)
            k += 1
        helpers.compare(shard, osh, report=rep)
        _check_dests(shard)
    assert opt.group_steps() == [2]
    assert rep.exact_fraction == 1.0, rep.exact_fraction
    opt.close()


def test_screen_sees_an_inf_that_arrives_by_accumulation():
    """The first micro-batch is finite; the second carries an inf in one
    rank's contribution: the accumulated shard holds the inf, the fused step
    is skipped, and the state is left as it was."""
    spec, shard, opt = _make("exchange_shard", check_finite=True)
    _set_micro_batch(opt, shard, spec, 0, accumulate=False)
    opt.grad_reduce()
    i = shard.plan_order()[2]
    shard.sources[2, shard.offsets[i] + 5] = float("inf")
    _set_micro_batch(opt, shard, spec, 1, accumulate=True)
    snap = helpers.snapshot(shard)
    opt.step_reduce()
    torch.cuda.synchronize()
    assert opt.noop.item() == 1 and opt.group_steps() == [0]
    assert helpers.state_equal(shard, snap)
    assert torch.isinf(shard.grads[i][5].float())
    opt.close()


def test_accumulating_step_captured_in_one_graph():
    """A whole step of two micro-batches (the flags switched on the host
    between the captured launches, which keep the flags they were captured
    with) replayed three times equals three eager steps."""
    spec, a, oa = _make("exchange_shard")
    _, b, ob = _make("exchange_shard")

    def step(opt, shard):
        _set_micro_batch(opt, shard, spec, 0, accumulate=False)
        opt.grad_reduce()
        _set_micro_batch(opt, shard, spec, 1, accumulate=True)
        opt.step_reduce()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(ob, b)
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(ob, b)
    for _ in range(4):
        step(oa, a)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x.view(torch.int8), y.view(torch.int8))
    assert torch.equal(a.buckets["g"], b.buckets["g"]) and torch.equal(a.dests, b.dests)
    assert oa.group_steps() == ob.group_steps() == [4]
    oa.close()
    ob.close()


def test_unknown_reduce_flag_bits_are_refused():
    spec, shard, opt = _make("exchange_shard")
    from adamw_optimizer_step_persistent_gb300 import _abi
    import ctypes
    src = (ctypes.c_void_p * 1)(shard.sources[0].data_ptr())
    st = _abi.lib().fadam_plan_set_exchange(opt._plan, shard.buckets["g"].data_ptr(), src, 1, 4,
                                            None, None, 0)
    assert st == _abi.EINVAL and b"reduce_flags" in _abi.lib().fadam_last_error()
    opt.close()
