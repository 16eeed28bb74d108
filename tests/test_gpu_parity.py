"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small versions of the five shard recipes, element by element over every
tensor, several steps each, plus the edge cases: ragged and empty tensors,
misaligned views, aliasing param-out, every grad/param-out dtype, noop and
inf screens, shared and per-group step counters, graph replay, one-shot and
host-gradient entry points.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from adamw_optimizer_step_persistent_gb300 import FusedAdamShard, _abi, step_once
from tests import helpers

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(spec, steps, *, capturable=None, check_finite=False, fresh=True, shared_step=False,
         start_step=0):
    """Run `steps` steps on the GPU and on the oracle from the same inputs
    (every group's counter starting at `start_step` steps taken)."""
    capturable = spec.capturable if capturable is None else capturable
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=capturable, check_finite=check_finite,
                         remainders=spec.remainders, grad_scale=spec.grad_scale,
                         shared_step=shared_step)
    osh = helpers.oracle_shard(shard, step_slot=[0] * len(spec.groups) if shared_step else None)
    if start_step:
        opt.set_group_steps([start_step] * len(spec.groups))
        osh.steps = [start_step] * len(osh.steps)
    for k in range(1, steps + 1):
        if fresh and k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard)
        opt.step()
        oracle.shard_step(osh, capturable=capturable)
    torch.cuda.synchronize()
    return shard, opt, osh


@pytest.mark.parametrize("name", ["tiny_adamw", "capturable_l2", "large_uniform",
                                  "remainder_shard", "many_small"])
def test_small_shards_match_oracle(name):
    spec = workloads.small_versions()[name]
    steps = 10  # the tolerance is stated for the state after ten steps
    shard, opt, osh = _run(spec, steps)
    rep = helpers.compare(shard, osh)
    assert opt.group_steps() == oracle.group_steps(osh) == [steps] * len(spec.groups)
    print(f"{name}: {rep.n} values, {rep.exact_fraction:.6f} bit-identical, "
          f"worst {rep.worst:.3g} of tolerance")


@pytest.mark.parametrize("name", ["tiny_adamw", "many_small"])
def test_regular_and_capturable_are_bit_identical(name):
    spec = workloads.small_versions()[name]
    a, _, _ = _run(spec, 4, capturable=False)
    b, opt_b, _ = _run(spec, 4, capturable=True)
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y)
    assert opt_b.group_steps() == [4] * len(spec.groups)


def test_check_finite_without_inf_matches_plain_capturable():
    spec = workloads.small_versions()["many_small"]
    a, _, _ = _run(spec, 3, capturable=True)
    b, opt_b, _ = _run(spec, 3, capturable=True, check_finite=True)
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x, y)
    assert opt_b.noop.item() == 0 and opt_b.device_status() == 0


@pytest.mark.parametrize("screen", ["upstream_flag", "in_kernel_check"])
def test_inf_gradient_skips_the_step_bit_exactly(screen):
    """capturable L2 shard, bf16 grads and param-out: the step whose grads
    hold a +inf changes nothing and does not advance the counter."""
    spec = workloads.small_versions()["capturable_l2"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True,
                         check_finite=(screen == "in_kernel_check"), grad_scale=spec.grad_scale)
    osh = helpers.oracle_shard(shard)
    t_inf, e_inf = workloads.inf_position(spec)
    for k in range(1, 6):
        if k > 1:
            workloads.fresh_grads(shard, k)
            helpers.refresh_grads(osh, shard)
        inject = k == spec.inf_at_step
        if inject:
            shard.grads[t_inf][e_inf] = float("inf")
            before = helpers.snapshot(shard)
            if screen == "upstream_flag":  # as the page's step(): found_inf copied to the flag
                opt.noop.copy_(torch.isinf(shard.grads[t_inf]).any().to(torch.int32).view(1))
        opt.step()
        torch.cuda.synchronize()
        if inject:
            assert opt.noop.item() == 1
            assert helpers.state_equal(shard, before)
            assert opt.group_steps() == [k - 1]
            oracle.shard_step(osh, capturable=True, noop=True)
            opt.noop.zero_()
        else:
            oracle.shard_step(osh, capturable=True)
    rep = helpers.compare(shard, osh)
    assert opt.group_steps() == oracle.group_steps(osh) == [4]
    assert rep.n > 0


def test_graph_replay_matches_eager():
    spec = workloads.small_versions()["many_small"]
    a = workloads.materialize(spec, DEV)
    b = workloads.materialize(spec, DEV)
    oa = FusedAdamShard(a.param_groups(), capturable=True)
    ob = FusedAdamShard(b.param_groups(), capturable=True)
    for _ in range(3):
        oa.step()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ob.step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ob.step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x, y)
    assert ob.group_steps() == oa.group_steps() == [3, 3, 3]


@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out_dtype", [None, torch.float32, torch.bfloat16, torch.float16])
def test_dtype_combinations(g_dtype, out_dtype):
    spec = workloads.large_uniform(n_tensors=3, numel=40_003)
    spec.g_dtype, spec.out_dtype = g_dtype, out_dtype
    shard, _, osh = _run(spec, 3, capturable=False)
    helpers.compare(shard, osh)


def _custom_shard(sizes, offsets_p, offsets_mvg, group_of, groups, out_alias=False,
                  out_dtype=None):
    """Tensors as views at chosen element offsets into fresh buffers."""
    spec = workloads.ShardSpec("custom", groups, list(sizes), list(group_of), out_dtype=out_dtype,
                               seed=99)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(99)
    P, M, V, G, O = [], [], [], [], []
    for n, op, oq in zip(sizes, offsets_p, offsets_mvg):
        bp = torch.randn(n + op, generator=gen, device=DEV)
        bm = torch.zeros(n + oq, device=DEV)
        bv = torch.zeros(n + oq, device=DEV)
        bg = torch.randn(n + oq, generator=gen, device=DEV) * 1e-3
        P.append(bp[op:op + n])
        M.append(bm[oq:oq + n])
        V.append(bv[oq:oq + n])
        G.append(bg[oq:oq + n])
        if out_alias:
            O.append(P[-1])
        elif out_dtype is not None:
            O.append(torch.zeros(n + op, dtype=out_dtype, device=DEV)[op:op + n])
        else:
            O.append(None)
    return workloads.Shard(spec, P, M, V, G, O, [None] * len(sizes))


def test_ragged_empty_and_misaligned_views():
    g = workloads.GroupSpec(adam_w_mode=True, weight_decay=0.05, betas=(0.9, 0.95))
    sizes = [0, 1, 3, 4, 5, 31, 1000, 4097, 70001, 0, 65536]
    offs_p = [0, 1, 2, 3, 1, 0, 5, 3, 1, 0, 2]      # same residue as m, v, g: peeled head
    offs_q = [0, 1, 2, 3, 2, 1, 5, 0, 1, 0, 2]      # some differ: whole tensor scalar
    shard = _custom_shard(sizes, offs_p, offs_q, [0] * len(sizes), [g], out_dtype=torch.bfloat16)
    opt = FusedAdamShard(shard.param_groups(), capturable=False)
    osh = helpers.oracle_shard(shard)
    for k in range(1, 4):
        opt.step()
        oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    helpers.compare(shard, osh)


def test_param_out_aliasing_the_master():
    g = workloads.GroupSpec(adam_w_mode=False, weight_decay=0.1)
    shard = _custom_shard([1234, 50000], [0, 0], [0, 0], [0, 0], [g], out_alias=True,
                          out_dtype=torch.float32)
    opt = FusedAdamShard(shard.param_groups(), capturable=False)
    osh = helpers.oracle_shard(shard)
    for t in osh.tensors:
        t.p_out = t.p
    for _ in range(3):
        opt.step()
        oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    helpers.compare(shard, osh)
    info = opt.info()
    assert info["bytes_per_step"] == (1234 + 50000) * 28.0  # the alias is one stream


def test_bias_correction_off_and_mixed_modes():
    groups = [workloads.GroupSpec(adam_w_mode=True, weight_decay=0.1, bias_correction=False),
              workloads.GroupSpec(adam_w_mode=False, weight_decay=0.1, bias_correction=True,
                                  betas=(0.8, 0.9)),
              workloads.GroupSpec(adam_w_mode=True, weight_decay=0.0, eps=1e-6)]
    sizes = [5000, 777, 4096, 3, 100_000]
    shard = _custom_shard(sizes, [0] * 5, [0] * 5, [0, 1, 2, 0, 1], groups)
    for cap in (False, True):
        sh = _custom_shard(sizes, [0] * 5, [0] * 5, [0, 1, 2, 0, 1], groups)
        opt = FusedAdamShard(sh.param_groups(), capturable=cap)
        osh = helpers.oracle_shard(sh)
        for _ in range(4):
            opt.step()
            oracle.shard_step(osh, capturable=cap)
        torch.cuda.synchronize()
        helpers.compare(sh, osh)
        assert opt.group_steps() == [4, 4, 4]
    del shard


def test_shared_step_counter_advances_once():
    spec = workloads.small_versions()["many_small"]
    shard, opt, osh = _run(spec, 3, shared_step=True)
    helpers.compare(shard, osh)
    assert opt.group_steps() == [3, 3, 3]
    assert opt.step_dev[0].data_ptr() == opt.step_dev[2].data_ptr()


def test_step_preadvanced_uses_counter_as_is():
    spec = workloads.small_versions()["tiny_adamw"]
    a, _, _ = _run(spec, 2, capturable=True, fresh=False)
    b = workloads.materialize(spec, DEV)
    ob = FusedAdamShard(b.param_groups(), capturable=True, step_preadvanced=True)
    for k in (1, 2):
        for s in ob.step_dev:
            s.fill_(k)  # the caller advances, as the page's step() does
        ob.step()
    torch.cuda.synchronize()
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x, y)
    assert ob.group_steps() == [2, 2]


def test_all_empty_plan_still_advances_capturable_steps():
    groups = [dict(params=[], exp_avgs=[], exp_avg_sqs=[], grads=[], lr=1e-3) for _ in range(3)]
    opt = FusedAdamShard(groups, capturable=True)
    for _ in range(3):
        opt.step()
    torch.cuda.synchronize()
    assert opt.group_steps() == [3, 3, 3]
    reg = FusedAdamShard(groups, capturable=False)
    for _ in range(3):
        reg.step()
    assert reg.group_steps() == [3, 3, 3]


def test_step_once_regular_and_capturable():
    spec = workloads.large_uniform(n_tensors=3, numel=10_007)
    for cap in (False, True):
        shard = workloads.materialize(spec, DEV)
        osh = helpers.oracle_shard(shard)
        g = spec.groups[0]
        lr_dev = torch.tensor([g.lr], device=DEV) if cap else None
        step_dev = torch.zeros(1, dtype=torch.int32, device=DEV) if cap else None
        gs_dev = torch.tensor([1.0], device=DEV) if cap else None
        for k in (1, 2):
            step_once(shard.params, shard.exp_avgs, shard.exp_avg_sqs, shard.grads, lr=g.lr,
                      betas=g.betas, eps=g.eps, weight_decay=g.weight_decay, step=k,
                      lr_dev=lr_dev, step_dev=step_dev, grad_scale_dev=gs_dev)
            oracle.shard_step(osh, capturable=cap)
        torch.cuda.synchronize()
        helpers.compare(shard, osh)
        if cap:
            assert step_dev.item() == 2


@pytest.mark.parametrize("name", ["capturable_l2", "remainder_shard", "many_small"])
def test_host_gradients_entry_point_matches_device_gradients(name):
    """Pinned host gradients are read in place (zero copy) by every item
    form: bf16 grads with a param-out copy, the remainder form, and the
    many-small shard's ragged and unaligned tensors."""
    spec = workloads.small_versions()[name]
    a, _, _ = _run(spec, 2, capturable=True, fresh=False)
    b = workloads.materialize(spec, DEV)
    ob = FusedAdamShard(b.param_groups(), capturable=True, grad_scale=spec.grad_scale,
                        remainders=spec.remainders)
    host = [g.cpu().pin_memory() for g in (b.grads[i] for i in b.plan_order())]
    for gr in b.grads:
        gr.zero_()  # the host copy is the only source of the grads
    steps = [ob.step_from_host(host) for _ in range(2)]
    assert steps == [[1] * len(spec.groups), [2] * len(spec.groups)]
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x, y)


@pytest.mark.parametrize("state_dtype,start", [(torch.float32, 0), (torch.bfloat16, 0),
                                               (torch.bfloat16, 20000)])
def test_largest_group_table_each_group_its_own_hyperparameters(state_dtype, start):
    """32 groups (the most a plan takes), each with its own mode, betas,
    eps, weight decay, lr and bias correction, two of them empty, ragged
    tensors of 1 to 70,000 elements: every value equals the oracle bit for
    bit and every counter advances, regular and capturable.  20,000 steps
    in, some groups' bias corrections are 1 and others' not (beta2 up to
    0.9999), so the 16-bit state's launch-wide choice of update loop must
    keep the divisions that any group needs."""
    rng = np.random.default_rng(5)
    groups = [workloads.GroupSpec(adam_w_mode=bool(k % 2), lr=float(10 ** rng.uniform(-4, -2)),
                                  betas=(float(rng.uniform(0.8, 0.95)),
                                         float(rng.uniform(0.95, 0.9999))),
                                  eps=float(10 ** rng.uniform(-10, -6)),
                                  weight_decay=float(rng.uniform(0.0, 0.2)),
                                  bias_correction=k % 5 != 0)
              for k in range(_abi.MAX_GROUPS)]
    for k in (3, 11):  # beta2 near 1: bias correction 2 stays below 1 long after step 20,000
        groups[k].betas = (groups[k].betas[0], 0.9999)
    sizes, group_of = [], []
    for k in range(_abi.MAX_GROUPS):
        if k in (7, 19):
            continue  # empty groups
        for _ in range(1 + k % 3):
            sizes.append(int(rng.integers(1, 70_000)))
            group_of.append(k)
    spec = workloads.ShardSpec("groups32", groups, sizes, group_of, g_dtype=torch.bfloat16,
                               out_dtype=torch.bfloat16, grad_std=1e-2, seed=1300,
                               state_dtype=state_dtype)
    if start:
        unit2 = [not g.bias_correction or oracle.bias_correction(g.betas[1], start + 1) == 1.0
                 for g in groups]
        assert any(unit2) and not all(unit2)
    for capturable in (False, True):
        shard, opt, osh = _run(spec, 3, capturable=capturable, start_step=start)
        rep = helpers.compare(shard, osh)
        assert rep.exact_fraction == 1.0, rep.exact_fraction
        assert opt.group_steps() == oracle.group_steps(osh) == [start + 3] * _abi.MAX_GROUPS
        opt.close()


@pytest.mark.parametrize("form", ["bf16_state", "f16_state", "bf16_moments", "f16_moments"])
def test_host_gradients_in_the_16bit_forms(form):
    """The in-place host-gradient path with a 16-bit state or 16-bit
    moments, over the many-small shard's ragged and unaligned tensors:
    the same bits as two steps with the gradients on the device."""
    spec = workloads.small_versions()["many_small"]
    dt = torch.bfloat16 if form.startswith("bf16") else torch.float16
    if form.endswith("state"):
        spec.state_dtype = dt
    else:
        spec.moment_dtype = dt
    a, _, _ = _run(spec, 2, capturable=True, fresh=False)
    b = workloads.materialize(spec, DEV)
    ob = FusedAdamShard(b.param_groups(), capturable=True, grad_scale=spec.grad_scale)
    host = [g.cpu().pin_memory() for g in (b.grads[i] for i in b.plan_order())]
    for gr in b.grads:
        gr.zero_()
    steps = [ob.step_from_host(host) for _ in range(2)]
    assert steps == [[1] * len(spec.groups), [2] * len(spec.groups)]
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32),
                           y.view(torch.int16) if y.element_size() == 2 else y.view(torch.int32))
    ob.close()


@pytest.mark.parametrize("memory", ["pageable", "misaligned_pinned"])
def test_host_gradients_copy_path(memory):
    """Host gradients that cannot be read in place (pageable, or pinned at
    another 16-byte alignment than the device gradient) are copied in
    first; the result is the same, and the device gradients hold them."""
    spec = workloads.small_versions()["capturable_l2"]
    a, _, _ = _run(spec, 2, fresh=False)
    b = workloads.materialize(spec, DEV)
    ob = FusedAdamShard(b.param_groups(), capturable=True, grad_scale=spec.grad_scale)
    if memory == "pageable":
        host = [g.cpu() for g in (b.grads[i] for i in b.plan_order())]
    else:
        host = []
        for i in b.plan_order():
            g = b.grads[i]
            buf = torch.empty(g.numel() + 8, dtype=g.dtype).pin_memory()
            view = buf[1:1 + g.numel()]  # 2 bytes off the pinned allocation's alignment
            view.copy_(g.cpu())
            host.append(view)
    want = [g.clone() for g in b.grads]
    for gr in b.grads:
        gr.zero_()
    steps = [ob.step_from_host(host) for _ in range(2)]
    assert steps == [[1], [2]]
    for x, y in zip(helpers.snapshot(a), helpers.snapshot(b)):
        assert torch.equal(x, y)
    for g, w in zip(b.grads, want):
        assert torch.equal(g, w)  # the copy path filled the device gradients


def test_abi_rejects_bad_calls_without_launching():
    L = _abi.lib()
    spec = workloads.large_uniform(n_tensors=2, numel=1000)
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, check_finite=True)
    snap = helpers.snapshot(shard)
    # a check-finite plan refuses a missing noop flag, and a misaligned one
    st = L.fadam_step(opt._plan, None, None)
    assert st == _abi.EINVAL and b"noop" in L.fadam_last_error()
    st = L.fadam_step(opt._plan, opt.noop.data_ptr() + 2, None)
    assert st == _abi.EALIGN
    torch.cuda.synchronize()
    assert helpers.state_equal(shard, snap)
    assert opt.group_steps() == [0] and opt.device_status() == 0
    # set_groups refuses a different group count
    grp = (_abi.Group * 2)()
    assert L.fadam_plan_set_groups(opt._plan, grp, 2) == _abi.EINVAL


def test_grid_barrier_wait_runs_out_and_the_plan_recovers():
    """The screen's grid barrier of the plan's first step is told to wait for
    one CTA more than the launch has (a count nothing reaches): every wait
    gives up after its limit, nothing is updated and no counter moves.  The
    same plan's next steps, with the status word left unread in between, run
    normally and match the oracle; the status then reads FADAM_ETIMEOUT once
    (kept from the first launch until read) and FADAM_OK after that."""
    spec = workloads.small_versions()["tiny_adamw"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, check_finite=True,
                         extra_flags=_abi.TEST_BARRIER_TIMEOUT)
    snap = helpers.snapshot(shard)
    opt.step()
    torch.cuda.synchronize()
    assert helpers.state_equal(shard, snap)
    assert opt.group_steps() == [0, 0] and opt.noop.item() == 0
    osh = helpers.oracle_shard(shard)
    for k in (2, 3):
        workloads.fresh_grads(shard, k)
        helpers.refresh_grads(osh, shard)
        opt.step()
        oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)
    assert rep.n == 3 * sum(spec.sizes)
    assert opt.group_steps() == oracle.group_steps(osh) == [2, 2]
    assert opt.device_status() == _abi.ETIMEOUT
    assert opt.device_status() == _abi.OK  # reading clears it
    opt.step()
    oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    helpers.compare(shard, osh)
    assert opt.group_steps() == [3, 3] and opt.device_status() == _abi.OK
    opt.close()


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out_dtype", [None, torch.float32, torch.bfloat16])
def test_16bit_state_matches_oracle(state_dtype, g_dtype, out_dtype):
    """p, m, v in one 16-bit dtype (the functor's single type T), several
    steps, ragged sizes, both modes and bias corrections."""
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=state_dtype,
                                   g_dtype=g_dtype)
    spec.sizes = [40_003, 7, 131_072 + 5]
    spec.group_of = [0, 1, 1]
    spec.groups = [spec.groups[0], workloads.GroupSpec(adam_w_mode=False, weight_decay=0.05,
                                                       bias_correction=False)]
    spec.out_dtype = out_dtype
    for capturable in (False, True):
        shard, opt, osh = _run(spec, 4, capturable=capturable)
        rep = helpers.compare(shard, osh)
        assert opt.group_steps() == [4, 4]
        assert rep.exact_fraction == 1.0, rep.exact_fraction


@pytest.mark.parametrize("moment_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("out_dtype", [None, torch.bfloat16])
def test_16bit_moments_match_oracle(moment_dtype, g_dtype, out_dtype):
    """An fp32 master with m and v in one 16-bit dtype (exp_avg_dtype =
    exp_avg_sq_dtype), several steps, ragged sizes, both modes and bias
    corrections, regular and capturable."""
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, g_dtype=g_dtype,
                                   moment_dtype=moment_dtype)
    spec.sizes = [40_003, 7, 131_072 + 5]
    spec.group_of = [0, 1, 1]
    spec.groups = [spec.groups[0], workloads.GroupSpec(adam_w_mode=False, weight_decay=0.05,
                                                       bias_correction=False)]
    spec.out_dtype = out_dtype
    for capturable in (False, True):
        shard, opt, osh = _run(spec, 4, capturable=capturable)
        assert opt.moment_dtype == moment_dtype
        rep = helpers.compare(shard, osh)
        assert opt.group_steps() == [4, 4]
        assert rep.exact_fraction == 1.0, rep.exact_fraction


@pytest.mark.parametrize("state_dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("start", [162, 336, 20000])
def test_16bit_state_late_steps_match_oracle(state_dtype, start):
    """Late steps, where a bias correction rounds to 1 in float (bc1 from
    step 165 with beta1 0.9, bc2 from 338 with beta2 0.95 and 17,321 with
    0.999): the 16-bit state takes tile instances without those divisions,
    and every step across each switch point equals the oracle bit for
    bit."""
    spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=state_dtype,
                                   g_dtype=torch.bfloat16)
    spec.sizes = [40_003, 7, 131_072 + 5]
    spec.group_of = [0, 1, 1]
    spec.groups = [spec.groups[0], workloads.GroupSpec(adam_w_mode=False, weight_decay=0.05,
                                                       betas=(0.9, 0.999))]
    spec.out_dtype = torch.bfloat16
    # the steps run are start + 1 .. start + 5: 163-167 cross bc1's switch,
    # 337-341 bc2's (beta2 0.95), 20001-20005 have both at 1 in both groups
    bc = {(b, k): float(oracle.bias_correction(b, k)) for b in (0.9, 0.95, 0.999)
          for k in (start + 1, start + 5)}
    if start == 162:
        assert bc[0.9, 163] < 1.0 and bc[0.9, 167] == 1.0
    if start == 336:
        assert bc[0.95, 337] < 1.0 and bc[0.95, 341] == 1.0
    if start == 20000:
        assert all(v == 1.0 for v in bc.values())
    for capturable in (False, True):
        shard, opt, osh = _run(spec, 5, capturable=capturable, start_step=start)
        rep = helpers.compare(shard, osh)
        assert opt.group_steps() == [start + 5, start + 5]
        assert rep.exact_fraction == 1.0, rep.exact_fraction
        opt.close()


@pytest.mark.parametrize("capturable", [False, True])
def test_carried_bias_corrections_follow_betas_and_steps(capturable):
    """Each launch computes the next step's bias corrections for the next
    launch to read, keyed by betas and step.  New betas, a counter set back
    to an earlier step and a counter moved far ahead must each take freshly
    computed corrections, and the steps after them the carried ones: every
    value bit-identical to the oracle throughout."""
    spec = workloads.small_versions()["tiny_adamw"]
    spec.groups = [workloads.GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.999),
                                       weight_decay=0.01),
                   workloads.GroupSpec(adam_w_mode=False, lr=2e-3, betas=(0.85, 0.99),
                                       weight_decay=0.02)]
    spec.group_of = [0, 1, 0, 1]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=capturable)
    osh = helpers.oracle_shard(shard)
    lib = _abi.lib()

    def steps(n):
        for _ in range(n):
            opt.step()
            oracle.shard_step(osh, capturable=capturable)
        torch.cuda.synchronize()
        rep = helpers.compare(shard, osh)
        assert rep.exact_fraction == 1.0, rep.exact_fraction

    steps(3)
    opt.groups[0]["betas"] = (0.8, 0.99)  # read by the next launch's group table
    osh.groups[0].beta1, osh.groups[0].beta2 = 0.8, 0.99
    if capturable:  # a capturable plan's table changes only through set_groups
        opt._fill_groups()
        _abi.check(lib.fadam_plan_set_groups(opt._plan, opt._groups_c, len(opt.groups)), "set")
    steps(2)
    opt.set_group_steps([1, 1])  # back: the next step is 2 again
    osh.steps = [1] * len(osh.steps)
    steps(2)
    opt.set_group_steps([5000, 77])  # far ahead, one group at a time
    osh.steps = [5000, 77]
    steps(2)
    assert opt.group_steps() == [5002, 79]
    opt.close()


def test_set_group_steps_checks_and_shared_counter():
    spec = workloads.small_versions()["many_small"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, shared_step=True)
    with pytest.raises(ValueError):
        opt.set_group_steps([1, 2, 3])
    with pytest.raises(ValueError):
        opt.set_group_steps([1, 1])
    with pytest.raises(ValueError):
        opt.set_group_steps([-1, -1, -1])
    opt.set_group_steps([7, 7, 7])
    opt.step()
    assert opt.group_steps() == [8, 8, 8]
    opt.close()


def test_16bit_moments_regular_capturable_and_graph_are_bit_identical():
    spec = workloads.small_versions()["many_small"]
    spec.moment_dtype = torch.bfloat16
    outs = []
    for mode in ("regular", "capturable", "graph"):
        shard = workloads.materialize(spec, DEV)
        opt = FusedAdamShard(shard.param_groups(), capturable=mode != "regular",
                             grad_scale=spec.grad_scale)
        if mode == "graph":
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                opt.step()
            torch.cuda.current_stream().wait_stream(s)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                opt.step()
            for _ in range(2):
                graph.replay()
        else:
            for _ in range(3):
                opt.step()
        torch.cuda.synchronize()
        outs.append([t.clone() for t in shard.params + shard.exp_avgs + shard.exp_avg_sqs])
        opt.close()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32))
    for a, c in zip(outs[1], outs[2]):
        assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                           c.view(torch.int16) if c.dtype != torch.float32 else c.view(torch.int32))


def test_16bit_state_shard_full_oracle_and_graph():
    spec = workloads.small_versions()["many_small"]
    spec.state_dtype = torch.bfloat16
    shard, opt, osh = _run(spec, 3)
    helpers.compare(shard, osh)
    assert opt.group_steps() == [3, 3, 3]


@pytest.mark.parametrize("name", ["tiny_adamw", "capturable_l2", "remainder_shard", "many_small"])
def test_plan_work_lists_match_the_host_dry_runs(name):
    # the packer and the chunk list a plan uploads are the ones the host-only
    # dry runs (fadam_pack_dry, fadam_chunk_dry) describe for the plan's grid
    spec = workloads.small_versions()[name]
    shard = workloads.materialize(spec, DEV)
    groups = shard.param_groups()
    opt = FusedAdamShard(groups, capturable=spec.capturable, remainders=spec.remainders,
                         grad_scale=spec.grad_scale)
    info = opt.info()
    descs = []
    for gi, g in enumerate(groups):
        outs = g.get("params_out") or [None] * len(g["params"])
        rems = g.get("remainders") or [None] * len(g["params"])
        for p, m, v, gr, o, r in zip(g["params"], g["exp_avgs"], g["exp_avg_sqs"], g["grads"],
                                     outs, rems):
            descs.append(_abi.Tensor(p=p.data_ptr(), m=m.data_ptr(), v=v.data_ptr(),
                                     g=gr.data_ptr(), p_out=o.data_ptr() if o is not None else None,
                                     rem=r.data_ptr() if r is not None else None,
                                     numel=p.numel(), group=gi))
    arr = (_abi.Tensor * max(1, len(descs)))(*descs)
    codes = {None: _abi.DT_NONE, torch.float32: _abi.DT_F32, torch.bfloat16: _abi.DT_BF16,
             torch.float16: _abi.DT_F16}
    p_dt = _abi.DT_BF16 if spec.remainders else codes[spec.state_dtype]
    g_dt, o_dt = codes[spec.g_dtype], codes[spec.out_dtype]
    flags = _abi.REMAINDERS if spec.remainders else 0
    L = _abi.lib()
    n = ctypes.c_int64()
    assert L.fadam_pack_dry(arr, len(descs), len(groups), p_dt, g_dt, o_dt, flags, info["grid"],
                            None, 0, None, ctypes.byref(n)) == _abi.OK, L.fadam_last_error()
    assert n.value == info["n_items"]
    assert L.fadam_chunk_dry(arr, len(descs), len(groups), p_dt, g_dt, o_dt, flags, info["grid"],
                             131072, None, 0, ctypes.byref(n)) == _abi.OK, L.fadam_last_error()
    assert n.value == info["n_chunks"]
    opt.close()


_SPECIAL = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.1754944e-38,
                     3.4e38, -3.4e38, 1e-20, 65504.0, 1.0, -1.0], dtype=np.float32)


def _sprinkle(t: torch.Tensor, gen: np.random.Generator, every: int) -> None:
    """Put the special values at every `every`-th element (from a random start)."""
    n = t.numel()
    pos = np.arange(int(gen.integers(0, every)), n, every)
    vals = _SPECIAL[gen.integers(0, len(_SPECIAL), size=len(pos))]
    t.view(-1)[torch.as_tensor(pos, device=t.device)] = torch.as_tensor(vals, device=t.device).to(t.dtype)


@pytest.mark.parametrize("start_step", [0, 9998])
def test_special_values_and_extreme_hyper_parameters(start_step):
    # infinities, NaNs, signed zeros, subnormals and values near overflow in
    # p, m, v and g (no screen: they flow through the arithmetic), and groups
    # with lr 0, betas 0, eps 0, large and negative decay, bias correction
    # off, and a late step where 1 - beta^step rounds to 1: every value as
    # the oracle's IEEE sequence gives it (NaN where it gives NaN)
    groups = [
        workloads.GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.999), eps=1e-8,
                            weight_decay=0.1),
        workloads.GroupSpec(adam_w_mode=False, lr=0.0, betas=(0.0, 0.0), eps=0.0,
                            weight_decay=0.0),
        workloads.GroupSpec(adam_w_mode=True, lr=10.0, betas=(0.99, 0.9999), eps=1e-30,
                            weight_decay=1e-4, bias_correction=False),
        workloads.GroupSpec(adam_w_mode=False, lr=3e-4, betas=(0.5, 0.75), eps=1e-6,
                            weight_decay=-0.1),
    ]
    sizes = [37, 4099, 5, 70003]
    shard = _custom_shard(sizes * 2, [0, 1, 0, 3] * 2, [0, 1, 0, 3] * 2,
                          [0, 1, 2, 3, 3, 2, 1, 0], groups, out_dtype=torch.bfloat16)
    gen = np.random.default_rng(5)
    for i in range(len(shard.params)):
        shard.exp_avgs[i].copy_(torch.randn_like(shard.exp_avgs[i]) * 1e-2)
        shard.exp_avg_sqs[i].copy_(torch.rand_like(shard.exp_avg_sqs[i]) * 1e-4)
        for t, every in ((shard.params[i], 7), (shard.exp_avgs[i], 11),
                         (shard.exp_avg_sqs[i], 13), (shard.grads[i], 5)):
            _sprinkle(t, gen, every)
    opt = FusedAdamShard(shard.param_groups(), capturable=False)
    opt.host_steps = [start_step] * len(groups)
    osh = helpers.oracle_shard(shard)
    osh.steps = [start_step] * len(groups)
    for _ in range(3):
        opt.step()
        oracle.shard_step(osh, capturable=False)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)
    assert rep.exact_fraction == 1.0


@pytest.mark.parametrize("form", ["bf16_state_fp16_grads", "remainders", "fp16_moments"])
def test_special_values_in_16bit_and_remainder_forms(form):
    # the special values again, stored in the 16-bit state (bf16, with fp16
    # gradients, so 3.4e38 becomes an fp16 infinity) or in the bf16 high
    # halves of the remainder form
    if form == "remainders":
        spec = workloads.small_versions()["remainder_shard"]
    elif form == "fp16_moments":
        spec = workloads.large_uniform(n_tensors=3, numel=40_003, g_dtype=torch.bfloat16,
                                       moment_dtype=torch.float16)
        spec.out_dtype = torch.bfloat16
    else:
        spec = workloads.large_uniform(n_tensors=3, numel=40_003, state_dtype=torch.bfloat16,
                                       g_dtype=torch.float16)
        spec.out_dtype = torch.float16
    shard = workloads.materialize(spec, DEV)
    gen = np.random.default_rng(6)
    for i in range(len(shard.params)):
        for t, every in ((shard.params[i], 7), (shard.grads[i], 5)):
            _sprinkle(t, gen, every)
        if form != "remainders":
            shard.exp_avgs[i].copy_(torch.randn_like(shard.exp_avgs[i]) * 1e-2)
            shard.exp_avg_sqs[i].copy_(torch.rand_like(shard.exp_avg_sqs[i]) * 1e-4)
            _sprinkle(shard.exp_avgs[i], gen, 11)
            _sprinkle(shard.exp_avg_sqs[i], gen, 13)
    opt = FusedAdamShard(shard.param_groups(), capturable=spec.capturable,
                         remainders=spec.remainders, grad_scale=spec.grad_scale)
    osh = helpers.oracle_shard(shard)
    for _ in range(3):
        opt.step()
        oracle.shard_step(osh, capturable=spec.capturable)
    torch.cuda.synchronize()
    rep = helpers.compare(shard, osh)
    assert rep.exact_fraction == 1.0


@pytest.mark.parametrize("name", ["tiny_adamw", "remainder_shard"])
def test_two_hundred_graph_replays_stay_bit_identical(name):
    # a long run: 200 steps of a captured capturable step, new gradients
    # before each replay (written into the same buffers the graph reads);
    # the counters reach 200, beta1^step underflows the bias correction to
    # 1, and every value still equals the oracle's
    spec = workloads.small_versions()[name]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, remainders=spec.remainders,
                         grad_scale=spec.grad_scale)
    osh = helpers.oracle_shard(shard)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager step on the side stream before capture
        opt.step()
    torch.cuda.current_stream().wait_stream(s)
    oracle.shard_step(osh, capturable=True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        opt.step()
    for k in range(2, 201):
        workloads.fresh_grads(shard, k)
        helpers.refresh_grads(osh, shard)
        graph.replay()
        oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    assert opt.group_steps() == [200] * len(spec.groups)
    rep = helpers.compare(shard, osh)
    assert rep.exact_fraction == 1.0


def test_learning_rate_and_grad_scale_schedules_under_graph_replay():
    # the capturable step reads lr and grad_scale from device memory at each
    # launch: a schedule written between replays (a warm-up ramp and a decay
    # per group, a loss-scale change) reaches every replay without a new
    # capture
    spec = workloads.small_versions()["many_small"]
    shard = workloads.materialize(spec, DEV)
    opt = FusedAdamShard(shard.param_groups(), capturable=True, grad_scale=spec.grad_scale)
    osh = helpers.oracle_shard(shard)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        opt.step()
    torch.cuda.current_stream().wait_stream(s)
    oracle.shard_step(osh, capturable=True)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        opt.step()
    for k in range(2, 9):
        for gi, g in enumerate(spec.groups):
            lr = np.float32(g.lr * min(1.0, k / 4) * 0.9 ** max(0, k - 4) * (gi + 1))
            opt.set_lr(gi, float(lr))
            osh.groups[gi].lr = float(lr)
        scale = float(np.float32(2.0 ** (k % 3) * spec.grad_scale))
        opt.set_grad_scale(scale)
        for grp in osh.groups:
            grp.grad_scale = scale
        workloads.fresh_grads(shard, k)
        helpers.refresh_grads(osh, shard)
        graph.replay()
        oracle.shard_step(osh, capturable=True)
    torch.cuda.synchronize()
    assert opt.group_steps() == [8] * len(spec.groups)
    rep = helpers.compare(shard, osh)
    assert rep.exact_fraction == 1.0
