"""C-ABI checks that need no GPU.

* libfadam.so loads and exports every function include/fadam.h declares;
* every host-side argument check returns its status before any CUDA call
  (so nothing could be launched) and leaves a message;
* the packer (through the host-only dry run) covers every element of every
  tensor exactly once, keeps vector runs aligned, and balances the CTAs.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads
from adamw_optimizer_step_persistent_gb300 import _abi

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "fadam.h")
L = _abi.lib()

# the packer's cost model (fadam_plan.cu): bytes per element + a fixed
# per-item overhead, items cut at multiples of 32 elements
ITEM_OVERHEAD = 4096.0
CUT = 32


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^(?:fadam_status|const char\*|int32_t)\s+(fadam_\w+)\(", text, re.M)


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(L, name), name
    assert {n for n, _, _ in _abi.SIGNATURES} == set(names)
    assert L.fadam_version() == 10000


def test_status_strings():
    for code in range(7):
        assert L.fadam_status_string(code)
    assert L.fadam_status_string(99) == b"unknown status"


# ---- argument checks ------------------------------------------------------------

FAKE = 0x7F0000000000  # never dereferenced: the checks fail before any use


def _tensor(i=0, numel=1024, group=0, p=None, m=None, v=None, g=None, out=None, rem=None):
    base = FAKE + i * (1 << 32)
    return _abi.Tensor(p=base if p is None else p, m=base + (1 << 28) if m is None else m,
                       v=base + (2 << 28) if v is None else v, g=base + (3 << 28) if g is None else g,
                       p_out=out, rem=rem, numel=numel, group=group)


def _group(**kw):
    g = _abi.Group(mode=1, bias_correction=1, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0,
                   lr=1e-3, grad_scale=1.0, step=1)
    for k, v in kw.items():
        setattr(g, k, v)
    return g


def _create(tensors, groups, p=_abi.DT_F32, g=_abi.DT_F32, out=_abi.DT_NONE, flags=0):
    arr = (_abi.Tensor * max(1, len(tensors)))(*tensors)
    grp = (_abi.Group * max(1, len(groups)))(*groups)
    plan = ctypes.c_void_p(123)
    st = L.fadam_plan_create(arr, len(tensors), grp, len(groups), p, g, out, flags,
                             ctypes.byref(plan))
    return st, plan


@pytest.mark.parametrize("case,want", [
    ("no_groups", _abi.EINVAL), ("too_many_groups", _abi.EINVAL), ("bad_g_dtype", _abi.EDTYPE),
    ("rem_needs_bf16_p", _abi.EDTYPE), ("bad_state_dtype", _abi.EDTYPE),
    ("rem_needs_bf16_out", _abi.EDTYPE), ("unknown_flag", _abi.EINVAL),
    ("preadvanced_needs_capturable", _abi.EINVAL), ("group_out_of_range", _abi.EINVAL),
    ("negative_numel", _abi.EINVAL), ("null_p", _abi.EINVAL), ("out_ptr_without_dtype", _abi.EINVAL),
    ("missing_out_ptr", _abi.EINVAL), ("rem_without_flag", _abi.EINVAL),
    ("misaligned_m", _abi.EALIGN), ("misaligned_bf16_g", _abi.EALIGN),
    ("numel_beyond_max", _abi.ELIMIT), ("bad_mode", _abi.EINVAL), ("beta_one", _abi.EINVAL),
    ("misaligned_16bit_state_m", _abi.EALIGN), ("timeout_diag_needs_screen", _abi.EINVAL),
    ("negative_eps", _abi.EINVAL), ("nan_lr", _abi.EINVAL),
    ("capturable_without_step_dev", _abi.EINVAL), ("capturable_without_lr_dev", _abi.EINVAL),
    ("misaligned_step_dev", _abi.EALIGN),
    ("both_moment_flags", _abi.EINVAL), ("moments_need_fp32_master", _abi.EDTYPE),
    ("moments_not_with_remainders", _abi.EDTYPE), ("moments_not_with_scaled", _abi.EDTYPE),
    ("misaligned_16bit_moment", _abi.EALIGN),
])
def test_plan_create_rejects(case, want):
    t, g, kw = [_tensor()], [_group()], {}
    if case == "no_groups":
        g = []
    elif case == "too_many_groups":
        g = [_group()] * 33
    elif case == "bad_g_dtype":
        kw["g"] = 7
    elif case == "rem_needs_bf16_p":
        kw.update(flags=_abi.REMAINDERS, out=_abi.DT_BF16)
    elif case == "bad_state_dtype":
        kw["p"] = 9
    elif case == "rem_needs_bf16_out":
        kw.update(flags=_abi.REMAINDERS, p=_abi.DT_BF16, out=_abi.DT_F32)
    elif case == "unknown_flag":
        kw["flags"] = 1 << 10
    elif case == "both_moment_flags":
        kw["flags"] = _abi.MOMENTS_BF16 | _abi.MOMENTS_F16
    elif case == "moments_need_fp32_master":
        kw.update(flags=_abi.MOMENTS_BF16, p=_abi.DT_BF16)
    elif case == "moments_not_with_remainders":
        kw.update(flags=_abi.MOMENTS_BF16 | _abi.REMAINDERS, p=_abi.DT_BF16, out=_abi.DT_BF16)
        t = [_tensor(rem=FAKE + (6 << 28), out=FAKE + (5 << 28))]
    elif case == "moments_not_with_scaled":
        kw.update(flags=_abi.MOMENTS_F16 | _abi.SCALED_STATES)
    elif case == "misaligned_16bit_moment":
        t = [_tensor(v=FAKE + 1)]
        kw["flags"] = _abi.MOMENTS_F16
    elif case == "preadvanced_needs_capturable":
        kw["flags"] = _abi.STEP_PREADVANCED
    elif case == "group_out_of_range":
        t = [_tensor(group=1)]
    elif case == "negative_numel":
        t = [_tensor(numel=-1)]
    elif case == "null_p":
        t = [_tensor(p=0)]
    elif case == "out_ptr_without_dtype":
        t = [_tensor(out=FAKE + (5 << 28))]
    elif case == "missing_out_ptr":
        kw["out"] = _abi.DT_BF16
    elif case == "rem_without_flag":
        t = [_tensor(rem=FAKE + (6 << 28))]
    elif case == "misaligned_m":
        t = [_tensor(m=FAKE + 2)]
    elif case == "misaligned_bf16_g":
        t = [_tensor(g=FAKE + 1)]
        kw["g"] = _abi.DT_BF16
    elif case == "numel_beyond_max":
        t = [_tensor(numel=(1 << 40) + 1)]
    elif case == "misaligned_16bit_state_m":
        t = [_tensor(m=FAKE + 1)]
        kw["p"] = _abi.DT_BF16
    elif case == "timeout_diag_needs_screen":
        kw["flags"] = _abi.TEST_BARRIER_TIMEOUT
    elif case == "bad_mode":
        g = [_group(mode=2)]
    elif case == "beta_one":
        g = [_group(beta1=1.0)]
    elif case == "negative_eps":
        g = [_group(eps=-1.0)]
    elif case == "nan_lr":
        g = [_group(lr=float("nan"))]
    elif case == "capturable_without_step_dev":
        g = [_group(lr_dev=FAKE, grad_scale_dev=FAKE + 64)]
        kw["flags"] = _abi.CAPTURABLE
    elif case == "capturable_without_lr_dev":
        g = [_group(step_dev=FAKE, grad_scale_dev=FAKE + 64)]
        kw["flags"] = _abi.CAPTURABLE
    elif case == "misaligned_step_dev":
        g = [_group(step_dev=FAKE + 2, lr_dev=FAKE + 64, grad_scale_dev=FAKE + 128)]
        kw["flags"] = _abi.CAPTURABLE
    st, plan = _create(t, g, **kw)
    assert st == want, (case, st, L.fadam_last_error())
    assert not plan.value  # *plan_out is cleared on error
    assert L.fadam_last_error()


def test_empty_capturable_group_may_omit_lr_and_scale():
    # a group with no tensor needs only its step counter; the call then gets
    # past every argument check (on a machine without a GPU it stops at the
    # first CUDA call instead)
    g = [_group(step_dev=FAKE, lr_dev=FAKE + 64, grad_scale_dev=FAKE + 128), _group(step_dev=FAKE + 256)]
    st, _ = _create([_tensor()], g, flags=_abi.CAPTURABLE)
    assert st in (_abi.OK, _abi.ECUDA)


def test_null_handles():
    assert L.fadam_step(None, None, None) == _abi.EINVAL
    st = ctypes.c_int32()
    assert L.fadam_plan_status(None, ctypes.byref(st)) == _abi.EINVAL
    assert L.fadam_plan_get_info(None, None) == _abi.EINVAL
    assert L.fadam_plan_destroy(None) == _abi.OK
    assert L.fadam_plan_set_groups(None, None, 1) == _abi.EINVAL
    assert L.fadam_step_host_grads(None, None, None, None, None) == _abi.EINVAL
    plan = ctypes.c_void_p()
    grp = (_abi.Group * 1)(_group())
    assert L.fadam_plan_create(None, 0, grp, 1, 1, 1, 0, 0, None) == _abi.EINVAL


def test_step_once_checks():
    arr = (_abi.Tensor * 1)(_tensor())
    # some but not all device scalars
    st = L.fadam_step_once(arr, 1, 1, 1, 0.9, 0.999, 1e-8, 0.0, 1e-3, FAKE, 1, None, 1.0, None,
                           None, _abi.DT_F32, _abi.DT_NONE, None)
    assert st == _abi.EINVAL
    arr2 = (_abi.Tensor * 1)(_tensor(group=1))
    st = L.fadam_step_once(arr2, 1, 1, 1, 0.9, 0.999, 1e-8, 0.0, 1e-3, None, 1, None, 1.0, None,
                           None, _abi.DT_F32, _abi.DT_NONE, None)
    assert st == _abi.EINVAL
    st = L.fadam_step_once(arr, 1, 1, 1, 0.9, 0.999, 1e-8, 0.0, 1e-3, None, 1, None, 1.0, None,
                           FAKE + 2, _abi.DT_F32, _abi.DT_NONE, None)
    assert st == _abi.EALIGN
    # the one-shot regular step needs step >= 1 with bias correction
    st = L.fadam_step_once(arr, 1, 1, 1, 0.9, 0.999, 1e-8, 0.0, 1e-3, None, 0, None, 1.0, None,
                           None, _abi.DT_F32, _abi.DT_NONE, None)
    assert st == _abi.EINVAL and b"step" in L.fadam_last_error()


# ---- the packer -------------------------------------------------------------------

def _dry(tensors, grid, n_groups=1, p=_abi.DT_F32, g=_abi.DT_F32, out=_abi.DT_NONE, flags=0):
    arr = (_abi.Tensor * max(1, len(tensors)))(*tensors)
    n = ctypes.c_int64()
    st = L.fadam_pack_dry(arr, len(tensors), n_groups, p, g, out, flags, grid, None, 0, None,
                          ctypes.byref(n))
    assert st == _abi.OK, L.fadam_last_error()
    items = (_abi.PackItem * max(1, n.value))()
    cta = (ctypes.c_int32 * (grid + 1))()
    st = L.fadam_pack_dry(arr, len(tensors), n_groups, p, g, out, flags, grid, items, n.value,
                          cta, ctypes.byref(n))
    assert st == _abi.OK, L.fadam_last_error()
    return [(it.tensor, it.offset, it.n, it.vec) for it in items[: n.value]], list(cta)


def _aligned_tensors(sizes, start=1 << 40):
    """Separate allocations, 256-byte aligned like cudaMalloc's."""
    ts, addr = [], start
    for s in sizes:
        ptrs = []
        for _ in range(4):
            ptrs.append(addr)
            addr += (s * 4 + 255) // 256 * 256 + 256
        ts.append(_abi.Tensor(p=ptrs[0], m=ptrs[1], v=ptrs[2], g=ptrs[3], numel=s, group=0))
    return ts


def _check_cover(tensors, items):
    pos = {}
    for t_idx, off, n, _ in items:
        assert n > 0
        assert pos.get(t_idx, 0) == off, "items of a tensor must be contiguous and in order"
        pos[t_idx] = off + n
    for i, t in enumerate(tensors):
        assert pos.get(i, 0) == max(t.numel, 0)


def _cta_costs(items, cta, bpe):
    cost = [ITEM_OVERHEAD + n * bpe for _, _, n, _ in items]
    return [sum(cost[cta[b]:cta[b + 1]]) for b in range(len(cta) - 1)]


@pytest.mark.parametrize("recipe", ["large_uniform", "many_small", "capturable_l2"])
def test_pack_covers_and_balances_full_workloads(recipe):
    spec = workloads.full_versions()[recipe]
    tensors = _aligned_tensors(spec.sizes)
    grid = 152 * 2
    gdt = _abi.DT_BF16 if spec.g_dtype != workloads.torch.float32 else _abi.DT_F32
    items, cta = _dry(tensors, grid, g=gdt)
    _check_cover(tensors, items)
    assert cta[0] == 0 and cta[-1] == len(items) and all(a <= b for a, b in zip(cta, cta[1:]))
    bpe = 24 + (2 if gdt == _abi.DT_BF16 else 4)
    costs = _cta_costs(items, cta, bpe)
    quota = sum(costs) / grid
    slack = 2 * (ITEM_OVERHEAD + CUT * bpe)
    assert max(costs) <= quota * 1.0001 + slack, (max(costs), quota)
    # the last CTA may end short by the overhead the packer reserved for cuts
    assert min(costs[:-1]) >= quota * 0.9999 - slack, (min(costs), quota)
    # every run of a 256-byte aligned allocation takes the bulk-copy path and
    # starts on a cut
    assert all(vec == 2 for *_, vec in items)
    assert all(off % CUT == 0 for _, off, _, _ in items)


def test_pack_peels_heads_and_falls_back_to_scalar():
    base = 1 << 40
    ts = [
        # all streams one fp32 element past a 16-byte boundary: peel 3, then bulk
        _abi.Tensor(p=base + 4, m=base + 4096 + 4, v=base + 8192 + 4, g=base + 12288 + 4,
                    numel=1001, group=0),
        # residues disagree: the whole tensor runs scalar
        _abi.Tensor(p=base + 16384, m=base + 20480 + 4, v=base + 24576, g=base + 28672,
                    numel=500, group=0),
        _abi.Tensor(p=base, m=base, v=base, g=base, numel=0, group=0),
        _abi.Tensor(p=base + 32768, m=base + 36864, v=base + 40960, g=base + 45056, numel=2,
                    group=0),
    ]
    items, cta = _dry(ts, 1)
    _check_cover(ts, items)
    assert items[0] == (0, 0, 3, 0) and items[1] == (0, 3, 998, 2)
    assert items[2] == (1, 0, 500, 0)
    assert items[3][0] == 3 and items[3][3] == 2  # a 2-element aligned run: tail only
    assert cta == [0, len(items)]


def test_pack_peels_up_to_seven_for_16_byte_alignment():
    base = 1 << 40
    # fp32 p/m/v at +8 bytes and bf16 g at +4 bytes: 6 elements later every
    # stream sits on a 16-byte boundary
    t = _abi.Tensor(p=base + 8, m=base + 4096 + 8, v=base + 8192 + 8, g=base + 12288 + 4,
                    numel=100, group=0)
    items, _ = _dry([t], 1, g=_abi.DT_BF16)
    assert items[0] == (0, 0, 6, 0) and items[1] == (0, 6, 94, 2)


def test_pack_vector_level_when_16_bytes_is_out_of_reach():
    base = 1 << 40
    # two 16-bit streams that agree modulo one vector (8 bytes) but not
    # modulo 16 bytes: 128-bit loads yes, bulk copies no
    t = _abi.Tensor(p=base, m=base + 4096, v=base + 8192, g=base + 12288, p_out=base + 16384 + 8,
                    numel=100, group=0)
    items, _ = _dry([t], 1, g=_abi.DT_BF16, out=_abi.DT_BF16)
    assert items == [(0, 0, 100, 1)]


def test_pack_empty_shard():
    items, cta = _dry([], 4)
    assert items == [] and cta == [0, 0, 0, 0, 0]


def test_pack_splits_huge_tensor_into_bounded_items():
    t = _aligned_tensors([(1 << 31) + 12345])
    items, cta = _dry(t, 8)
    _check_cover(t, items)
    assert max(n for _, _, n, _ in items) <= 1 << 26
    assert len(items) >= 32


def test_pack_16bit_state_aligns_every_stream_to_16_bytes():
    base = 1 << 40
    # bf16 p, m, v and fp32 g: p, m, v at +4 bytes (2 elements), g at +8 bytes
    # (2 elements): 6 elements later all four sit on 16-byte boundaries
    t = _abi.Tensor(p=base + 4, m=base + 4096 + 4, v=base + 8192 + 4, g=base + 12288 + 8,
                    numel=200, group=0)
    items, _ = _dry([t], 1, p=_abi.DT_BF16)
    assert items[0] == (0, 0, 6, 0) and items[1] == (0, 6, 194, 2)


# ---- the chunk list -------------------------------------------------------------

PLAN_MAX_CHUNKS = 131072
NOALLOC_MAX_CHUNKS = 4096
TAPER_MIN = 4


def _chunks(tensors, grid, max_chunks, g=_abi.DT_F32):
    arr = (_abi.Tensor * max(1, len(tensors)))(*tensors)
    n = ctypes.c_int64()
    st = L.fadam_chunk_dry(arr, len(tensors), 1, _abi.DT_F32, g, _abi.DT_NONE, 0, grid,
                           max_chunks, None, 0, ctypes.byref(n))
    assert st == _abi.OK, L.fadam_last_error()
    out = (ctypes.c_int32 * max(3, 3 * n.value))()
    st = L.fadam_chunk_dry(arr, len(tensors), 1, _abi.DT_F32, g, _abi.DT_NONE, 0, grid,
                           max_chunks, out, n.value, ctypes.byref(n))
    assert st == _abi.OK, L.fadam_last_error()
    return [tuple(out[3 * i:3 * i + 3]) for i in range(n.value)]


def _tiles_of(item):
    _, _, n, vec = item
    return ((n // 4) & ~1) // -1024 * -1 if vec == 2 else 0


def _check_chunk_cover(items, chunks):
    """Every tile of every bulk item in exactly one chunk, items in order."""
    nxt = {}
    for k, t0, nt in chunks:
        assert nt >= 1 and nxt.get(k, 0) == t0
        nxt[k] = t0 + nt
    for k, it in enumerate(items):
        assert nxt.get(k, 0) == _tiles_of(it), k
    order = [k for k, _, _ in chunks]
    assert order == sorted(order)


@pytest.mark.parametrize("recipe", ["large_uniform", "many_small", "capturable_l2"])
def test_chunk_list_covers_every_tile_and_tapers(recipe):
    spec = workloads.full_versions()[recipe]
    tensors = _aligned_tensors(spec.sizes)
    grid = 152
    gdt = _abi.DT_BF16 if spec.g_dtype != workloads.torch.float32 else _abi.DT_F32
    items, _ = _dry(tensors, grid, g=gdt)
    chunks = _chunks(tensors, grid, PLAN_MAX_CHUNKS, g=gdt)
    _check_chunk_cover(items, chunks)
    assert len(chunks) <= PLAN_MAX_CHUNKS
    sizes = [nt for _, _, nt in chunks]
    last = {k: t0 + nt for k, t0, nt in chunks}
    # each chunk takes min(16, max(4, tiles left / (2 grid))) tiles, cut
    # short only by the end of its item
    left = sum(sizes)
    for k, t0, nt in chunks:
        want = min(16, max(TAPER_MIN, left // (2 * grid)))
        assert nt == want or t0 + nt == last[k], (k, t0, nt, want, left)
        left -= nt
    # the end of the list is in small chunks: the CTAs finish together
    assert max(sizes[-grid:]) <= TAPER_MIN
    assert max(sizes) == 16


def test_chunk_list_keeps_to_the_noalloc_limit():
    # 201 x 20,971,520 has about a million tiles: 4096 chunks need bigger
    # chunks than 16 tiles, so the list is untapered and grown to fit
    spec = workloads.full_versions()["large_uniform"]
    tensors = _aligned_tensors(spec.sizes)
    items, _ = _dry(tensors, 152)
    chunks = _chunks(tensors, 152, NOALLOC_MAX_CHUNKS)
    _check_chunk_cover(items, chunks)
    assert len(chunks) <= NOALLOC_MAX_CHUNKS
    assert max(nt for _, _, nt in chunks) > 16


def test_chunk_list_small_and_empty_shards():
    assert _chunks([], 4, PLAN_MAX_CHUNKS) == []
    tensors = _aligned_tensors([1000, 4097, 65536, 3])
    items, _ = _dry(tensors, 4)
    chunks = _chunks(tensors, 4, PLAN_MAX_CHUNKS)
    _check_chunk_cover(items, chunks)
    # 65536 elements are 16 tiles: near the end of the list, so tapered
    assert all(nt <= TAPER_MIN for _, _, nt in chunks)


def test_chunk_dry_rejects_bad_arguments():
    tensors = _aligned_tensors([4096])
    arr = (_abi.Tensor * 1)(*tensors)
    n = ctypes.c_int64()
    assert L.fadam_chunk_dry(arr, 1, 1, _abi.DT_F32, _abi.DT_F32, _abi.DT_NONE, 0, 4, 0, None, 0,
                             ctypes.byref(n)) == _abi.EINVAL
    assert L.fadam_chunk_dry(arr, 1, 1, _abi.DT_F32, _abi.DT_F32, _abi.DT_NONE, 0, 0, 16, None,
                             0, ctypes.byref(n)) == _abi.EINVAL
    assert L.fadam_chunk_dry(arr, 1, 1, _abi.DT_F32, _abi.DT_F32, _abi.DT_NONE, 0, 4, 16, None,
                             0, None) == _abi.EINVAL
    out = (ctypes.c_int32 * 3)()
    tensors = _aligned_tensors([1 << 20])
    arr = (_abi.Tensor * 1)(*tensors)
    assert L.fadam_chunk_dry(arr, 1, 1, _abi.DT_F32, _abi.DT_F32, _abi.DT_NONE, 0, 4, 16, out, 1,
                             ctypes.byref(n)) == _abi.ELIMIT


def test_chunk_list_keeps_its_taper_beyond_the_headline_shard():
    # 260 tensors of 20,971,520 (30 % more than the 201-tensor shard) still
    # fit the plan's chunk limit with 16-tile chunks and the tapered end
    spec = workloads.large_uniform(n_tensors=260)
    tensors = _aligned_tensors(spec.sizes)
    items, _ = _dry(tensors, 152)
    chunks = _chunks(tensors, 152, PLAN_MAX_CHUNKS)
    _check_chunk_cover(items, chunks)
    sizes = [nt for _, _, nt in chunks]
    assert max(sizes) == 16 and max(sizes[-152:]) <= TAPER_MIN
