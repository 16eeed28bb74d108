"""Property tests of the host packer and chunk list (CPU, no GPU): on random
shards (ragged, empty and large tensors, every stream at its own
element-aligned offset, every state / gradient / param-out dtype) the work
list covers every element once and in order, each item keeps the alignment
its access level needs on every stream, the CTA ranges are well formed, and
the chunk list covers every tile of every bulk item once."""
import ctypes

import pytest

from adamw_optimizer_step_persistent_gb300 import _abi
from tests.test_abi_cpu import (L, NOALLOC_MAX_CHUNKS, PLAN_MAX_CHUNKS, _check_chunk_cover,
                                _check_cover, _chunks, _dry)

hypothesis = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
given, settings, HealthCheck = hypothesis.given, hypothesis.settings, hypothesis.HealthCheck

SIZE = {_abi.DT_F32: 4, _abi.DT_BF16: 2, _abi.DT_F16: 2}

sizes = st.one_of(st.integers(0, 9), st.integers(10, 5000), st.integers(5001, 300_000),
                  st.integers(1 << 20, (1 << 20) + 4099))


@st.composite
def shards(draw):
    p = draw(st.sampled_from([_abi.DT_F32, _abi.DT_BF16, _abi.DT_F16]))
    g = draw(st.sampled_from([_abi.DT_F32, _abi.DT_BF16, _abi.DT_F16]))
    out = draw(st.sampled_from([_abi.DT_NONE, _abi.DT_BF16, _abi.DT_F16, _abi.DT_F32]))
    n = draw(st.integers(0, 24))
    # each stream of each tensor in its own allocation, offset by a whole
    # number of its elements (0-15) past a 256-byte boundary
    elem = {"p": SIZE[p], "m": SIZE[p], "v": SIZE[p], "g": SIZE[g]}
    if out != _abi.DT_NONE:
        elem["p_out"] = SIZE[out]
    addr = 1 << 40
    tensors = []
    for _ in range(n):
        numel = draw(sizes)
        # mostly one element offset for every stream (the streams reach a
        # 16-byte boundary together after at most 7 elements), sometimes one
        # stream off by a whole vector, sometimes every stream on its own
        k = draw(st.integers(0, 15))
        how = draw(st.sampled_from(["same", "same", "same", "one_vector_off", "independent"]))
        odd = draw(st.sampled_from(sorted(elem)))
        ptrs = {}
        for name, es in elem.items():
            off = k
            if how == "independent":
                off = draw(st.integers(0, 15))
            elif how == "one_vector_off" and name == odd:
                off = k + 4
            ptrs[name] = addr + es * off
            addr += (numel * es + 511) // 256 * 256 + 256
        tensors.append(_abi.Tensor(numel=numel, group=0, **ptrs))
    grid = draw(st.sampled_from([1, 3, 152]))
    return tensors, elem, p, g, out, grid


def _stream_addr(t, name, es, offset):
    return getattr(t, name) + es * offset


@settings(max_examples=150, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(shards())
def test_pack_covers_aligns_and_balances(shard):
    tensors, elem, p, g, out, grid = shard
    items, cta = _dry(tensors, grid, p=p, g=g, out=out)
    _check_cover(tensors, items)
    assert cta[0] == 0 and cta[-1] == len(items)
    assert all(a <= b for a, b in zip(cta, cta[1:]))
    for t_idx, off, n, vec in items:
        t = tensors[t_idx]
        for name, es in elem.items():
            a = _stream_addr(t, name, es, off)
            if vec == 2:  # bulk copies: every stream on a 16-byte boundary
                assert a % 16 == 0, (name, t_idx, off)
            elif vec == 1:  # 4-element vector loads
                assert a % (4 * es) == 0, (name, t_idx, off)


@settings(max_examples=100, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(shards(), st.sampled_from([PLAN_MAX_CHUNKS, NOALLOC_MAX_CHUNKS]))
def test_chunk_list_covers_every_bulk_tile_once(shard, max_chunks):
    tensors, elem, p, g, out, grid = shard
    if p != _abi.DT_F32 or out != _abi.DT_NONE:
        # the chunk dry run takes the fp32-state layout with no param-out
        tensors = [_abi.Tensor(p=t.p, m=t.m, v=t.v, g=t.g, numel=t.numel, group=0)
                   for t in tensors if t.p % 4 == 0 and t.m % 4 == 0 and t.v % 4 == 0]
    items, _ = _dry(tensors, grid, g=g)
    arr = (_abi.Tensor * max(1, len(tensors)))(*tensors)
    n = ctypes.c_int64()
    status = L.fadam_chunk_dry(arr, len(tensors), 1, _abi.DT_F32, g, _abi.DT_NONE, 0, grid,
                               max_chunks, None, 0, ctypes.byref(n))
    if status == _abi.ELIMIT:  # more chunks than the limit allows: refused, not cut
        assert max_chunks == NOALLOC_MAX_CHUNKS
        return
    assert status == _abi.OK, L.fadam_last_error()
    chunks = _chunks(tensors, grid, max_chunks, g=g)
    _check_chunk_cover(items, chunks)
    assert len(chunks) <= max_chunks
