"""Guard bands: no launch writes outside the tensors it was given.

compute-sanitizer is not available to these tests, so out-of-bounds writes
are looked for directly: every tensor is a view into a larger byte buffer
filled with a random pattern, with guard bytes before and after it (and,
for the exchange, gaps between the fragments of one shard buffer), at
element offsets that give every alignment class (16-byte aligned bodies,
peeled heads, vector-aligned and scalar tensors).  After a few steps of each
write path (the update with every kind of tail, 16-bit state, the remainder
form, the scaled state, the exchange's reduction and all-gather side, the
host-gradient step) every guard byte must still hold its pattern.
"""
import pytest
import torch

from adamw_optimizer_step_persistent_gb300 import FusedAdamShard

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 208  # bytes on each side of a view (a multiple of 16)

SIZES = [1, 3, 4, 5, 31, 1000, 4097, 70001, 65539, 262144, 300007]
# each view starts GUARD + shift elements into its buffer: p and param-out
# shifted by SHIFT_P, m, v, g by SHIFT_Q.  Equal shifts of 0 give 16-byte
# aligned bodies (bulk copies), equal shifts of 1 or 2 a peeled head and
# vector-aligned loads, unequal shifts the element-wise path.
SHIFT_P = [0, 1, 2, 3, 1, 0, 0, 1, 0, 2, 0]
SHIFT_Q = [0, 1, 2, 3, 2, 1, 0, 1, 3, 2, 0]
# param-out follows p, except one tensor 4 elements further on: with 16-bit
# state and param-out, 8 bytes apart modulo 16, so only 128-bit vector loads
SHIFT_O = [0, 1, 2, 3, 1, 0, 4, 1, 0, 2, 0]


class Arena:
    """Byte buffers with one view each and guard bytes around the view."""

    def __init__(self, seed):
        self.gen = torch.Generator(device=DEV)
        self.gen.manual_seed(seed)
        self.regions = []  # (buffer, snapshot, [(start, end) of each view])

    def buffer(self, nbytes):
        buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV, generator=self.gen)
        self.regions.append([buf, None, []])
        return buf, len(self.regions) - 1

    def carve(self, idx, start, n, dtype):
        """View of n elements at byte `start` of buffer idx (start aligned to the dtype)."""
        buf = self.regions[idx][0]
        es = torch.empty(0, dtype=dtype).element_size()
        assert start % es == 0
        self.regions[idx][2].append((start, start + n * es))
        return buf[start:start + n * es].view(dtype)

    def view(self, n, dtype, shift):
        es = torch.empty(0, dtype=dtype).element_size()
        buf, idx = self.buffer(GUARD + shift * es + n * es + GUARD)
        return self.carve(idx, GUARD + shift * es, n, dtype)

    def seal(self):
        """Snapshot every buffer after the views got their initial values."""
        torch.cuda.synchronize()
        for r in self.regions:
            r[1] = r[0].clone()

    def check(self):
        torch.cuda.synchronize()
        bad = []
        for k, (buf, snap, views) in enumerate(self.regions):
            keep = torch.ones(buf.numel(), dtype=torch.bool, device=DEV)
            for a, b in views:
                keep[a:b] = False
            changed = (buf != snap) & keep
            if bool(changed.any()):
                first = int(changed.nonzero()[0])
                bad.append(f"buffer {k}: {int(changed.sum())} guard bytes changed, first at {first}")
        assert not bad, "; ".join(bad)


def _fill(p, m, v, g, gen):
    p.copy_(torch.randn(p.numel(), generator=gen, device=DEV).to(p.dtype))
    m.zero_()
    v.zero_()
    g.copy_((torch.randn(g.numel(), generator=gen, device=DEV) * 1e-3).to(g.dtype))


def _group(lists, **kw):
    d = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, adam_w_mode=True)
    d.update(kw)
    d.update(lists)
    return d


def _update_lists(arena, state_dtype, g_dtype, out_dtype, moment_dtype=None):
    gen = torch.Generator(device=DEV)
    gen.manual_seed(7)
    L = {"params": [], "exp_avgs": [], "exp_avg_sqs": [], "grads": [], "params_out": []}
    for n, sp, sq, so in zip(SIZES, SHIFT_P, SHIFT_Q, SHIFT_O):
        p = arena.view(n, state_dtype, sp)
        m = arena.view(n, moment_dtype or state_dtype, sq)
        v = arena.view(n, moment_dtype or state_dtype, sq)
        g = arena.view(n, g_dtype, sq)
        _fill(p, m, v, g, gen)
        L["params"].append(p)
        L["exp_avgs"].append(m)
        L["exp_avg_sqs"].append(v)
        L["grads"].append(g)
        if out_dtype is not None:
            L["params_out"].append(arena.view(n, out_dtype, so))
    if out_dtype is None:
        del L["params_out"]
    return L


@pytest.mark.parametrize("state_dtype,g_dtype,out_dtype", [
    (torch.float32, torch.float32, torch.bfloat16),
    (torch.float32, torch.bfloat16, torch.float16),
    (torch.bfloat16, torch.float16, torch.float16),
    (torch.float16, torch.float32, None),
])
@pytest.mark.parametrize("capturable", [False, True])
def test_update_writes_only_its_tensors(state_dtype, g_dtype, out_dtype, capturable):
    arena = Arena(11)
    L = _update_lists(arena, state_dtype, g_dtype, out_dtype)
    groups = [_group(L), _group({k: [] for k in L}, adam_w_mode=False)]
    opt = FusedAdamShard(groups, capturable=capturable, check_finite=capturable)
    arena.seal()
    for _ in range(3):
        opt.step()
    opt.grad_norm_sq()
    arena.check()
    opt.close()


@pytest.mark.parametrize("moment_dtype", [torch.bfloat16, torch.float16])
def test_16bit_moments_write_only_their_tensors(moment_dtype):
    arena = Arena(16)
    L = _update_lists(arena, torch.float32, torch.bfloat16, torch.bfloat16, moment_dtype)
    opt = FusedAdamShard([_group(L)], capturable=True, check_finite=True)
    arena.seal()
    for _ in range(3):
        opt.step()
    arena.check()
    opt.close()


def test_host_gradient_step_writes_only_its_tensors():
    arena = Arena(12)
    L = _update_lists(arena, torch.float32, torch.float32, torch.bfloat16)
    opt = FusedAdamShard([_group(L)], capturable=True)
    host = [g.cpu().pin_memory() for g in L["grads"]]
    arena.seal()
    for _ in range(2):
        opt.step_from_host(host)
    arena.check()
    opt.close()


def test_remainder_form_writes_only_its_tensors():
    arena = Arena(13)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(8)
    L = {"params": [], "remainders": [], "exp_avgs": [], "exp_avg_sqs": [], "grads": [],
         "params_out": []}
    for n, sp, sq in zip(SIZES, SHIFT_P, SHIFT_Q):
        hi = arena.view(n, torch.bfloat16, sp)
        rem = arena.view(n, torch.int16, sp)
        m = arena.view(n, torch.float32, sq)
        v = arena.view(n, torch.float32, sq)
        g = arena.view(n, torch.bfloat16, sq)
        _fill(hi, m, v, g, gen)
        hi.masked_fill_(hi == 0, 1.0)
        rem.copy_(torch.randint(-32768, 32768, (n,), dtype=torch.int32, device=DEV,
                                generator=gen).to(torch.int16))
        L["params"].append(hi)
        L["remainders"].append(rem)
        L["exp_avgs"].append(m)
        L["exp_avg_sqs"].append(v)
        L["grads"].append(g)
        L["params_out"].append(hi)  # the new high halves in place
    opt = FusedAdamShard([_group(L)], capturable=True, remainders=True)
    arena.seal()
    for _ in range(3):
        opt.step()
    arena.check()
    opt.close()


def test_scaled_state_writes_only_its_tensors():
    arena = Arena(14)
    L = _update_lists(arena, torch.float16, torch.bfloat16, torch.bfloat16)
    scales = torch.full((len(SIZES), 3), 1e-3, dtype=torch.float32, device=DEV)
    opt = FusedAdamShard([_group(L)], capturable=False, state_scales=scales)
    arena.seal()
    for _ in range(3):
        opt.step()
    arena.check()
    opt.close()


def test_exchange_writes_only_the_shard_fragments_and_destinations():
    # every tensor's g is a fragment of one gradient shard and its param-out
    # a fragment of one param-out shard, with random bytes in the gaps; the
    # sources and destinations are laid out like those shards
    arena = Arena(15)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(9)
    gap = 24  # elements between fragments (48 bytes of bf16)
    starts, pos = [], gap + 8
    for n in SIZES:
        starts.append(pos)
        pos += n + gap
        pos += (-pos) % 8  # fragment starts on 16 bytes
    total = pos + gap
    g_buf, gi = arena.buffer(2 * total)
    o_buf, oi = arena.buffer(2 * total)
    grads = [arena.carve(gi, 2 * s, n, torch.bfloat16) for s, n in zip(starts, SIZES)]
    outs = [arena.carve(oi, 2 * s, n, torch.bfloat16) for s, n in zip(starts, SIZES)]
    g_shard = g_buf.view(torch.bfloat16)
    o_shard = o_buf.view(torch.bfloat16)
    sources = []
    for _ in range(4):  # read only: every byte of them must stay as it was
        s_buf, _ = arena.buffer(2 * total)
        src = s_buf.view(torch.bfloat16)
        src.copy_((torch.randn(total, generator=gen, device=DEV) * 1e-2).to(torch.bfloat16))
        sources.append(src)
    dests = []
    for _ in range(3):
        d_buf, di = arena.buffer(2 * total)
        for s, n in zip(starts, SIZES):
            arena.carve(di, 2 * s, n, torch.bfloat16)
        dests.append(d_buf.view(torch.bfloat16))
    L = {"params": [], "exp_avgs": [], "exp_avg_sqs": [], "grads": grads, "params_out": outs}
    for k, n in enumerate(SIZES):
        shift = 0 if k % 2 == 0 else 1  # 16-byte aligned with the fragments, or not
        p = arena.view(n, torch.float32, shift)
        m = arena.view(n, torch.float32, shift)
        v = arena.view(n, torch.float32, shift)
        p.copy_(torch.randn(n, generator=gen, device=DEV))
        m.zero_()
        v.zero_()
        L["params"].append(p)
        L["exp_avgs"].append(m)
        L["exp_avg_sqs"].append(v)
    opt = FusedAdamShard([_group(L)], capturable=True, check_finite=True)
    opt.set_exchange(g_shard, sources, average=True, out_shard=o_shard, dests=dests)
    arena.seal()
    for _ in range(2):
        opt.step_reduce()
    opt.grad_reduce()
    arena.check()
    opt.close()
