"""Seeded synthetic shards for the tests and the benchmark.

This module only draws inputs: tensor sizes, layouts and random values.  It
holds none of the optimizer's arithmetic and is shared by the CUDA-path
tests, the oracle tests and bench.py, so both sides see the same inputs.

Five shard recipes, all synthetic (no dataset or checkpoint is involved):

1. ``tiny_adamw``: 4 fp32 tensors of 1000, 4097, 65536 and 3 elements
   (separate allocations, ragged tails) plus one empty group; AdamW,
   lr 1e-3, betas (0.9, 0.999), eps 1e-8, wd 0.01, host scalars.
2. ``capturable_l2``: a GPT-style layer list, per layer 4096x4096,
   4096x11008 (twice), 11008x4096 and two 4096 norm vectors, 8 layers
   (1,216,413,696 elements); L2 mode, wd 0.1, betas (0.9, 0.95), eps 1e-8,
   lr 1e-3 and grad_scale 1/65536 on the device, bf16 grads ~ N(0, 1e-2),
   bf16 param-out copy; one seeded element is set to +inf at one step.
3. ``large_uniform``: 201 fp32 tensors of 20,971,520 elements (the sizes of
   the TE issue's adam_bench.py), p ~ N(0,1), g = N(0,1)*1e-3, AdamW,
   lr 1.6e-3, betas (0.9, 0.95), eps 1e-8, wd 0.1, no param-out copy.
   A variant keeps p, m, v in bf16 or fp16 (``state_dtype``), with bf16
   grads: 14 bytes per element.
4. ``remainder_shard``: one contiguous 1.2e9-element bucket cut into 512
   views of log-uniform size in [4096, 16,777,216] scaled to sum to 1.2e9,
   view starts rounded up to 64 elements (the 128-byte alignment rule of
   distributed_fused_adam.py for 16-bit grads); bf16 high half + int16
   remainder, bf16 grads ~ N(0, 1e-3), AdamW wd 0.1, betas (0.9, 0.95),
   eps 1e-8, lr 1e-3 on the device; param-out is the bf16 high half itself.
5. ``many_small``: 20,000 fp32 tensors in their own allocations, 30% of
   log-uniform size in [1, 4096) and 70% in [4096, 1,048,576], shuffled;
   group 0 AdamW wd 0.1 (the large ones), group 1 L2 wd 0 (the small ones),
   group 2 empty; per-group device step counters.
6. ``exchange_shard``: the one-GPU stand-in for one data-parallel rank of
   R = 8 with its exchange: the GPT-style layer list of ``capturable_l2``
   as fragments of one gradient shard buffer and one bf16 param-out shard
   buffer (fragment starts rounded up to 64 elements, the 128-byte rule for
   16-bit grads), fp32 p, m, v, AdamW wd 0.1, betas (0.9, 0.95), eps 1e-8,
   lr 1e-3 on the device; R source buffers laid out like the gradient shard
   (each rank's bf16 gradient for this shard, ~ N(0, 1e-2)), averaged into
   the shard, and R - 1 destination buffers laid out like the param-out
   shard (the other ranks' places for it).
7. ``scaled_state_shard``: the GPT-style layer list with p, m, v stored as
   fp16 values and one fp32 scale each per tensor (the page's scaled state,
   meant for fp16 optimizer states), bf16 grads ~ N(0, 1e-2), bf16
   param-out, AdamW wd 0.1, betas (0.9, 0.95), eps 1e-8, lr 1e-3, host
   scalars (the page's scaled path is the regular one).  The stored values
   are draws of N(0, 1000^2) (|.| for v) rounded to the state dtype and the
   scales 1e-3, 1e-6 and 1e-9 (p ~ N(0, 1), m ~ N(0, 1e-6), v ~ 1e-6):
   valid scaled states, not the output of a rescale.

Every recipe takes size arguments that shrink it for tests the oracle must
finish in seconds (``small_versions``); the defaults are the full workloads.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


@dataclass
class GroupSpec:
    adam_w_mode: bool = True
    lr: float = 1e-3
    betas: tuple = (0.9, 0.999)
    eps: float = 1e-8
    weight_decay: float = 0.0
    bias_correction: bool = True

    def as_dict(self) -> Dict:
        return dict(adam_w_mode=self.adam_w_mode, lr=self.lr, betas=self.betas, eps=self.eps,
                    weight_decay=self.weight_decay, bias_correction=self.bias_correction)


@dataclass
class ShardSpec:
    name: str
    groups: List[GroupSpec]
    sizes: List[int]                 # elements per tensor
    group_of: List[int]              # param group of each tensor
    g_dtype: torch.dtype = torch.float32
    out_dtype: Optional[torch.dtype] = None
    remainders: bool = False
    state_dtype: torch.dtype = torch.float32  # p, m, v (fp32 unless 16-bit state)
    capturable: bool = False
    grad_std: float = 1e-3
    grad_scale: float = 1.0
    bucket_offsets: Optional[List[int]] = None  # views into one bucket (remainder shard)
    bucket_len: int = 0
    seed: int = 0
    inf_at_step: Optional[int] = None  # step (1-based) whose grad holds one +inf
    exchange_ranks: int = 0    # > 0: gradients and param-out as views of one shard buffer each,
    exchange_dests: int = 0    # with this many source and destination buffers
    exchange_average: bool = True  # ReduceOp.AVG (else SUM)
    exchange_align: int = 64   # fragment starts rounded up to this many elements
    scaled_state: bool = False  # p, m, v in state_dtype with one fp32 scale each per tensor
    moment_dtype: Optional[torch.dtype] = None  # m, v in bf16 or fp16 under an fp32 master
    scale_of: tuple = (1e-3, 1e-6, 1e-9)  # the scales drawn states are stored with
    notes: Dict = field(default_factory=dict)

    @property
    def n_elements(self) -> int:
        return int(sum(self.sizes))


def _log_uniform(rng: np.random.Generator, lo: float, hi: float, n: int) -> np.ndarray:
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))


def tiny_adamw(seed: int = 1235) -> ShardSpec:
    g = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    return ShardSpec("tiny_adamw", [g, GroupSpec()], [1000, 4097, 65536, 3], [0, 0, 0, 0],
                     grad_std=1e-3, seed=seed)


def capturable_l2(layers: int = 8, hidden: int = 4096, ffn: int = 11008,
                  seed: int = 1236) -> ShardSpec:
    per_layer = [hidden * hidden, hidden * ffn, hidden * ffn, ffn * hidden, hidden, hidden]
    sizes = per_layer * layers
    g = GroupSpec(adam_w_mode=False, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    return ShardSpec("capturable_l2", [g], sizes, [0] * len(sizes), g_dtype=torch.bfloat16,
                     out_dtype=torch.bfloat16, capturable=True, grad_std=1e-2,
                     grad_scale=1.0 / 65536, seed=seed, inf_at_step=3)


def large_uniform(n_tensors: int = 201, numel: int = 320 * 65536, seed: int = 1237,
                  state_dtype: torch.dtype = torch.float32,
                  g_dtype: torch.dtype = torch.float32,
                  moment_dtype: Optional[torch.dtype] = None,
                  out_dtype: Optional[torch.dtype] = None) -> ShardSpec:
    g = GroupSpec(adam_w_mode=True, lr=1.6e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    name = ("large_uniform_16bit_moments" if moment_dtype is not None else
            "large_uniform" if state_dtype == torch.float32 else "large_uniform_16bit_state")
    if out_dtype is not None:
        name += "_param_out"
    return ShardSpec(name, [g], [numel] * n_tensors, [0] * n_tensors, g_dtype=g_dtype,
                     out_dtype=out_dtype, state_dtype=state_dtype, grad_std=1e-3, seed=seed,
                     moment_dtype=moment_dtype)


def remainder_shard(total: int = 1_200_000_000, n_views: int = 512, lo: int = 4096,
                    hi: int = 16_777_216, align: int = 64, seed: int = 1238) -> ShardSpec:
    rng = np.random.default_rng(seed)
    raw = _log_uniform(rng, lo, hi, n_views)
    sizes = np.maximum(1, np.round(raw * (total / raw.sum()))).astype(np.int64)
    sizes[-1] += total - int(sizes.sum())
    offsets, pos = [], 0
    for s in sizes:
        pos = (pos + align - 1) // align * align
        offsets.append(pos)
        pos += int(s)
    g = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    return ShardSpec("remainder_shard", [g], [int(s) for s in sizes], [0] * n_views,
                     g_dtype=torch.bfloat16, out_dtype=torch.bfloat16, remainders=True,
                     capturable=True, grad_std=1e-3, bucket_offsets=offsets, bucket_len=pos,
                     seed=seed)


def many_small(n_tensors: int = 20_000, frac_small: float = 0.3, small_hi: int = 4096,
               large_hi: int = 1_048_576, seed: int = 1239) -> ShardSpec:
    rng = np.random.default_rng(seed)
    n_small = int(round(n_tensors * frac_small))
    small = np.floor(_log_uniform(rng, 1, small_hi, n_small)).astype(np.int64)
    large = np.floor(_log_uniform(rng, small_hi, large_hi, n_tensors - n_small)).astype(np.int64)
    sizes = np.concatenate([small, large])
    rng.shuffle(sizes)
    sizes = np.clip(sizes, 1, large_hi)
    group_of = [0 if s >= small_hi else 1 for s in sizes]
    g0 = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1)
    g1 = GroupSpec(adam_w_mode=False, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0)
    g2 = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1)
    return ShardSpec("many_small", [g0, g1, g2], [int(s) for s in sizes], group_of,
                     capturable=True, grad_std=1e-3, seed=seed)


def exchange_shard(layers: int = 8, hidden: int = 4096, ffn: int = 11008, ranks: int = 8,
                   dests: Optional[int] = None, seed: int = 1240) -> ShardSpec:
    per_layer = [hidden * hidden, hidden * ffn, hidden * ffn, ffn * hidden, hidden, hidden]
    sizes = per_layer * layers
    g = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    return ShardSpec("exchange_shard", [g], sizes, [0] * len(sizes), g_dtype=torch.bfloat16,
                     out_dtype=torch.bfloat16, capturable=True, grad_std=1e-2, seed=seed,
                     exchange_ranks=ranks, exchange_dests=ranks - 1 if dests is None else dests)


def scaled_state_shard(layers: int = 8, hidden: int = 4096, ffn: int = 11008,
                       state_dtype: torch.dtype = torch.float16, seed: int = 1241) -> ShardSpec:
    per_layer = [hidden * hidden, hidden * ffn, hidden * ffn, ffn * hidden, hidden, hidden]
    sizes = per_layer * layers
    g = GroupSpec(adam_w_mode=True, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    return ShardSpec("scaled_state_shard", [g], sizes, [0] * len(sizes), g_dtype=torch.bfloat16,
                     out_dtype=torch.bfloat16, state_dtype=state_dtype, grad_std=1e-2, seed=seed,
                     scaled_state=True)


def scaled_versions(full: bool = False) -> Dict[str, ShardSpec]:
    """The scaled-state recipe: full size, or small ones (fp16 with an empty
    tensor and ragged sizes; bf16 with moments large enough that bf16's
    scale target keeps the reciprocals finite; bf16 with Adam-sized moments,
    whose reciprocals overflow as on the page)."""
    if full:
        return {"scaled_state_shard": scaled_state_shard()}
    f16 = scaled_state_shard(layers=2, hidden=256, ffn=689)
    f16.sizes = f16.sizes[:5] + [0] + f16.sizes[5:] + [3, 4097]
    f16.group_of = [0] * len(f16.sizes)
    b16 = scaled_state_shard(layers=1, hidden=320, ffn=1000, state_dtype=torch.bfloat16)
    b16.name, b16.scale_of = "scaled_bf16", (1e-3, 1e-3, 1e-3)
    b16_small = scaled_state_shard(layers=1, hidden=128, ffn=300, state_dtype=torch.bfloat16)
    b16_small.name = "scaled_bf16_small_moments"
    return {"scaled_state_shard": f16, "scaled_bf16": b16, "scaled_bf16_small_moments": b16_small}


def exchange_offsets(sizes: List[int], align: int = 64) -> List[int]:
    """Fragment starts in the shard buffer, each rounded up to `align`
    elements."""
    out, o = [], 0
    for n in sizes:
        o = (o + align - 1) // align * align
        out.append(o)
        o += n
    return out


def small_versions() -> Dict[str, ShardSpec]:
    """The same recipes at sizes the oracle finishes in seconds (several
    CTAs' worth of work each, ragged tails included)."""
    return {
        "tiny_adamw": tiny_adamw(),
        "capturable_l2": capturable_l2(layers=2, hidden=256, ffn=688),
        "large_uniform": large_uniform(n_tensors=6, numel=65536 * 3 + 5),
        "remainder_shard": remainder_shard(total=3_000_000, n_views=64, lo=64, hi=200_000),
        "many_small": many_small(n_tensors=2000, large_hi=65536),
    }


def exchange_versions(full: bool = False) -> Dict[str, ShardSpec]:
    """The exchange recipe: small (three ranks, a non-power-of-two average,
    ragged fragments) or at full size."""
    if full:
        return {"exchange_shard": exchange_shard()}
    # the second one sums, and packs its fragments with no alignment
    # padding (odd starts, ragged tails: the element-wise paths)
    packed = exchange_shard(layers=1, hidden=300, ffn=1001, ranks=5, dests=2)
    packed.name, packed.exchange_average, packed.exchange_align = "exchange_packed_sum", False, 1
    return {"exchange_shard": exchange_shard(layers=2, hidden=256, ffn=688, ranks=3),
            "exchange_packed_sum": packed}


def full_versions() -> Dict[str, ShardSpec]:
    return {"tiny_adamw": tiny_adamw(), "capturable_l2": capturable_l2(),
            "large_uniform": large_uniform(), "remainder_shard": remainder_shard(),
            "many_small": many_small(),
            "large_uniform_bf16_state": large_uniform(state_dtype=torch.bfloat16,
                                                      g_dtype=torch.bfloat16)}


# ---- materialising a shard ----------------------------------------------------

@dataclass
class Shard:
    """Tensors of one shard, per group, in plan order."""
    spec: ShardSpec
    params: List[torch.Tensor]
    exp_avgs: List[torch.Tensor]
    exp_avg_sqs: List[torch.Tensor]
    grads: List[torch.Tensor]
    params_out: List[Optional[torch.Tensor]]
    remainders: List[Optional[torch.Tensor]]
    buckets: Dict[str, torch.Tensor] = field(default_factory=dict)
    # exchange recipes: [R, L] sources laid out like buckets["g"], [D, L]
    # destinations laid out like buckets["p_out"], fragment starts
    sources: Optional[torch.Tensor] = None
    dests: Optional[torch.Tensor] = None
    offsets: Optional[List[int]] = None
    # scaled-state recipes: [n_tensors, 3] fp32 scales (p, m, v), spec order
    state_scales: Optional[torch.Tensor] = None

    def param_groups(self) -> List[Dict]:
        """The per-group dicts FusedAdamShard takes."""
        out = []
        for gi, gs in enumerate(self.spec.groups):
            idx = [i for i, g in enumerate(self.spec.group_of) if g == gi]
            d = gs.as_dict()
            d["params"] = [self.params[i] for i in idx]
            d["exp_avgs"] = [self.exp_avgs[i] for i in idx]
            d["exp_avg_sqs"] = [self.exp_avg_sqs[i] for i in idx]
            d["grads"] = [self.grads[i] for i in idx]
            if self.spec.out_dtype is not None:
                d["params_out"] = [self.params_out[i] for i in idx]
            if self.spec.remainders:
                d["remainders"] = [self.remainders[i] for i in idx]
            out.append(d)
        return out

    def plan_order(self) -> List[int]:
        """Tensor indices in the order FusedAdamShard hands them to the plan."""
        return [i for gi in range(len(self.spec.groups))
                for i, g in enumerate(self.spec.group_of) if g == gi]


def materialize(spec: ShardSpec, device="cuda") -> Shard:
    """Draw the shard's tensors on `device` from the spec's seed.

    p ~ N(0, 1) (for the remainder form: the bf16 rounding of such a draw,
    zero replaced by one, as the high half and a uniform int16 remainder),
    m = v = 0, and
    g ~ N(0, grad_std^2) in the grad dtype.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed)
    n = len(spec.sizes)
    params, ms, vs, gs, outs, rems = [], [], [], [], [], []
    buckets: Dict[str, torch.Tensor] = {}
    xoff = None
    if spec.exchange_ranks > 0:
        xoff = exchange_offsets(spec.sizes, spec.exchange_align)
        L = (xoff[-1] + spec.sizes[-1]) if spec.sizes else 0
        buckets["g"] = torch.zeros(L, dtype=spec.g_dtype, device=dev)
        buckets["p_out"] = torch.zeros(L, dtype=spec.out_dtype, device=dev)
    if spec.bucket_offsets is not None:
        L = spec.bucket_len
        buckets["p"] = torch.zeros(L, dtype=torch.bfloat16, device=dev)
        buckets["rem"] = torch.zeros(L, dtype=torch.int16, device=dev)
        buckets["m"] = torch.zeros(L, dtype=torch.float32, device=dev)
        buckets["v"] = torch.zeros(L, dtype=torch.float32, device=dev)
        buckets["g"] = torch.zeros(L, dtype=spec.g_dtype, device=dev)
    for i in range(n):
        s = spec.sizes[i]
        if spec.bucket_offsets is not None:
            o = spec.bucket_offsets[i]
            p = buckets["p"][o:o + s]
            r = buckets["rem"][o:o + s]
            m = buckets["m"][o:o + s]
            v = buckets["v"][o:o + s]
            g = buckets["g"][o:o + s]
        else:
            sdt = torch.float32 if spec.remainders else spec.state_dtype
            mdt = spec.moment_dtype if spec.moment_dtype is not None else sdt
            p = torch.empty(s, dtype=torch.bfloat16 if spec.remainders else sdt, device=dev)
            r = torch.empty(s, dtype=torch.int16, device=dev) if spec.remainders else None
            m = torch.zeros(s, dtype=mdt, device=dev)
            v = torch.zeros(s, dtype=mdt, device=dev)
            g = torch.empty(s, dtype=spec.g_dtype, device=dev)
            if xoff is not None:
                g = buckets["g"][xoff[i]:xoff[i] + s]
        if spec.remainders:
            hi = torch.randn(s, generator=gen, device=dev).to(torch.bfloat16)
            # a zero high half with a negative remainder is the split of no
            # finite master (it packs to a NaN pattern): draw nonzero halves
            hi[hi == 0] = 1.0
            p.copy_(hi)
            r.copy_(torch.randint(-32768, 32768, (s,), generator=gen, device=dev,
                                  dtype=torch.int32).to(torch.int16))
        elif spec.scaled_state:
            p.copy_((torch.randn(s, generator=gen, device=dev) * 1000).to(p.dtype))
            m.copy_((torch.randn(s, generator=gen, device=dev) * 1000).to(m.dtype))
            v.copy_((torch.randn(s, generator=gen, device=dev) * 1000).abs().to(v.dtype))
        else:
            p.copy_(torch.randn(s, generator=gen, device=dev).to(p.dtype))
        g.copy_((torch.randn(s, generator=gen, device=dev) * spec.grad_std).to(spec.g_dtype))
        params.append(p)
        ms.append(m)
        vs.append(v)
        gs.append(g)
        rems.append(r)
        if spec.remainders:
            outs.append(p)  # the new high half replaces the bf16 param in place
        elif xoff is not None:
            outs.append(buckets["p_out"][xoff[i]:xoff[i] + s])
        elif spec.out_dtype is not None:
            outs.append(torch.zeros(s, dtype=spec.out_dtype, device=dev))
        else:
            outs.append(None)
    sources = dests = None
    if xoff is not None:
        # rows padded to 64 elements, so every row starts 128-byte aligned
        L = buckets["g"].numel()
        Lp = (L + 63) // 64 * 64
        sources = torch.empty(spec.exchange_ranks, Lp, dtype=spec.g_dtype, device=dev)
        for r in range(spec.exchange_ranks):
            sources[r].copy_((torch.randn(Lp, generator=gen, device=dev) * spec.grad_std)
                             .to(spec.g_dtype))
        sources = sources[:, :L]
        dests = torch.zeros(spec.exchange_dests, Lp, dtype=spec.out_dtype, device=dev)[:, :L]
    scales = None
    if spec.scaled_state:
        scales = torch.tensor([list(spec.scale_of)] * n, dtype=torch.float32, device=dev).reshape(n, 3)
    return Shard(spec, params, ms, vs, gs, outs, rems, buckets, sources, dests, xoff, scales)


def inf_position(spec: ShardSpec) -> tuple:
    """(tensor index, element index) of the seeded +inf gradient."""
    rng = np.random.default_rng(spec.seed + 77)
    t = int(rng.integers(0, len(spec.sizes)))
    return t, int(rng.integers(0, spec.sizes[t]))


def fresh_grads(shard: Shard, step: int) -> None:
    """Redraw every gradient in place for `step` (same recipe, new seed)."""
    spec = shard.spec
    dev = shard.grads[0].device if shard.grads else torch.device("cpu")
    gen = torch.Generator(device=dev)
    gen.manual_seed(spec.seed * 7919 + step)
    for g in shard.grads:
        g.copy_((torch.randn(g.numel(), generator=gen, device=dev) * spec.grad_std).to(g.dtype))
