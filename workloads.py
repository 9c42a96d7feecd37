"""Seeded synthetic workloads for the block-scaled FP8 MoE path.

This module only draws random numbers and builds routings; it holds none of
the method's arithmetic (no quantisation, no plan, no GEMM).  It sits beside,
not inside, the library package and the oracle: each of them imports it and
neither imports the other.  Both consume what it produces: raw BF16 activations and
weights are quantised afterwards, by the oracle's quantiser on the CPU side
and by the library's quantiser kernels on the GPU side.

The shapes and distributions follow the workloads the pages measure
(FlashInfer PR #4287, "Final W8 kernel performance (v46)" fixtures; the
sglang-glm53-flash-sm120 PR #13 timing shape E288/H4096/I1024/top-8):

* activations BF16 ~ N(0, 1); weights BF16 ~ N(0, 0.02);
* routing either softmax-top-k of N(0,1) router logits with renormalised
  weights, or k distinct experts drawn uniformly with weights = softmax of k
  N(0,1) logits, or the skewed mix (hot experts + Zipf tail + masked routes);
* the prior output either zero or BF16 ~ N(0, 0.1).

Every tensor has its own stream: seed * 1000 + stream id, and weights one
sub-stream per expert, so one expert's weights can be regenerated alone.
"""

from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

STREAM_ACT = 1
STREAM_W13 = 2
STREAM_W2 = 3
STREAM_ROUTE = 4
STREAM_OUT = 5
STREAM_MASK = 6
STREAM_GARBAGE = 7


@dataclass(frozen=True)
class MoEConfig:
    name: str
    M: int
    H: int
    I: int
    E: int
    top_k: int
    block_m: int
    routing: str = "uniform"          # "softmax_topk" | "uniform" | "skewed"
    out_init: str = "zero"            # "zero" | "normal0.1"
    id_dtype: torch.dtype = torch.int32
    ue8m0: bool = False               # weight block scales requantised to powers of two
    act_ue8m0: bool = False           # activations quantised with power-of-two group scales
    routed_scale: float = 1.0
    garbage_plan: bool = False        # fill plan buffers with random bits first
    masked_frac: float = 0.0
    n_hot: int = 0
    hot_frac: float = 0.0
    zipf_s: float = 1.1
    n_zero_scale: int = 0
    seed: int = 0

    @property
    def N(self):
        return 2 * self.I

    @property
    def R(self):
        return self.M * self.top_k

    def with_(self, **kw):
        return replace(self, **kw)


def _gen(seed, stream, sub=0, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(stream) * 7919 + int(sub))
    return g


# The five workloads: tiny, decode (three token counts), prefill sweep (four
# token counts), skewed routing and large.
CONFIGS = {
    "tiny": MoEConfig("tiny", M=16, H=256, I=256, E=8, top_k=2, block_m=64,
                      routing="softmax_topk", out_init="normal0.1"),
    "decode_m1": MoEConfig("decode_m1", M=1, H=7168, I=256, E=257, top_k=9, block_m=64,
                           garbage_plan=True),
    "decode_m8": MoEConfig("decode_m8", M=8, H=7168, I=256, E=257, top_k=9, block_m=64,
                           garbage_plan=True),
    "decode_m64": MoEConfig("decode_m64", M=64, H=7168, I=256, E=257, top_k=9, block_m=64,
                            garbage_plan=True),
    "prefill_1024": MoEConfig("prefill_1024", M=1024, H=4096, I=1024, E=288, top_k=8, block_m=128),
    "prefill_2048": MoEConfig("prefill_2048", M=2048, H=4096, I=1024, E=288, top_k=8, block_m=128),
    "prefill_4096": MoEConfig("prefill_4096", M=4096, H=4096, I=1024, E=288, top_k=8, block_m=128),
    "prefill_8192": MoEConfig("prefill_8192", M=8192, H=4096, I=1024, E=288, top_k=8, block_m=128),
    "skewed": MoEConfig("skewed", M=4096, H=4096, I=512, E=512, top_k=10, block_m=128,
                        routing="skewed", masked_frac=0.05, n_hot=4, hot_frac=0.5,
                        n_zero_scale=2),
    "large": MoEConfig("large", M=8192, H=7168, I=1024, E=257, top_k=9, block_m=128,
                       out_init="normal0.1", id_dtype=torch.int64, ue8m0=True),
}


@dataclass
class Routing:
    topk_ids: torch.Tensor            # [M, k] int32/int64 (CPU)
    topk_weights: torch.Tensor        # [M, k] float32 (CPU)
    zero_scale_experts: List[int] = field(default_factory=list)
    hot_experts: List[int] = field(default_factory=list)


def _softmax_topk(cfg, g):
    logits = torch.randn(cfg.M, cfg.E, generator=g, dtype=torch.float32)
    probs = torch.softmax(logits, dim=-1)
    vals, ids = torch.topk(probs, cfg.top_k, dim=-1)
    w = vals / vals.sum(dim=-1, keepdim=True)
    return ids, w


def _uniform(cfg, g):
    keys = torch.rand(cfg.M, cfg.E, generator=g, dtype=torch.float32)
    ids = torch.topk(keys, cfg.top_k, dim=-1).indices
    logits = torch.randn(cfg.M, cfg.top_k, generator=g, dtype=torch.float32)
    w = torch.softmax(logits, dim=-1)
    return ids, w


def _skewed(cfg, g):
    """Hot experts take each slot with probability hot_frac; the rest follow
    Zipf(s) over the remaining experts; duplicates within a token are redrawn."""
    E, k = cfg.E, cfg.top_k
    perm = torch.randperm(E, generator=g)
    hot = perm[: cfg.n_hot]
    tail = perm[cfg.n_hot:]
    ranks = torch.arange(1, tail.numel() + 1, dtype=torch.float64)
    zipf_p = ranks ** (-cfg.zipf_s)
    zipf_p = zipf_p / zipf_p.sum()
    ids = torch.empty(cfg.M, k, dtype=torch.int64)
    for t in range(cfg.M):
        chosen = []
        while len(chosen) < k:
            if torch.rand(1, generator=g).item() < cfg.hot_frac:
                e = int(hot[torch.randint(cfg.n_hot, (1,), generator=g)].item())
            else:
                e = int(tail[torch.multinomial(zipf_p, 1, generator=g)].item())
            if e not in chosen:
                chosen.append(e)
        ids[t] = torch.tensor(chosen)
    logits = torch.randn(cfg.M, k, generator=g, dtype=torch.float32)
    w = torch.softmax(logits, dim=-1)
    zero = [int(tail[0]), int(tail[1])][: cfg.n_zero_scale]
    return ids, w, hot.tolist(), zero


def make_routing(cfg: MoEConfig) -> Routing:
    g = _gen(cfg.seed, STREAM_ROUTE)
    hot, zero = [], []
    if cfg.routing == "softmax_topk":
        ids, w = _softmax_topk(cfg, g)
    elif cfg.routing == "uniform":
        ids, w = _uniform(cfg, g)
    elif cfg.routing == "skewed":
        ids, w, hot, zero = _skewed(cfg, g)
    else:
        raise ValueError(cfg.routing)
    ids = ids.to(torch.int64)
    if cfg.masked_frac > 0:
        gm = _gen(cfg.seed, STREAM_MASK)
        n_mask = int(round(cfg.masked_frac * cfg.R))
        pick = torch.randperm(cfg.R, generator=gm)[:n_mask]
        flat = ids.reshape(-1).clone()
        flat[pick] = -1
        ids = flat.reshape(cfg.M, cfg.top_k)
    return Routing(ids.to(cfg.id_dtype).contiguous(), w.to(torch.float32).contiguous(), zero, hot)


def make_activations(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """BF16 [M, H] ~ N(0, 1)."""
    g = _gen(cfg.seed, STREAM_ACT, device=device)
    return torch.randn(cfg.M, cfg.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_expert_weights(cfg: MoEConfig, e: int, which: str, device="cpu") -> torch.Tensor:
    """One expert's BF16 weights ~ N(0, 0.02): W13 [2I, H] (gate rows, then up
    rows) or W2 [H, I]."""
    if which == "w13":
        g = _gen(cfg.seed, STREAM_W13, e, device=device)
        shape = (cfg.N, cfg.H)
    elif which == "w2":
        g = _gen(cfg.seed, STREAM_W2, e, device=device)
        shape = (cfg.H, cfg.I)
    else:
        raise ValueError(which)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)


def make_weights(cfg: MoEConfig, which: str, experts: Optional[List[int]] = None, device="cpu"):
    """Stacked BF16 weights of the given experts (all by default)."""
    experts = range(cfg.E) if experts is None else experts
    return torch.stack([make_expert_weights(cfg, e, which, device) for e in experts])


def make_out_prior(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    if cfg.out_init == "zero":
        return torch.zeros(cfg.M, cfg.H, device=device, dtype=torch.bfloat16)
    g = _gen(cfg.seed, STREAM_OUT, device=device)
    return (torch.randn(cfg.M, cfg.H, generator=g, device=device, dtype=torch.float32) * 0.1).to(torch.bfloat16)


def garbage_int32(n: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Random 32-bit patterns used to pre-fill plan buffers."""
    g = _gen(seed, STREAM_GARBAGE, device=device)
    return torch.randint(-2 ** 31, 2 ** 31 - 1, (n,), generator=g, device=device, dtype=torch.int64).to(torch.int32)
