"""Oracle-side inputs of a workload, and the comparison metrics.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The oracle never sees
a value produced by the CUDA library: its inputs are the raw BF16 values
regenerated from the seeded generator module (which holds none of the
method's arithmetic) and quantised by the oracle's own quantiser.
"""

import numpy as np
import torch

from fp8_block_scale_gb300 import workloads as W
from . import moe as O
from . import w4a8 as OW
from .numerics import e4m3_decode

# The numerical acceptance bar of the forward: relative L2 error of `out`,
# max |diff| relative to max |ref|, and the intermediate FP8 codes: at most
# 0.1% may differ, each to an adjacent E4M3 value.
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2
CODE_DIFF_FRAC = 1e-3

_E4M3_SORTED = np.unique(np.abs(e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))


def oracle_inputs(cfg, routing, tokens, device=None):
    """Oracle inputs for `tokens`: a compact problem over the experts they touch.

    Raw values are drawn on `device` (CUDA when available, as the GPU side
    draws them, else CPU) and copied to the host before quantisation.
    """
    if device is None:
        device = "cuda" if torch.cuda.is_available() else "cpu"
    tokens = np.asarray(tokens, dtype=np.int64)
    ids = routing.topk_ids.to(torch.int64).numpy()[tokens]
    experts = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < cfg.E})
    remap = {e: i for i, e in enumerate(experts)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids], dtype=np.int64)
    x = W.make_activations(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    a_q, a_s = O.quantize_act_1x128_ue8m0(x) if cfg.act_ue8m0 else O.quantize_act_1x128(x)
    w13_q, w13_s, w2_q, w2_s = [], [], [], []
    for e in experts:
        q, s = O.quantize_weight_128x128(W.make_expert_weights(cfg, e, "w13", device).float().cpu().numpy()[None])
        q2, s2 = O.quantize_weight_128x128(W.make_expert_weights(cfg, e, "w2", device).float().cpu().numpy()[None])
        if e in routing.zero_scale_experts:
            s[:] = 0
            s2[:] = 0
        if cfg.ue8m0:
            q, s, _ = O.requant_scales_ue8m0(q, s)
            q2, s2, _ = O.requant_scales_ue8m0(q2, s2)
        w13_q.append(q[0]); w13_s.append(s[0]); w2_q.append(q2[0]); w2_s.append(s2[0])
    if not experts:
        N, H, I = cfg.N, cfg.H, cfg.I
        w13_q, w13_s = [np.zeros((N, H), np.uint8)], [np.zeros((N // 128, H // 128), np.float32)]
        w2_q, w2_s = [np.zeros((H, I), np.uint8)], [np.zeros((H // 128, I // 128), np.float32)]
    prior = W.make_out_prior(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    inp = dict(a_q=a_q, a_s=a_s, w13_q=np.stack(w13_q), w13_s=np.stack(w13_s), w2_q=np.stack(w2_q),
               w2_s=np.stack(w2_s), topk_ids=ids_c, topk_w=routing.topk_weights.numpy()[tokens], out_prior=prior)
    return inp, experts


def oracle_inputs_w4a8(cfg, routing, tokens, device=None):
    """Oracle inputs of the E2M1-K32 x FP8 forward for `tokens` (oracle.w4a8),
    from the same raw values as ``oracle_inputs``: a compact problem over the
    experts the tokens touch, weights as unpacked E2M1 codes."""
    if device is None:
        device = "cuda" if torch.cuda.is_available() else "cpu"
    tokens = np.asarray(tokens, dtype=np.int64)
    ids = routing.topk_ids.to(torch.int64).numpy()[tokens]
    experts = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < cfg.E})
    remap = {e: i for i, e in enumerate(experts)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids], dtype=np.int64)
    x = W.make_activations(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    a_q, a_s = OW.quantize_act_per_row(x)
    w13_q, w13_s, w2_q, w2_s = [], [], [], []
    for e in experts:
        q, s = OW.quantize_weight_k32(W.make_expert_weights(cfg, e, "w13", device).float().cpu().numpy())
        q2, s2 = OW.quantize_weight_k32(W.make_expert_weights(cfg, e, "w2", device).float().cpu().numpy())
        if e in routing.zero_scale_experts:
            s[:] = 0
            s2[:] = 0
        w13_q.append(q); w13_s.append(s); w2_q.append(q2); w2_s.append(s2)
    if not experts:
        N, H, I = cfg.N, cfg.H, cfg.I
        w13_q, w13_s = [np.zeros((N, H), np.uint8)], [np.zeros((N, H // 32), np.float32)]
        w2_q, w2_s = [np.zeros((H, I), np.uint8)], [np.zeros((H, I // 32), np.float32)]
    prior = W.make_out_prior(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    inp = dict(a_q=a_q, a_s=a_s, w13_q=np.stack(w13_q), w13_s=np.stack(w13_s), w2_q=np.stack(w2_q),
               w2_s=np.stack(w2_s), topk_ids=ids_c, topk_w=routing.topk_weights.numpy()[tokens], out_prior=prior)
    return inp, experts


def out_metrics(got, ref, prior=None):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    rel = np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(d).max() / max(np.abs(ref).max(), 1e-30)
    res = {"rel_l2": float(rel), "max_rel": float(mx)}
    if prior is not None:
        delta = ref - np.asarray(prior, dtype=np.float64)
        res["rel_l2_delta"] = float(np.linalg.norm(d) / max(np.linalg.norm(delta), 1e-30))
    return res


def bf16_ulps(a, b):
    """Distance in BF16 steps between two float32 arrays holding BF16 values:
    the bit patterns mapped to integers that increase with the value (+0 and
    -0 coincide), then subtracted."""
    def ordered(x):
        bits = (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.int64)
        return np.where(bits & 0x8000, 0x8000 - bits, bits)
    return np.abs(ordered(a) - ordered(b))


def code_diffs(got_codes, ref_codes):
    """(number of differing codes, number of differences that are not to an
    adjacent E4M3 value).  +0 and -0 count as equal."""
    g = e4m3_decode(np.asarray(got_codes, dtype=np.uint8))
    r = e4m3_decode(np.asarray(ref_codes, dtype=np.uint8))
    diff = g != r
    n = int(diff.sum())
    if n == 0:
        return 0, 0
    gi = np.searchsorted(_E4M3_SORTED, np.abs(g[diff]))
    ri = np.searchsorted(_E4M3_SORTED, np.abs(r[diff]))
    same_sign = (np.sign(g[diff]) == np.sign(r[diff])) | (g[diff] == 0) | (r[diff] == 0)
    adjacent = same_sign & (np.abs(gi - ri) <= 1)
    return n, int((~adjacent).sum())
