"""Oracle-side inputs of a workload, and the comparison metrics.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The oracle never sees
a value produced by the CUDA library: its inputs are the raw BF16 values
regenerated from the seeded generator module (which holds none of the
method's arithmetic) and quantised by the oracle's own quantiser.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import workloads as W
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


def default_workers():
    """Threads for the oracle's per-expert work: the host's cores, at most 16
    (numpy releases the interpreter lock inside its array kernels)."""
    return max(1, min(16, os.cpu_count() or 1))


# Oracle-quantised weights per expert, kept for the life of the process: the
# prefill workloads share one weight set, and a full-size check touches every
# expert.  The key holds everything the expert's codes depend on.
_WEIGHT_CACHE = {}


def _expert_weights(cfg, routing, experts, device, kind, quantize, workers):
    """{expert: (w13 codes, w13 scales, w2 codes, w2 scales)} from the oracle's
    own quantiser.  Raw values are drawn in this thread (on `device`, where
    the library draws them too); the quantisation runs in a thread pool, a
    bounded number of experts in flight."""
    def key(e):
        return (kind, str(device), cfg.seed, cfg.H, cfg.I, cfg.ue8m0, e, e in routing.zero_scale_experts)

    todo = [e for e in experts if key(e) not in _WEIGHT_CACHE]

    def work(e, raw13, raw2):
        q, s, q2, s2 = quantize(raw13, raw2)
        if e in routing.zero_scale_experts:
            s[:] = 0
            s2[:] = 0
        return q, s, q2, s2

    workers = workers or default_workers()
    with ThreadPoolExecutor(max_workers=workers) as pool:
        for c0 in range(0, len(todo), 2 * workers):
            chunk = todo[c0:c0 + 2 * workers]
            futs = []
            for e in chunk:
                raw13 = W.make_expert_weights(cfg, e, "w13", device).float().cpu().numpy()
                raw2 = W.make_expert_weights(cfg, e, "w2", device).float().cpu().numpy()
                futs.append(pool.submit(work, e, raw13, raw2))
            for e, f in zip(chunk, futs):
                _WEIGHT_CACHE[key(e)] = f.result()
    return {e: _WEIGHT_CACHE[key(e)] for e in experts}


def _quantize_fp8_expert(ue8m0):
    def quantize(raw13, raw2):
        q, s = O.quantize_weight_128x128(raw13[None])
        q2, s2 = O.quantize_weight_128x128(raw2[None])
        if ue8m0:
            q, s, _ = O.requant_scales_ue8m0(q, s)
            q2, s2, _ = O.requant_scales_ue8m0(q2, s2)
        return q[0], s[0], q2[0], s2[0]
    return quantize


def _quantize_w4a8_expert(raw13, raw2):
    q, s = OW.quantize_weight_k32(raw13)
    q2, s2 = OW.quantize_weight_k32(raw2)
    return q, s, q2, s2


def _compact(cfg, routing, tokens, device, kind, quantize, workers, act_quant, empty_scales):
    if device is None:
        device = "cuda" if torch.cuda.is_available() else "cpu"
    tokens = np.asarray(tokens, dtype=np.int64)
    ids = routing.topk_ids.to(torch.int64).numpy()[tokens]
    experts = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < cfg.E})
    remap = {e: i for i, e in enumerate(experts)}
    ids_c = np.array([[remap.get(int(e), -1) for e in row] for row in ids], dtype=np.int64)
    x = W.make_activations(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    a_q, a_s = act_quant(x)
    weights = _expert_weights(cfg, routing, experts, device, kind, quantize, workers)
    if experts:
        w13_q, w13_s, w2_q, w2_s = (np.stack([weights[e][i] for e in experts]) for i in range(4))
    else:
        N, H, I = cfg.N, cfg.H, cfg.I
        s13, s2 = empty_scales
        w13_q, w13_s = np.zeros((1, N, H), np.uint8), np.zeros((1,) + s13, np.float32)
        w2_q, w2_s = np.zeros((1, H, I), np.uint8), np.zeros((1,) + s2, np.float32)
    prior = W.make_out_prior(cfg, device=device)[torch.as_tensor(tokens, device=device)].float().cpu().numpy()
    inp = dict(a_q=a_q, a_s=a_s, w13_q=w13_q, w13_s=w13_s, w2_q=w2_q, w2_s=w2_s, topk_ids=ids_c,
               topk_w=routing.topk_weights.numpy()[tokens], out_prior=prior)
    return inp, experts


def oracle_inputs(cfg, routing, tokens, device=None, workers=None):
    """Oracle inputs for `tokens`: a compact problem over the experts they touch.

    Raw values are drawn on `device` (CUDA when available, as the GPU side
    draws them, else CPU) and copied to the host before quantisation by the
    oracle's quantisers; `workers` threads quantise the experts' weights.
    """
    def act(x):
        return O.quantize_act_1x128_ue8m0(x) if cfg.act_ue8m0 else O.quantize_act_1x128(x)
    return _compact(cfg, routing, tokens, device, "fp8", _quantize_fp8_expert(cfg.ue8m0), workers, act,
                    ((cfg.N // 128, cfg.H // 128), (cfg.H // 128, cfg.I // 128)))


def oracle_inputs_w4a8(cfg, routing, tokens, device=None, workers=None):
    """Oracle inputs of the E2M1-K32 x FP8 forward for `tokens` (oracle.w4a8),
    from the same raw values as ``oracle_inputs``: a compact problem over the
    experts the tokens touch, weights as unpacked E2M1 codes."""
    return _compact(cfg, routing, tokens, device, "w4a8", _quantize_w4a8_expert, workers, OW.quantize_act_per_row,
                    ((cfg.N, cfg.H // 32), (cfg.H, cfg.I // 32)))


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
