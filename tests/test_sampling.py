"""The full-size parity sample holds a route of every plan block (host logic)."""

import types

import numpy as np
import torch

from oracle import moe as O
from tests.sampling import block_cover_tokens


def _fake_problem(M, k, E, bm, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(M)])
    ids[rng.random(ids.shape) < 0.05] = -1
    sorted_ids, expert_ids, P = O.moe_plan(ids, E, bm)
    cap = P + 3 * bm
    s = np.full(cap, -7, dtype=np.int32)                   # garbage past P
    s[:P] = sorted_ids
    e = np.full(cap // bm, 12345, dtype=np.int32)
    e[:P // bm] = expert_ids
    cfg = types.SimpleNamespace(M=M, top_k=k, E=E, block_m=bm, R=M * k)
    prob = types.SimpleNamespace(cfg=cfg, sorted_ids=torch.from_numpy(s), expert_ids=torch.from_numpy(e),
                                 ntpp=torch.tensor([P], dtype=torch.int32))
    return prob, ids, sorted_ids, P


def test_block_cover_tokens_hit_every_block():
    for seed, (M, k, E, bm) in enumerate([(300, 4, 7, 16), (1000, 8, 40, 64), (57, 3, 5, 8)]):
        prob, ids, sorted_ids, P = _fake_problem(M, k, E, bm, seed)
        tokens = block_cover_tokens(prob)
        assert np.all(np.diff(tokens) > 0) and tokens.min() >= 0 and tokens.max() < M
        held = sorted_ids.reshape(-1, bm)
        for b in range(P // bm):
            routes = held[b][held[b] < M * k]
            assert np.isin(routes // k, tokens).any(), (seed, b)
        # rows other than the first of their block are sampled too
        pos = [np.nonzero(np.isin(held[b] // k, tokens) & (held[b] < M * k))[0] for b in range(P // bm)]
        assert any((p > 0).any() for p in pos)
