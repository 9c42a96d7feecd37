"""Token samples for the full-size parity tests (host logic only).

Tokens are independent in the forward, so the oracle can check a full-size
run exactly on a subset of its tokens.  The subset is chosen from the plan
the GPU built (which the plan tests compare bit for bit with the oracle's);
only the choice of tokens depends on it, never an expected value.
"""

import numpy as np


def block_cover_tokens(prob):
    """Tokens that together hold a route in every plan block below P.

    Each block contributes the route at a row position that moves from block
    to block (position (37 b) mod the block's route count), so the sample
    reaches every plan block, first and last rows alike, every TMEM lane
    quarter of the tiles and both CTAs of a pair."""
    cfg = prob.cfg
    bm = cfg.block_m
    P = int(prob.ntpp.item())
    ids = prob.sorted_ids[:P].cpu().numpy().reshape(-1, bm)
    experts = prob.expert_ids[:P // bm].cpu().numpy()
    tokens = set()
    for b in range(ids.shape[0]):
        live = np.nonzero(ids[b] < cfg.R)[0]
        if live.size == 0 or not 0 <= experts[b] < cfg.E:
            continue
        tokens.add(int(ids[b, live[(37 * b) % live.size]]) // cfg.top_k)
    return np.asarray(sorted(tokens), dtype=np.int64)
