"""Router oracle: top-k expert selection and route weights from router logits.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the router only as the companion kernel of the expert path
(FlashInfer pull request #4287, description, "Related Issues": companion
router #4339; the serving traces list ``kernel_alpha_moe_fused_router`` ahead
of the expert kernel).  They give no formula, so this module states the
plainest reading of "softmax, top-k, renormalised weights, routed scale":

* the selected experts are the ``top_k`` largest logits of the token; equal
  logits are taken in ascending expert index (the selection compares input
  values only, so it is exact);
* ``renormalize``: the weights are the softmax over the selected logits,
  ``exp(l_j - m) / sum_{i in S} exp(l_i - m)``, which equals the full softmax
  renormalised over the selection (its denominator cancels);
* otherwise: the full-softmax probabilities of the selected experts,
  ``exp(l_j - m) / sum_{all i} exp(l_i - m)``;
* the weights are then multiplied by ``routed_scale``;
* ids and weights are listed in selection order (descending logit, ties by
  index).

Everything is computed in float64 from the logits' exact values.
"""

import numpy as np


def topk_select(logits, top_k):
    """[M, E] logits -> [M, top_k] int64 ids: descending value, ascending index
    among equal values."""
    l = np.asarray(logits, dtype=np.float64)
    M, E = l.shape
    if not 1 <= top_k <= E:
        raise ValueError("need 1 <= top_k <= E")
    ids = np.empty((M, top_k), dtype=np.int64)
    idx = np.arange(E)
    for t in range(M):
        # primary key -logit, secondary key expert index (lexsort: last key first)
        order = np.lexsort((idx, -l[t]))
        ids[t] = order[:top_k]
    return ids


def route_topk(logits, top_k, routed_scale=1.0, renormalize=True):
    """[M, E] logits -> (ids [M, top_k] int64, weights [M, top_k] float64)."""
    l = np.asarray(logits, dtype=np.float64)
    ids = topk_select(l, top_k)
    sel = np.take_along_axis(l, ids, axis=1)
    m = l.max(axis=1, keepdims=True)
    num = np.exp(sel - m)
    den = num.sum(axis=1, keepdims=True) if renormalize else np.exp(l - m).sum(axis=1, keepdims=True)
    return ids, num / den * routed_scale
