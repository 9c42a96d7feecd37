"""GPU parity of moe_route_topk against the router oracle: the ids bit for
bit (the selection compares input values only), the weights within FP32
rounding of the float64 oracle."""

import numpy as np
import pytest
import torch

from fp8_block_scale_gb300 import _lib as L
from oracle import moe as O
from oracle import router as R

pytestmark = pytest.mark.gpu
WEIGHT_RTOL = 4e-6   # expf (a few ulp) and an FP32 sum of at most 2048 terms


@pytest.fixture(scope="module", autouse=True)
def _load():
    L.load()


def _run(logits_np, top_k, dtype=torch.float32, id_dtype=torch.int32, routed_scale=1.0, renormalize=True):
    M, E = logits_np.shape
    lg = torch.from_numpy(logits_np.astype(np.float32)).to(dtype).cuda()
    ids = torch.full((M, top_k), -7, dtype=id_dtype, device="cuda")
    w = torch.full((M, top_k), float("nan"), dtype=torch.float32, device="cuda")
    L.moe_route_topk(lg, top_k, ids, w, routed_scale, renormalize)
    torch.cuda.synchronize()
    exact = lg.float().cpu().numpy().astype(np.float64)   # the values the kernel saw
    rid, rw = R.route_topk(exact, top_k, routed_scale, renormalize)
    return ids.cpu().numpy(), w.cpu().numpy(), rid, rw


CASES = [
    # (M, E, top_k, logits)
    (1, 257, 9, "normal"),          # decode router
    (8192, 288, 8, "normal"),       # prefill router
    (300, 512, 10, "normal"),
    (64, 2048, 32, "normal"),       # the largest E and top_k
    (33, 24, 24, "normal"),         # top_k = E
    (100, 64, 6, "ties"),           # many equal logits
    (50, 7, 1, "normal"),           # E < 32
    (17, 1, 1, "normal"),           # one expert
]


@pytest.mark.parametrize("M,E,k,kind", CASES)
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_route_topk_matches_oracle(M, E, k, kind, dtype):
    rng = np.random.default_rng(M * 7 + E * 3 + k)
    if kind == "ties":
        logits = rng.integers(-2, 3, size=(M, E)).astype(np.float32)
    else:
        logits = rng.standard_normal((M, E)).astype(np.float32) * 2.0
    ids, w, rid, rw = _run(logits, k, dtype)
    assert np.array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


def test_route_topk_int64_ids_plain_softmax_and_scale():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((500, 257)).astype(np.float32)
    ids, w, rid, rw = _run(logits, 9, id_dtype=torch.int64, routed_scale=2.5, renormalize=False)
    assert ids.dtype == np.int64 and np.array_equal(ids, rid)
    np.testing.assert_allclose(w, rw, rtol=WEIGHT_RTOL, atol=0)


def test_route_topk_feeds_the_plan():
    """Router output straight into moe_plan gives the oracle's plan."""
    rng = np.random.default_rng(9)
    M, E, k, bm = 700, 96, 6, 64
    logits = torch.from_numpy(rng.standard_normal((M, E)).astype(np.float32)).cuda()
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    L.moe_route_topk(logits, k, ids, w)
    cap = -(-(M * k + E * (bm - 1)) // bm) * bm
    sorted_ids = torch.empty(cap, dtype=torch.int32, device="cuda")
    expert_ids = torch.empty(cap // bm, dtype=torch.int32, device="cuda")
    ntpp = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device="cuda")
    L.moe_plan(ids, E, bm, sorted_ids, expert_ids, ntpp, ws)
    torch.cuda.synchronize()
    rid, _ = R.route_topk(logits.cpu().numpy().astype(np.float64), k)
    rs, rb, rP = O.moe_plan(rid, E, bm)
    P = int(ntpp.item())
    assert P == rP
    assert np.array_equal(sorted_ids[:P].cpu().numpy(), rs)
    assert np.array_equal(expert_ids[:P // bm].cpu().numpy(), rb)


# ------------------------------------------------------------ router + plan in one launch

ROUTE_PLAN_CASES = [
    # (M, E, top_k, block_m, logit dtype, id dtype, renormalize)
    (1, 257, 9, 64, torch.float32, torch.int32, True),      # decode_m1
    (8, 257, 9, 64, torch.bfloat16, torch.int64, True),     # decode_m8, BF16 logits, int64 ids
    (64, 257, 9, 64, torch.float32, torch.int32, False),    # decode_m64, plain softmax weights
    (113, 288, 9, 16, torch.float32, torch.int32, True),    # 1017 routes, ragged blocks
    (1024, 1024, 1, 128, torch.float32, torch.int32, True), # the largest R and E
    (16, 8, 2, 8, torch.float32, torch.int32, True),        # E < 32
    (0, 64, 4, 64, torch.float32, torch.int32, True),       # no tokens: an empty plan
]


@pytest.mark.parametrize("M,E,k,bm,dtype,id_dtype,renorm", ROUTE_PLAN_CASES,
                         ids=[f"m{c[0]}-e{c[1]}-k{c[2]}-bm{c[3]}" for c in ROUTE_PLAN_CASES])
def test_route_plan_matches_the_two_calls(M, E, k, bm, dtype, id_dtype, renorm):
    """moe_route_plan writes the same ids, weights and plan, byte for byte,
    as moe_route_topk followed by moe_plan on the same logits (every
    capacity entry compared, including the pads and the blocks past P)."""
    rng = np.random.default_rng(M * 31 + E + k)
    logits = torch.from_numpy((rng.standard_normal((max(M, 1), E)) * 2.0).astype(np.float32)[:M]).to(dtype).cuda()
    cap, bcap = L.moe_plan_capacity(M, k, E, bm)

    def buffers():
        return (torch.full((M, k), -7, dtype=id_dtype, device="cuda"),
                torch.full((M, k), float("nan"), dtype=torch.float32, device="cuda"),
                torch.full((cap,), -3, dtype=torch.int32, device="cuda"),
                torch.full((bcap,), -3, dtype=torch.int32, device="cuda"),
                torch.full((1,), -3, dtype=torch.int32, device="cuda"))

    ids1, w1, s1, e1, p1 = buffers()
    if M > 0:
        L.moe_route_topk(logits, k, ids1, w1, 2.5, renorm)
    ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device="cuda")
    L.moe_plan(ids1, E, bm, s1, e1, p1, ws)
    ids2, w2, s2, e2, p2 = buffers()
    L.moe_route_plan(logits, k, ids2, w2, bm, s2, e2, p2, 2.5, renorm)
    torch.cuda.synchronize()
    assert torch.equal(ids1, ids2)
    assert torch.equal(w1.view(torch.int32), w2.view(torch.int32))
    assert int(p1.item()) == int(p2.item())
    assert torch.equal(s1, s2)
    assert torch.equal(e1, e2)
    if M > 0:
        exact = logits.float().cpu().numpy().astype(np.float64)
        rid, rw = R.route_topk(exact, k, 2.5, renorm)
        assert np.array_equal(ids2.cpu().numpy(), rid)
        np.testing.assert_allclose(w2.cpu().numpy(), rw, rtol=WEIGHT_RTOL, atol=0)
