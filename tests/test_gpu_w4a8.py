"""GPU parity of the E2M1-K32 weight x FP8 activation path against its oracle.

The quantisers are compared bit for bit; the forward element by element on
every token of small and ragged problems and of the SM120 page's timing shape
(E288/H4096/I1024/top-8) at decode sizes, with the intermediate codes checked
through the debug hooks.
"""

import numpy as np
import pytest
import torch

from fp8_block_scale_gb300 import _lib as L
import workloads as W
from fp8_block_scale_gb300.problem import W4A8Problem
from oracle import w4a8 as OW
from oracle.inputs import (CODE_DIFF_FRAC, MAX_ABS_TOL, REL_L2_TOL, code_diffs, default_workers, oracle_inputs_w4a8,
                           out_metrics)
from tests.sampling import block_cover_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _load():
    L.load()


def test_quantize_act_per_row_bit_exact():
    g = torch.Generator().manual_seed(31)
    x = torch.randn(37, 4096, generator=g) * torch.logspace(-3, 3, 37)[:, None]
    x[5] = 0.0
    x[6, 100] = -1e4
    xb = x.to(torch.bfloat16)
    q = torch.empty(37, 4096, dtype=torch.uint8, device="cuda")
    s = torch.empty(37, dtype=torch.float32, device="cuda")
    L.moe_quantize_act_per_row(xb.cuda(), q, s)
    torch.cuda.synchronize()
    rq, rs = OW.quantize_act_per_row(xb.float().numpy())
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_quantize_weight_k32_bit_exact():
    g = torch.Generator().manual_seed(32)
    w = torch.randn(3, 96, 256, generator=g) * 0.02
    w[0, 1, 32:64] = 0.0                                   # a zero block
    # a block whose scale is exactly 1 and whose values sit on every tie
    ties = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0,
                         -0.0, 0.1, -0.1, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, -6.0, 0.0, 0.3, 0.6, 2.2, 2.9, 4.4, 5.5])
    w[1, 2, 64:96] = ties
    wb = w.to(torch.bfloat16)
    q = torch.empty(3, 96, 128, dtype=torch.uint8, device="cuda")
    s = torch.empty(3, 96, 8, dtype=torch.float32, device="cuda")
    L.moe_quantize_weight_k32(wb.cuda(), q, s)
    torch.cuda.synchronize()
    rq, rs = OW.quantize_weight_k32(wb.float().numpy())
    np.testing.assert_array_equal(OW.unpack_e2m1(q.cpu().numpy()), rq)
    np.testing.assert_array_equal(q.cpu().numpy(), OW.pack_e2m1(rq))
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert s[1, 2, 2].item() == 1.0


def _run(prob, debug=True, path=L.W4A8_AUTO):
    cap = prob.sorted_ids.numel()
    dq = torch.zeros(cap, prob.cfg.I, dtype=torch.uint8, device="cuda") if debug else None
    ds = torch.zeros(cap, dtype=torch.float32, device="cuda") if debug else None
    prob.run_plan()
    prob.run_forward(prob.fwd_args(dq, ds, path=path))
    torch.cuda.synchronize()
    return dq, ds


def _check(prob, tokens, dq, ds):
    cfg = prob.cfg
    inp, experts = oracle_inputs_w4a8(cfg, prob.routing, tokens)
    # the GPU quantisers saw the same raw values: their codes must match bit for bit
    for i, e in enumerate(experts[:2]):
        assert np.array_equal(OW.unpack_e2m1(prob.w13[e].cpu().numpy()), inp["w13_q"][i]), f"W13 codes of expert {e}"
        assert np.array_equal(prob.w2_scale[e].cpu().numpy().view(np.uint32), inp["w2_s"][i].view(np.uint32))
    ref, inter = OW.moe_forward_w4a8(**inp, routed_scale=cfg.routed_scale, return_inter=True,
                                     workers=default_workers())
    got = prob.out[torch.as_tensor(tokens, device="cuda")].float().cpu().numpy()
    m = out_metrics(got, ref, inp["out_prior"])
    print(f"{cfg.name} tokens={len(tokens)} {m}")
    assert m["rel_l2"] <= REL_L2_TOL, m
    assert m["max_rel"] <= MAX_ABS_TOL, m
    sorted_ids = prob.sorted_ids.cpu().numpy()
    P = int(prob.ntpp.item())
    slot_of = {int(r): s for s, r in enumerate(sorted_ids[:P]) if r < cfg.R}
    dqn, dsn = dq.cpu().numpy(), ds.cpu().numpy()
    n_codes = n_diff = n_far = 0
    for (ti, j), (codes, scale) in inter.items():
        s = slot_of[int(tokens[ti]) * cfg.top_k + j]
        nd, nf = code_diffs(dqn[s], codes)
        n_codes += codes.size
        n_diff += nd
        n_far += nf
        np.testing.assert_allclose(dsn[s], scale, rtol=1e-5, atol=0)
    print(f"   intermediate codes: {n_diff}/{n_codes} differ, {n_far} not adjacent")
    assert n_far == 0
    assert n_diff <= max(1, CODE_DIFF_FRAC * n_codes)
    assert int(prob.status.item()) == 0


CASES = {
    "w4a8_tiny": W.MoEConfig("w4a8_tiny", M=16, H=256, I=128, E=8, top_k=2, block_m=16,
                             routing="softmax_topk", out_init="normal0.1"),
    "w4a8_ragged_bm8": W.MoEConfig("w4a8_ragged_bm8", M=37, H=384, I=96, E=5, top_k=3, block_m=8,
                                   routed_scale=2.5, masked_frac=0.1, id_dtype=torch.int64),
    "w4a8_ragged_bm64": W.MoEConfig("w4a8_ragged_bm64", M=200, H=512, I=160, E=6, top_k=4, block_m=64,
                                    out_init="normal0.1", garbage_plan=True),
    "w4a8_skewed": W.MoEConfig("w4a8_skewed", M=96, H=256, I=256, E=16, top_k=4, block_m=16, routing="skewed",
                               masked_frac=0.05, n_hot=2, hot_frac=0.5, n_zero_scale=1),
    # shapes the tensor-core projections take (H, I multiples of 128): groups
    # of 8 blocks of 8 rows, groups of two 24-row blocks (48 columns), single
    # 64-row blocks over a garbage-filled plan
    "w4a8_tc_bm8": W.MoEConfig("w4a8_tc_bm8", M=37, H=384, I=256, E=5, top_k=3, block_m=8, routed_scale=2.5,
                               masked_frac=0.1, id_dtype=torch.int64),
    "w4a8_tc_bm24": W.MoEConfig("w4a8_tc_bm24", M=120, H=256, I=128, E=6, top_k=2, block_m=24, routing="skewed",
                                n_hot=1, hot_frac=0.6, out_init="normal0.1"),
    "w4a8_tc_bm64": W.MoEConfig("w4a8_tc_bm64", M=200, H=512, I=384, E=6, top_k=4, block_m=64,
                                out_init="normal0.1", garbage_plan=True),
}


@pytest.mark.parametrize("path", [L.W4A8_AUTO, L.W4A8_CUDA_CORES], ids=["auto", "cuda_cores"])
@pytest.mark.parametrize("name", list(CASES))
def test_w4a8_forward_small(name, path):
    """Every case on the automatic choice (the tensor cores where H and I are
    multiples of 128) and on the CUDA cores."""
    prob = W4A8Problem(CASES[name])
    dq, ds = _run(prob, path=path)
    _check(prob, np.arange(prob.cfg.M), dq, ds)


# The SM120 page's timing shape (288 experts, hidden 4096, intermediate 1024,
# top-8; plan blocks of 16 rows) at decode token counts.
PAGE = dict(H=4096, I=1024, E=288, top_k=8, block_m=16, garbage_plan=True)


def test_w4a8_forward_page_shape_decode():
    prob = W4A8Problem(W.MoEConfig("w4a8_e288_m1", M=1, **PAGE))
    dq, ds = _run(prob)
    _check(prob, np.asarray([0]), dq, ds)


def test_w4a8_forward_page_shape_1024_tokens():
    """The page's timing shape at the token count the benchmark times, on a
    token set holding a route in every plan block."""
    prob = W4A8Problem(W.MoEConfig("w4a8_e288_m1024", M=1024, **PAGE))
    dq, ds = _run(prob)
    tokens = block_cover_tokens(prob)
    assert tokens.size >= 64
    _check(prob, tokens, dq, ds)


def test_w4a8_all_masked_leaves_out_unchanged():
    cfg = CASES["w4a8_tiny"].with_(name="w4a8_masked", masked_frac=1.0)
    prob = W4A8Problem(cfg)
    _run(prob, debug=False)
    assert int(prob.ntpp.item()) == 0
    assert torch.equal(prob.out, prob.out_prior)


def test_w4a8_bad_expert_is_reported_and_skipped():
    prob = W4A8Problem(CASES["w4a8_tiny"])
    prob.run_plan()
    P = int(prob.ntpp.item())
    assert P >= 16
    prob.expert_ids[0] = prob.cfg.E + 5                    # neither an expert nor -1
    prob.run_forward()
    torch.cuda.synchronize()
    assert int(prob.status.item()) & L.MOE_DEV_BAD_EXPERT
