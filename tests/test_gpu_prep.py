"""GPU parity of the integer / byte kernels: quantisers, interleave, UE8M0
requant and the routing plan, all bit-exact against the oracle."""

import numpy as np
import pytest
import torch

from fp8_block_scale_gb300 import _lib as L
import workloads as W
from oracle import moe as O
from oracle.numerics import bf16_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _load():
    L.load()


def _bf16(rng, shape, scale):
    return torch.from_numpy(bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))).to(torch.bfloat16)


@pytest.mark.parametrize("M,H", [(1, 128), (37, 384), (300, 7168)])
def test_quantize_act_bit_exact(M, H):
    rng = np.random.default_rng(M + H)
    x = _bf16(rng, (M, H), 1.0)
    x[M // 2, :128] = 0                                   # an all-zero group
    x[0, 5] = 1e-30                                       # a value far below the group's scale
    x[0, 6] = -1e-30
    q = torch.empty(M, H, dtype=torch.uint8, device="cuda")
    s = torch.empty(M, H // 128, dtype=torch.float32, device="cuda")
    L.moe_quantize_act_1x128(x.cuda(), q, s)
    rq, rs = O.quantize_act_1x128(x.float().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("M,H", [(1, 128), (37, 384), (300, 7168)])
def test_quantize_act_ue8m0_bit_exact(M, H):
    rng = np.random.default_rng(M * 3 + H)
    x = _bf16(rng, (M, H), 1.0)
    x[M // 2, :128] = 0                                   # an all-zero group
    x[0, 5] = 1e-30                                       # a value far below the group's scale
    x[-1, :128] = torch.from_numpy(bf16_round(rng.uniform(-13, 13, 128).astype(np.float32))).to(torch.bfloat16)
    x[-1, 3] = 14.0                                       # amax/448 = 2^-5: already a power of two
    q = torch.empty(M, H, dtype=torch.uint8, device="cuda")
    s = torch.empty(M, H // 128, dtype=torch.float32, device="cuda")
    L.moe_quantize_act_1x128_ue8m0(x.cuda(), q, s)
    rq, rs = O.quantize_act_1x128_ue8m0(x.float().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("E,R,C", [(1, 128, 128), (3, 256, 384), (2, 2048, 1024)])
def test_quantize_weight_bit_exact(E, R, C):
    rng = np.random.default_rng(E * R + C)
    w = _bf16(rng, (E, R, C), 0.02)
    w[0, :128, :128] = 0                                  # a zero block -> scale 0, codes 0
    q = torch.empty(E, R, C, dtype=torch.uint8, device="cuda")
    s = torch.empty(E, R // 128, C // 128, dtype=torch.float32, device="cuda")
    L.moe_quantize_weight_128x128(w.cuda(), q, s)
    rq, rs = O.quantize_weight_128x128(w.float().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("E,I,H", [(1, 128, 128), (5, 256, 384), (3, 1024, 4096)])
def test_prep_weights_interleave_bit_exact(E, I, H):
    g = torch.Generator().manual_seed(E * I + H)
    w = torch.randint(0, 256, (E, 2 * I, H), generator=g, dtype=torch.uint8)
    out = torch.empty_like(w, device="cuda")
    L.moe_prep_weights(w.cuda(), out)
    ref = O.interleave_gate_up(w.numpy())
    assert np.array_equal(out.cpu().numpy(), ref)


def test_requant_ue8m0_bit_exact():
    rng = np.random.default_rng(3)
    E, R, C = 3, 256, 384
    w = bf16_round((rng.standard_normal((E, R, C)) * 0.02).astype(np.float32))
    q, s = O.quantize_weight_128x128(w)
    s[0, 0, 0] = 0.0                                     # zero block: unchanged
    s[1, 1, 2] = np.float32(2.0 ** -9)                    # already a power of two: unchanged
    s[2, 0, 1] = np.float32(3e-39)                        # subnormal scale
    s[1, 0, 0] = np.float32(1.5e38)                       # rounds up to 2^127
    s[2, 1, 1] = np.float32(2.5e38)                       # no FP32 power of two above it: kept
    qd = torch.from_numpy(q).cuda()
    sd = torch.from_numpy(s).cuda()
    eb = torch.full(s.shape, 0xAB, dtype=torch.uint8, device="cuda")
    L.moe_requant_scales_ue8m0(qd, sd, eb)
    rq, rs, reb = O.requant_scales_ue8m0(q, s)
    torch.cuda.synchronize()
    assert np.array_equal(sd.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(qd.cpu().numpy(), rq)
    assert np.array_equal(eb.cpu().numpy(), reb)


# ------------------------------------------------------------------ plan

def _run_plan(ids_np, E, bm, id_dtype=torch.int32, garbage=True):
    M, k = ids_np.shape
    cap = -(-(M * k + E * (bm - 1)) // bm) * bm
    bcap = cap // bm
    ids = torch.from_numpy(ids_np).to(id_dtype).cuda()
    sorted_ids = W.garbage_int32(cap, 7, device="cuda") if garbage else torch.zeros(cap, dtype=torch.int32, device="cuda")
    expert_ids = W.garbage_int32(bcap, 8, device="cuda") if garbage else torch.zeros(bcap, dtype=torch.int32, device="cuda")
    s0, e0 = sorted_ids.clone(), expert_ids.clone()
    ntpp = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device="cuda")
    L.moe_plan(ids, E, bm, sorted_ids, expert_ids, ntpp, ws)
    torch.cuda.synchronize()
    return sorted_ids.cpu().numpy(), expert_ids.cpu().numpy(), int(ntpp.item()), s0.cpu().numpy(), e0.cpu().numpy()


def _check_plan(ids_np, E, bm, id_dtype=torch.int32):
    s, b, P, s0, e0 = _run_plan(ids_np, E, bm, id_dtype)
    rs, rb, rP = O.moe_plan(ids_np, E, bm)
    assert P == rP
    assert np.array_equal(s[:P], rs)
    assert np.array_equal(b[:P // bm], rb)
    # nothing past the extent is written
    assert np.array_equal(s[P:], s0[P:])
    assert np.array_equal(b[P // bm:], e0[P // bm:])


@pytest.mark.parametrize("name", ["tiny", "decode_m1", "decode_m8", "decode_m64", "prefill_1024", "prefill_8192",
                                  "skewed", "large"])
def test_plan_bit_exact_configs(name):
    cfg = W.CONFIGS[name]
    r = W.make_routing(cfg)
    _check_plan(r.topk_ids.to(torch.int64).numpy(), cfg.E, cfg.block_m, cfg.id_dtype)


@pytest.mark.parametrize("case", ["all_masked", "out_of_range", "one_expert", "bm8", "bm1024", "int64", "hot",
                                  "r1024", "r1025", "e1024", "e1025", "e2048"])
def test_plan_bit_exact_edges(case):
    rng = np.random.default_rng(11)
    E, bm, dt = 64, 64, torch.int32
    if case == "all_masked":
        ids = -np.ones((7, 3), dtype=np.int64)
    elif case == "out_of_range":
        ids = rng.integers(-9, E + 9, size=(50, 4))
    elif case == "one_expert":
        E = 1
        ids = np.zeros((33, 1), dtype=np.int64)
    elif case == "bm8":
        bm = 8
        ids = rng.integers(0, E, size=(100, 6))
    elif case == "bm1024":
        bm = 1024
        ids = rng.integers(0, 4, size=(700, 2))
        E = 4
    elif case == "int64":
        dt = torch.int64
        ids = rng.integers(-1, E, size=(123, 5))
    elif case == "r1024":  # the largest plan the single-CTA path takes
        ids = rng.integers(-1, E, size=(256, 4))
    elif case == "r1025":  # one route more: the three-launch path
        ids = rng.integers(-1, E, size=(205, 5))
    elif case in ("e1024", "e1025", "e2048"):  # expert counts around the single-CTA limit, and the maximum
        E = int(case[1:])
        ids = rng.integers(-1, E, size=(90, 7))
    else:  # one expert takes most routes, spanning many blocks and chunks
        ids = np.where(rng.random((3000, 4)) < 0.7, 3, rng.integers(0, E, size=(3000, 4)))
    _check_plan(ids, E, bm, dt)


def test_plan_is_deterministic():
    cfg = W.CONFIGS["prefill_2048"]
    ids = W.make_routing(cfg).topk_ids.numpy()
    a = _run_plan(ids, cfg.E, cfg.block_m)
    b = _run_plan(ids, cfg.E, cfg.block_m)
    assert a[2] == b[2] and np.array_equal(a[0][:a[2]], b[0][:b[2]])
