"""Pins for the oracle's plan, weight prep, quantisers and forward (CPU only).

Nothing here compares the oracle with itself: each check is a closed form, an
invariant, an independent brute force, or a special case that reduces to a
torch/numpy routine.
"""

import itertools
import os

import numpy as np
import pytest
import torch

from oracle import moe
from oracle.numerics import bf16_round, e4m3_decode, e4m3_encode, f32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- plan

def _plan_by_stable_sort(ids, E, bm):
    """Independent formulation: stable argsort by expert, then pad segments."""
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    R = flat.size
    valid = np.nonzero((flat >= 0) & (flat < E))[0]
    order = valid[np.argsort(flat[valid], kind="stable")]
    out, blocks = [], []
    i = 0
    while i < order.size:
        e = flat[order[i]]
        j = i
        while j < order.size and flat[order[j]] == e:
            j += 1
        seg = list(order[i:j])
        pad = (-len(seg)) % bm
        out += seg + [R] * pad
        blocks += [e] * ((len(seg) + pad) // bm)
        i = j
    return np.asarray(out, dtype=np.int32), np.asarray(blocks, dtype=np.int32)


def _check_plan_invariants(ids, E, bm, s, b, P):
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    R = flat.size
    assert P == s.size == b.size * bm
    counts = np.bincount(flat[(flat >= 0) & (flat < E)], minlength=E)
    assert P == int(sum(-(-c // bm) * bm for c in counts))
    seen = np.zeros(R, dtype=int)
    for blk in range(b.size):
        e = b[blk]
        seg = s[blk * bm:(blk + 1) * bm]
        real = seg[seg < R]
        assert (flat[real] == e).all()
        seen[real] += 1
    valid = (flat >= 0) & (flat < E)
    assert (seen[valid] == 1).all() and (seen[~valid] == 0).all()
    # ascending route order inside each expert, sentinels only at segment tails
    for e in np.unique(b):
        seg = s[np.repeat(b == e, bm)]
        real = seg[seg < R]
        assert (np.diff(real) > 0).all()
        assert (seg[: real.size] == real).all() and (seg[real.size:] == R).all()
    assert (np.diff(b) >= 0).all()


def test_plan_brute_force_all_tiny_routings():
    """Every routing of M=2 tokens, k=2, over ids {-1, 0, 1, 2}, block_m 2 and 4."""
    E = 3
    for combo in itertools.product([-1, 0, 1, 2], repeat=4):
        ids = np.asarray(combo).reshape(2, 2)
        for bm in (2, 4):
            s, b, P = moe.moe_plan(ids, E, bm)
            _check_plan_invariants(ids, E, bm, s, b, P)
            s2, b2 = _plan_by_stable_sort(ids, E, bm)
            assert np.array_equal(s, s2) and np.array_equal(b, b2)
            cap, bcap = moe.plan_capacity(2, 2, E, bm)
            assert P <= cap and bcap * bm == cap


@pytest.mark.parametrize("M,k,E,bm", [(16, 2, 8, 64), (37, 9, 257, 64), (64, 10, 512, 128), (5, 3, 4, 8)])
def test_plan_random_against_stable_sort(M, k, E, bm):
    rng = np.random.default_rng(M * 1000 + E)
    ids = rng.integers(-1, E + 2, size=(M, k))
    s, b, P = moe.moe_plan(ids, E, bm)
    _check_plan_invariants(ids, E, bm, s, b, P)
    s2, b2 = _plan_by_stable_sort(ids, E, bm)
    assert np.array_equal(s, s2) and np.array_equal(b, b2)
    cap, _ = moe.plan_capacity(M, k, E, bm)
    assert P <= cap


def test_plan_capacity_is_tight():
    # one route per expert: every expert pads to a full block
    M, k, E, bm = 4, 2, 8, 64
    ids = np.arange(8).reshape(4, 2)
    _, _, P = moe.moe_plan(ids, E, bm)
    assert P == moe.plan_capacity(M, k, E, bm)[0] == 8 * 64
    # more experts than routes: at most R experts are non-empty, so the bound
    # is R * block_m (a decode step, 9 routes over 257 experts), and a step
    # whose routes all go to different experts attains it
    assert moe.plan_capacity(1, 9, 257, 64) == (9 * 64, 9)
    _, b, P = moe.moe_plan(np.arange(0, 257, 29)[None, :9], 257, 64)
    assert P == 9 * 64 and b.size == 9


def test_plan_all_masked_is_empty():
    s, b, P = moe.moe_plan(-np.ones((3, 2), dtype=np.int64), 4, 8)
    assert P == 0 and s.size == 0 and b.size == 0


# ---------------------------------------------------------------- interleave

def test_interleave_matches_golden_map():
    rows = [tuple(map(int, l.split())) for l in open(os.path.join(GOLDEN, "interleave_i16.txt"))
            if l.strip() and not l.startswith("#")]
    w = np.arange(32, dtype=np.uint8).reshape(1, 32, 1).repeat(3, axis=2)
    out = moe.interleave_gate_up(w)
    for o, logical in rows:
        assert (out[0, o] == logical).all()


def test_interleave_is_a_bijection_with_inverse():
    rng = np.random.default_rng(5)
    E, I, H = 3, 256, 128
    w = rng.integers(0, 256, size=(E, 2 * I, H), dtype=np.uint8)
    out = moe.interleave_gate_up(w)
    # inverse: de-interleave
    back = np.empty_like(out)
    for q in range(I // 8):
        back[:, 8 * q:8 * q + 8] = out[:, 16 * q:16 * q + 8]
        back[:, I + 8 * q:I + 8 * q + 8] = out[:, 16 * q + 8:16 * q + 16]
    assert np.array_equal(back, w)
    assert not np.array_equal(out, w)


# ---------------------------------------------------------------- quantisers

def test_quantize_act_properties():
    rng = np.random.default_rng(6)
    x = bf16_round(rng.standard_normal((9, 384)).astype(np.float32))
    x[3, 128:256] = 0.0                                # an all-zero group
    x[5, 0:128] = -0.0                                 # and one of negative zeros
    q, s = moe.quantize_act_1x128(x)
    assert q.shape == x.shape and s.shape == (9, 3)
    assert s[3, 1] == 0 and (q[3, 128:256] == 0).all()
    assert s[5, 0] == 0 and (q[5, 0:128] == 0).all()  # scale 0 gives code 0x00, not -0 (0x80)
    deq = e4m3_decode(q) * np.repeat(s.astype(np.float64), 128, axis=1)
    for m in range(9):
        for g in range(3):
            grp = x[m, 128 * g:128 * (g + 1)].astype(np.float64)
            amax = np.abs(grp).max()
            if amax == 0:
                continue
            assert s[m, g] == np.float32(np.float32(amax) / np.float32(448))
            # the amax element lands on the top code
            i = np.argmax(np.abs(grp))
            assert abs(e4m3_decode(q[m:m + 1, 128 * g + i])[0]) == 448.0
            # error at most half an E4M3 spacing (relative 2^-4) plus FP32 slack
            err = np.abs(deq[m, 128 * g:128 * (g + 1)] - grp)
            bound = np.maximum(np.abs(grp) * 2.0 ** -4, 2.0 ** -10 * s[m, g]) * (1 + 1e-6)
            assert (err <= bound + 1e-30).all()


def test_quantize_act_ue8m0_properties():
    """Power-of-two scales: each group's scale is the smallest power of two
    not below amax/448, so the group's largest code lands in [224, 448], the
    reconstruction error is at most half an E4M3 spacing, and a group whose
    amax/448 already is a power of two quantises exactly as with the plain
    amax/448 scale."""
    rng = np.random.default_rng(16)
    x = bf16_round(rng.standard_normal((7, 512)).astype(np.float32))
    x[2, 128:256] = 0.0                                 # an all-zero group
    x[4, :128] = bf16_round(rng.uniform(-13.0, 13.0, 128).astype(np.float32))
    x[4, 17] = 14.0                                     # amax/448 = 2^-5 exactly
    q, s = moe.quantize_act_1x128_ue8m0(x)
    assert q.shape == x.shape and s.shape == (7, 4)
    assert s[2, 1] == 0 and (q[2, 128:256] == 0).all()
    q0, s0 = moe.quantize_act_1x128(x)
    assert s[4, 0] == np.float32(2.0 ** -5) and s0[4, 0] == s[4, 0]
    assert np.array_equal(q[4, :128], q0[4, :128])
    for m in range(7):
        for g in range(4):
            grp = x[m, 128 * g:128 * (g + 1)].astype(np.float64)
            amax = np.abs(grp).max()
            if amax == 0:
                continue
            sg = float(s[m, g])
            frac, _ = np.frexp(sg)
            assert frac == 0.5                                          # a power of two
            base = float(np.float32(np.float32(amax) / np.float32(448)))
            assert base <= sg < 2 * base or sg == base
            top = np.abs(e4m3_decode(q[m, 128 * g:128 * (g + 1)])).max()
            assert 224.0 <= top <= 448.0
            deq = e4m3_decode(q[m, 128 * g:128 * (g + 1)]) * sg
            err = np.abs(deq - grp)
            bound = np.maximum(np.abs(grp) * 2.0 ** -4, 2.0 ** -10 * sg) * (1 + 1e-6)
            assert (err <= bound + 1e-30).all()


def test_quantize_weight_blocks_match_act_quantiser_on_blocks():
    """A 128x128 block quantises like one group of 16384 values."""
    rng = np.random.default_rng(7)
    w = bf16_round((rng.standard_normal((2, 256, 384)) * 0.02).astype(np.float32))
    q, s = moe.quantize_weight_128x128(w)
    assert s.shape == (2, 2, 3)
    for e in range(2):
        for rb in range(2):
            for cb in range(3):
                blk = w[e, 128 * rb:128 * (rb + 1), 128 * cb:128 * (cb + 1)]
                amax = np.abs(blk).max()
                sc = np.float32(np.float32(amax) / np.float32(448))
                assert s[e, rb, cb] == sc
                want = e4m3_encode(f32(blk / sc))
                assert np.array_equal(q[e, 128 * rb:128 * (rb + 1), 128 * cb:128 * (cb + 1)], want)


# ---------------------------------------------------------------- UE8M0

def test_ue8m0_round_up_closed_form():
    rng = np.random.default_rng(8)
    s = np.concatenate([(rng.random(20000) * 1e-2).astype(np.float32),
                        np.float32(2.0) ** np.arange(-30, 10, dtype=np.float32),
                        np.array([1e-38, 3e-39, 1.5, 0.75], dtype=np.float32)])
    s = s[s > 0]
    p = moe.ue8m0_round_up(s).astype(np.float64)
    m, _ = np.frexp(p)
    assert (m == 0.5).all()                          # powers of two
    assert (p >= s).all() and (p < 2.0 * s).all()     # rounded up, within a factor 2
    assert np.array_equal(moe.ue8m0_round_up(p.astype(np.float32)).astype(np.float64), p)  # idempotent
    pw = np.float32(2.0) ** np.arange(-20, 20, dtype=np.float32)
    assert np.array_equal(moe.ue8m0_round_up(pw), pw)


def test_ue8m0_requant_properties():
    rng = np.random.default_rng(9)
    w = bf16_round((rng.standard_normal((2, 256, 256)) * 0.02).astype(np.float32))
    q, s = moe.quantize_weight_128x128(w)
    s[1, 0, 1] = 0.0                                  # a zero-scale block stays as it is
    q2, s2, eb = moe.requant_scales_ue8m0(q, s)
    assert np.array_equal(q2[1, :128, 128:], q[1, :128, 128:]) and s2[1, 0, 1] == 0 and eb[1, 0, 1] == 0
    pos = s > 0
    assert np.array_equal(np.exp2(eb[pos].astype(np.float64) - 127), s2[pos].astype(np.float64))
    # per element: new value = nearest E4M3 to decode(w)*s/s' (brute force), scaled by s'
    vals = np.unique(np.abs(e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))
    for e in range(2):
        for rb in range(2):
            for cb in range(2):
                if s[e, rb, cb] == 0:
                    continue
                sl = (e, slice(128 * rb, 128 * (rb + 1)), slice(128 * cb, 128 * (cb + 1)))
                target = e4m3_decode(q[sl]) * (float(s[e, rb, cb]) / float(s2[e, rb, cb]))
                got = e4m3_decode(q2[sl])
                # |got - target| is at most the distance to the nearest grid value
                d_best = np.min(np.abs(np.abs(target)[..., None] - vals[None, None, :]), axis=-1)
                assert (np.abs(got - target) <= d_best * (1 + 1e-6) + 1e-12).all()
    # already power-of-two scales: nothing changes
    q3, s3, _ = moe.requant_scales_ue8m0(q2, s2)
    assert np.array_equal(q3, q2) and np.array_equal(s3, s2)


# ---------------------------------------------------------------- forward

def _tiny_problem(seed, M=3, H=256, I=128, E=3, k=2, masked=()):
    rng = np.random.default_rng(seed)
    x = bf16_round(rng.standard_normal((M, H)).astype(np.float32))
    aq, as_ = moe.quantize_act_1x128(x)
    w13 = bf16_round((rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32))
    w2 = bf16_round((rng.standard_normal((E, H, I)) * 0.02).astype(np.float32))
    w13q, w13s = moe.quantize_weight_128x128(w13)
    w2q, w2s = moe.quantize_weight_128x128(w2)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int64)
    for (t, j) in masked:
        ids[t, j] = -1
    tw = rng.random((M, k)).astype(np.float32)
    prior = bf16_round((rng.standard_normal((M, H)) * 0.1).astype(np.float32))
    return dict(a_q=aq, a_s=as_, w13_q=w13q, w13_s=w13s, w2_q=w2q, w2_s=w2s,
                topk_ids=ids, topk_w=tw, out_prior=prior)


def _near_tie(ratio):
    """True where a float64 value lies within 1e-5 (relative) of an E4M3 rounding midpoint."""
    a = np.abs(ratio)
    vals = np.unique(np.abs(e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = (vals[1:] + vals[:-1]) / 2
    d = np.min(np.abs(a[..., None] - mids[None, :]), axis=-1)
    return d <= 1e-5 * np.maximum(a, 2.0 ** -9)


@pytest.mark.parametrize("seed,shape", [(10, dict(M=3, H=256, I=128, E=3, k=2)),
                                        (11, dict(M=2, H=128, I=256, E=4, k=3)),
                                        (12, dict(M=4, H=256, I=256, E=2, k=1))])
def test_forward_matches_fp64_brute_force(seed, shape):
    p = _tiny_problem(seed, **shape)
    out32, inter = moe.moe_forward(**p, routed_scale=2.5, return_inter=True, round_bf16=False)
    out64, inter64 = moe.moe_forward_fp64(**p, routed_scale=2.5)
    # intermediate codes identical except where the exact value is a near-tie
    n_diff = 0
    for key, (codes, scales) in inter.items():
        c64, s64, ratio = inter64[key]
        diff = codes != c64
        assert (~diff | _near_tie(ratio)).all()
        n_diff += int(diff.sum())
        np.testing.assert_allclose(scales, s64, rtol=1e-6)
    assert n_diff <= 2
    # outputs agree to FP32 accuracy (before the BF16 rounding)
    rel = np.linalg.norm(out32 - out64) / np.linalg.norm(out64 - p["out_prior"])
    assert rel < 1e-5, rel


def test_forward_special_case_reduces_to_matmul_and_silu():
    """All scales 1, k = 1, route weight 1: GEMM1 is a plain matmul of the
    decoded values, SwiGLU is torch's silu(gate) * up."""
    rng = np.random.default_rng(13)
    M, H, I, E = 5, 384, 256, 2
    aq = e4m3_encode((rng.standard_normal((M, H)) * 2).astype(np.float32))
    w13q = e4m3_encode((rng.standard_normal((E, 2 * I, H)) * 0.5).astype(np.float32))
    ones_a = np.ones((M, H // 128), dtype=np.float32)
    ones_w = np.ones((2 * I // 128, H // 128), dtype=np.float32)
    for e in range(E):
        acc = moe.gemm1_expert(aq, ones_a, w13q[e], ones_w)
        ref = torch.from_numpy(e4m3_decode(aq)) @ torch.from_numpy(e4m3_decode(w13q[e])).T
        np.testing.assert_allclose(acc, ref.numpy(), rtol=2e-6, atol=1e-4)
        h = moe.swiglu(acc, I)
        g = torch.from_numpy(acc[:, :I].astype(np.float64))
        u = torch.from_numpy(acc[:, I:].astype(np.float64))
        ref_h = torch.nn.functional.silu(g) * u
        np.testing.assert_allclose(h, ref_h.numpy(), rtol=1e-6, atol=1e-6)
    # GEMM2 the same way: y = decode(q) @ decode(W2)^T
    qi = e4m3_encode(rng.standard_normal((M, I)).astype(np.float32))
    w2q = e4m3_encode((rng.standard_normal((H, I)) * 0.5).astype(np.float32))
    y = moe.gemm2_expert(qi, np.ones((M, I // 128), np.float32), w2q, np.ones((H // 128, I // 128), np.float32))
    ref = torch.from_numpy(e4m3_decode(qi)) @ torch.from_numpy(e4m3_decode(w2q)).T
    np.testing.assert_allclose(y, ref.numpy(), rtol=2e-6, atol=1e-4)


def test_forward_block_scales_index_rows_and_columns():
    """Scaling one weight block by 2 (codes unchanged) doubles exactly the
    slices that block covers: catches transposed or mis-indexed scale blocks."""
    rng = np.random.default_rng(14)
    M, H, I = 2, 256, 256
    aq = e4m3_encode(rng.standard_normal((M, H)).astype(np.float32))
    a_s = np.ones((M, 2), np.float32)
    w13q = e4m3_encode((rng.standard_normal((2 * I, H)) * 0.5).astype(np.float32))
    ws = np.ones((4, 2), np.float32)
    base = moe.gemm1_expert(aq, a_s, w13q, ws)
    ws2 = ws.copy()
    ws2[2, 1] = 2.0                              # rows 256..383, K slice 1
    got = moe.gemm1_expert(aq, a_s, w13q, ws2)
    dots = moe.slice_dots(aq, w13q)
    want = base.copy()
    want[:, 256:384] = f32(f32(dots[:, 256:384, 0]) + f32(dots[:, 256:384, 1] * np.float32(2)))
    np.testing.assert_array_equal(got, want)
    # activation scale of token 1, slice 0
    a_s2 = a_s.copy()
    a_s2[1, 0] = 4.0
    got = moe.gemm1_expert(aq, a_s2, w13q, ws)
    want = base.copy()
    want[1] = f32(f32(dots[1, :, 0] * np.float32(4)) + dots[1, :, 1])
    np.testing.assert_array_equal(got, want)


def test_forward_zero_weight_scales_contribute_nothing():
    p = _tiny_problem(15, M=4, E=3, k=2)
    p["w13_s"][1] = 0
    p["w2_s"][1] = 0
    out = moe.moe_forward(**p)
    ids = p["topk_ids"].copy()
    ids[ids == 1] = -1
    out_masked = moe.moe_forward(**dict(p, topk_ids=ids))
    assert np.array_equal(out, out_masked)


def test_forward_all_masked_leaves_out_unchanged():
    p = _tiny_problem(16, M=3, k=2)
    p["topk_ids"][:] = -1
    out = moe.moe_forward(**p)
    assert np.array_equal(out.view(np.uint32), p["out_prior"].view(np.uint32))


def test_forward_accumulates_onto_prior():
    p = _tiny_problem(17, M=3, E=3, k=1)
    zero = np.zeros_like(p["out_prior"])
    r0 = moe.moe_forward(**dict(p, out_prior=zero), round_bf16=False)
    rp = moe.moe_forward(**p, round_bf16=False)
    assert np.array_equal(rp, f32(p["out_prior"] + r0))       # k = 1: one FP32 add
    assert np.array_equal(moe.moe_forward(**p), bf16_round(f32(p["out_prior"] + r0)))


def test_forward_token_permutation_equivariance():
    p = _tiny_problem(18, M=4, E=3, k=2)
    perm = np.array([2, 0, 3, 1])
    q = dict(p)
    for key in ("a_q", "a_s", "topk_ids", "topk_w", "out_prior"):
        q[key] = p[key][perm]
    assert np.array_equal(moe.moe_forward(**q), moe.moe_forward(**p)[perm])


def test_forward_split_route_with_halved_weight():
    p = _tiny_problem(19, M=3, E=3, k=1)
    q = dict(p)
    q["topk_ids"] = np.repeat(p["topk_ids"], 2, axis=1)
    q["topk_w"] = np.repeat(p["topk_w"] / np.float32(2), 2, axis=1).astype(np.float32)
    a = moe.moe_forward(**p, round_bf16=False)
    b = moe.moe_forward(**q, round_bf16=False)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-7)


def test_forward_routed_scale_equals_scaled_weights():
    p = _tiny_problem(20, M=3, E=3, k=2)
    a = moe.moe_forward(**p, routed_scale=2.5)
    b = moe.moe_forward(**dict(p, topk_w=f32(p["topk_w"] * np.float32(2.5))), routed_scale=1.0)
    assert np.array_equal(a, b)


def test_forward_token_subset_equals_full_rows():
    p = _tiny_problem(21, M=5, E=3, k=2)
    full = moe.moe_forward(**p)
    sub = moe.moe_forward(**p, tokens=[4, 1])
    assert np.array_equal(sub, full[[4, 1]])


def test_forward_expert_partitioned_is_bit_identical():
    """Experts computed in several threads, combined in the same fixed order,
    give exactly the single-threaded output and intermediate."""
    p = _tiny_problem(22, M=6, E=5, k=3, masked=((1, 2),))
    a, ia = moe.moe_forward(**p, return_inter=True)
    b, ib = moe.moe_forward(**p, return_inter=True, workers=3)
    assert np.array_equal(a, b)
    assert ia.keys() == ib.keys()
    for key in ia:
        assert np.array_equal(ia[key][0], ib[key][0]) and np.array_equal(ia[key][1], ib[key][1])


def _route_contributions(p):
    """c[j] [M, H]: route j's weighted down projection alone (other routes
    masked, zero prior; with one route the FP32 accumulator is c_j exactly)."""
    k = p["topk_ids"].shape[1]
    zero = np.zeros_like(p["out_prior"])
    out = []
    for j in range(k):
        ids = np.full_like(p["topk_ids"], -1)
        ids[:, j] = p["topk_ids"][:, j]
        out.append(moe.moe_forward(**dict(p, topk_ids=ids, out_prior=zero), round_bf16=False).astype(np.float64))
    return out


def test_forward_combine_modes():
    """The three ways route contributions reach `out` agree exactly for one
    route onto a zero prior (a single rounding each way), and otherwise stay
    within the bounds their extra BF16 roundings allow: half a BF16 ulp
    (2^-8 relative: 7 stored mantissa bits) per rounded contribution for
    per-route rounding, and per step of the running sum for the stepwise
    reduce-add."""
    one = _tiny_problem(23, M=3, E=3, k=1)
    one["out_prior"] = np.zeros_like(one["out_prior"])
    ref = moe.moe_forward(**one)
    for mode in ("bf16_route", "bf16_stepwise"):
        assert np.array_equal(moe.moe_forward(**one, combine=mode), ref)

    p = _tiny_problem(24, M=4, E=4, k=3)
    c = _route_contributions(p)
    prior = p["out_prior"].astype(np.float64)
    acc = moe.moe_forward(**p, round_bf16=False).astype(np.float64)
    slack = 1e-5 * (np.abs(prior) + sum(np.abs(cj) for cj in c)) + 1e-30
    # per-route rounding: every contribution moves by at most 2^-8 of itself
    route = moe.moe_forward(**p, combine="bf16_route", round_bf16=False).astype(np.float64)
    assert (np.abs(route - acc) <= 2.0 ** -8 * sum(np.abs(cj) for cj in c) + slack).all()
    assert not np.array_equal(route, acc)                 # the per-route rounding shows somewhere
    # and it decomposes into the single-route runs: each contribution rounded
    # to BF16 on its own, then added in slot order in FP32 onto the prior
    s = p["out_prior"].astype(np.float32)
    for cj in c:
        s = f32(s + bf16_round(f32(cj)))
    assert np.array_equal(route, s.astype(np.float64))
    # stepwise: the prior and each running sum are rounded once more
    step = moe.moe_forward(**p, combine="bf16_stepwise").astype(np.float64)
    running = [np.abs(prior)]
    s = prior.copy()
    for cj in c:
        s = s + cj
        running.append(np.abs(s))
    bound = 2.0 ** -8 * sum(running) * (1 + 2.0 ** -7) + slack
    assert (np.abs(step - acc) <= bound).all()
    # and the modes do differ somewhere on this problem
    assert not np.array_equal(moe.moe_forward(**p, combine="bf16_stepwise"), moe.moe_forward(**p))
