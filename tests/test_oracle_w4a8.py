"""Pins for the E2M1-K32 x FP8 oracle (CPU only).

As for the block-FP8 oracle, nothing here compares the oracle with itself:
the codec against the format's value table and a brute-force nearest-value
search, the dot products against integer arithmetic, the quantisers and the
GEMM against invariants and special cases that reduce to torch routines, the
forward against an independently written float64 twin and against the
block-FP8 oracle where the two formats describe the same numbers.
"""

import numpy as np
import pytest
import torch

from oracle import w4a8
from oracle.numerics import bf16_round, e4m3_decode, e4m3_encode, f32

# The sixteen E2M1 values of the OCP Microscaling Formats (MX) specification,
# FP4 element type, by code (sign bit 3): written out by hand, not computed.
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
              -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


# ---------------------------------------------------------------- codec

def test_e2m1_decode_matches_format_table():
    v = w4a8.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(v, np.array(E2M1_TABLE))
    assert np.signbit(v[8]) and not np.signbit(v[0])


def test_e2m1_round_trip_every_code():
    codes = np.arange(16, dtype=np.uint8)
    np.testing.assert_array_equal(w4a8.e2m1_encode(w4a8.e2m1_decode(codes)), codes)


def _nearest_by_search(x):
    """Brute force: the code whose value is nearest to x; on a tie the code
    with the even mantissa bit; beyond 6 the largest magnitude."""
    best = None
    for c in range(16):
        v = E2M1_TABLE[c]
        if (c >> 3) != int(np.signbit(x)):
            continue                       # the sign of x is kept, zero included
        d = abs(min(abs(x), 6.0) - abs(v))
        key = (d, c & 1)                   # smaller distance, then even mantissa
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e2m1_encode_brute_force_dense_grid():
    # every multiple of 1/64 in [-8, 8] (all midpoints and ties included), the
    # signed zeros, infinities and a sprinkle of random values
    grid = np.concatenate([np.arange(-512, 513) / 64.0, [0.0, -0.0, np.inf, -np.inf, 1e30, -1e-30],
                           np.random.default_rng(1).standard_normal(2000) * 3])
    got = w4a8.e2m1_encode(grid)
    want = np.array([_nearest_by_search(float(x)) for x in grid], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e2m1_encode_ties_go_to_even_mantissa():
    # the midpoints between neighbouring magnitudes, by hand
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for x, v in ties.items():
        assert w4a8.e2m1_decode(w4a8.e2m1_encode(x)) == v, x
        assert w4a8.e2m1_decode(w4a8.e2m1_encode(-x)) == -v, x


def test_pack_hand_worked_example_and_round_trip():
    # codes 1, 2, 15, 8 -> bytes 0x21 (2 high, 1 low) and 0x8F (8 high, 15 low)
    np.testing.assert_array_equal(w4a8.pack_e2m1(np.array([1, 2, 15, 8], np.uint8)),
                                  np.array([0x21, 0x8F], np.uint8))
    c = np.random.default_rng(2).integers(0, 16, size=(3, 5, 64)).astype(np.uint8)
    np.testing.assert_array_equal(w4a8.unpack_e2m1(w4a8.pack_e2m1(c)), c)
    every_byte = np.arange(256, dtype=np.uint8)[:, None]
    np.testing.assert_array_equal(w4a8.pack_e2m1(w4a8.unpack_e2m1(every_byte)), every_byte)


# ---------------------------------------------------------------- quantisers

def _half_gap(mag):
    """Half the E2M1 spacing around a magnitude in [0, 6]."""
    return np.where(mag <= 2.0, 0.25, np.where(mag <= 4.0, 0.5, 1.0))


def test_quantize_weight_k32_properties():
    rng = np.random.default_rng(3)
    w = bf16_round((rng.standard_normal((2, 5, 128)) * 0.05).astype(np.float32))
    w[0, 1, 32:64] = 0.0                                    # one all-zero block
    w[0, 2, 0:32] = -0.0                                    # one block of negative zeros
    w[1, 2, 96:128] *= 1000.0                               # one block far larger than the rest
    codes, scale = w4a8.quantize_weight_k32(w)
    assert scale[0, 2, 0] == 0 and not codes[0, 2, 0:32].any()   # code 0, not -0 (8)
    assert codes.shape == w.shape and scale.shape == (2, 5, 4) and scale.dtype == np.float32
    assert scale[0, 1, 1] == 0 and not codes[0, 1, 32:64].any()
    g = w.reshape(2, 5, 4, 32)
    cg = codes.reshape(2, 5, 4, 32)
    live = scale > 0
    # the block's largest element takes the largest code, with its sign
    idx = np.argmax(np.abs(g), axis=-1)
    top = np.take_along_axis(cg, idx[..., None], axis=-1)[..., 0]
    top_sign = np.signbit(np.take_along_axis(g, idx[..., None], axis=-1)[..., 0])
    assert (np.where(live, (top & 7) == 7, True)).all()
    assert (np.where(live, (top >> 3) == top_sign, True)).all()
    # every element within half a step of its value (in units of its scale)
    deq = w4a8.dequantize_weight_k32(codes, scale).reshape(g.shape)
    s = scale.astype(np.float64)[..., None]
    err = np.abs(g - deq)
    bound = _half_gap(np.minimum(np.abs(g) / np.where(s > 0, s, 1.0), 6.0)) * s * (1 + 1e-6)
    assert (err <= bound).all()
    # scales are per row and per 32 columns: changing one block moves only its own scale
    w2 = w.copy()
    w2[1, 3, 40] = 7.0
    _, scale2 = w4a8.quantize_weight_k32(w2)
    changed = scale2 != scale
    assert changed[1, 3, 1] and changed.sum() == 1


def test_quantize_act_per_row_properties():
    rng = np.random.default_rng(4)
    x = bf16_round(rng.standard_normal((6, 256)).astype(np.float32) * np.array([1, 1e-3, 1e3, 1, 1, 1])[:, None])
    x[4] = 0.0
    x[5] = -0.0
    codes, scale = w4a8.quantize_act_per_row(x)
    assert scale.shape == (6,) and scale[4] == 0 and not codes[4].any()
    assert scale[5] == 0 and not codes[5].any()             # code 0x00, not -0 (0x80)
    for t in (0, 1, 2, 3):
        i = int(np.argmax(np.abs(x[t])))
        assert codes[t, i] & 0x7F == 0x7E                  # 448, the largest finite E4M3 magnitude
        assert (codes[t, i] >> 7) == int(np.signbit(x[t, i]))
        deq = e4m3_decode(codes[t]) * float(scale[t])
        # E4M3 keeps 3 mantissa bits: relative error at most 2**-4 above the subnormal range
        big = np.abs(x[t]) >= 2.0 ** -6 * scale[t]
        assert (np.abs(deq - x[t])[big] <= 2.0 ** -4 * np.abs(x[t])[big] * (1 + 1e-6)).all()
    # rows are independent
    c2, s2 = w4a8.quantize_act_per_row(x[[3, 0]])
    np.testing.assert_array_equal(c2, codes[[3, 0]])
    np.testing.assert_array_equal(s2, scale[[3, 0]])


# ---------------------------------------------------------------- GEMM

def test_k32_dots_equal_integer_arithmetic():
    """E4M3 values x 2**9 and E2M1 values x 2 are integers: the block dots are
    integer sums (Python ints, no rounding) times 2**-10, then one FP32 rounding."""
    rng = np.random.default_rng(5)
    xq = rng.integers(0, 256, size=(3, 96)).astype(np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x00                          # no NaN codes
    xq[0, :32] = 0x7E                                       # a block of +448s
    wq = rng.integers(0, 16, size=(4, 96)).astype(np.uint8)
    wq[1, :32] = 7                                          # against a block of +6s
    xi = [[int(round(v * 512)) for v in row] for row in e4m3_decode(xq)]
    wi = [[int(round(v * 2)) for v in row] for row in w4a8.e2m1_decode(wq)]
    got = w4a8.k32_dots(xq, wq)
    for i in range(3):
        for j in range(4):
            for kb in range(3):
                total = sum(xi[i][c] * wi[j][c] for c in range(32 * kb, 32 * kb + 32))
                assert got[i, j, kb] == np.float32(total / 1024.0), (i, j, kb)
    assert got[0, 1, 0] == 448 * 6 * 32


def test_gemm_special_case_reduces_to_matmul():
    """All scales 1: the projection is a plain matmul of the decoded values
    (to FP32 accuracy over K/32 block additions)."""
    rng = np.random.default_rng(6)
    xq = e4m3_encode((rng.standard_normal((5, 256)) * 2).astype(np.float32))
    wq = w4a8.e2m1_encode(rng.standard_normal((64, 256)) * 2)
    y = w4a8.gemm_w4a8(xq, np.ones(5, np.float32), wq, np.ones((64, 8), np.float32))
    ref = torch.from_numpy(e4m3_decode(xq)) @ torch.from_numpy(w4a8.e2m1_decode(wq)).T
    np.testing.assert_allclose(y, ref.numpy(), rtol=2e-6, atol=1e-4)


def test_gemm_scales_index_blocks_and_rows():
    rng = np.random.default_rng(7)
    xq = e4m3_encode(rng.standard_normal((4, 128)).astype(np.float32))
    xs = (rng.random(4) + 0.5).astype(np.float32)
    wq = w4a8.e2m1_encode(rng.standard_normal((8, 128)) * 2)
    ws = (rng.random((8, 4)) + 0.5).astype(np.float32)
    y = w4a8.gemm_w4a8(xq, xs, wq, ws)
    # doubling one row's activation scale doubles exactly that row
    xs2 = xs.copy()
    xs2[2] *= 2
    y2 = w4a8.gemm_w4a8(xq, xs2, wq, ws)
    np.testing.assert_array_equal(y2[2], 2 * y[2])
    np.testing.assert_array_equal(np.delete(y2, 2, 0), np.delete(y, 2, 0))
    # doubling one weight block scale adds that block's contribution to that column only
    ws2 = ws.copy()
    ws2[5, 1] *= 2
    y3 = w4a8.gemm_w4a8(xq, xs, wq, ws2)
    np.testing.assert_array_equal(np.delete(y3, 5, 1), np.delete(y, 5, 1))
    blk = e4m3_decode(xq)[:, 32:64] @ w4a8.e2m1_decode(wq)[5, 32:64]
    np.testing.assert_allclose(y3[:, 5] - y[:, 5], blk * float(ws[5, 1]) * xs.astype(np.float64),
                               rtol=1e-5, atol=1e-5 * np.abs(y[:, 5]).max())
    # a zero weight scale removes its block
    ws3 = ws.copy()
    ws3[:, 3] = 0
    y4 = w4a8.gemm_w4a8(xq, xs, wq, ws3)
    ref = (e4m3_decode(xq)[:, :96] * xs[:, None].astype(np.float64)) @ \
          (w4a8.e2m1_decode(wq)[:, :96] * np.repeat(ws[:, :3].astype(np.float64), 32, axis=1)).T
    np.testing.assert_allclose(y4, ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------- forward

def _tiny_problem(seed, M=3, H=64, I=64, E=3, k=2, masked=()):
    rng = np.random.default_rng(seed)
    x = bf16_round(rng.standard_normal((M, H)).astype(np.float32))
    aq, as_ = w4a8.quantize_act_per_row(x)
    w13 = bf16_round((rng.standard_normal((E, 2 * I, H)) * 0.1).astype(np.float32))
    w2 = bf16_round((rng.standard_normal((E, H, I)) * 0.1).astype(np.float32))
    w13q, w13s = w4a8.quantize_weight_k32(w13)
    w2q, w2s = w4a8.quantize_weight_k32(w2)
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


@pytest.mark.parametrize("seed,shape", [(20, dict(M=3, H=64, I=64, E=3, k=2)),
                                        (21, dict(M=2, H=96, I=32, E=4, k=3, masked=((1, 2),))),
                                        (22, dict(M=4, H=32, I=96, E=2, k=1))])
def test_forward_matches_fp64_brute_force(seed, shape):
    p = _tiny_problem(seed, **shape)
    out32, inter = w4a8.moe_forward_w4a8(**p, routed_scale=2.5, return_inter=True, round_bf16=False)
    out64, inter64 = w4a8.moe_forward_w4a8_fp64(**p, routed_scale=2.5)
    assert inter.keys() == inter64.keys()
    n_diff = 0
    for key, (codes, scale) in inter.items():
        c64, s64, ratio = inter64[key]
        diff = codes != c64
        assert (~diff | _near_tie(ratio)).all()
        n_diff += int(diff.sum())
        np.testing.assert_allclose(scale, s64, rtol=1e-6)
    assert n_diff <= 2
    rel = np.linalg.norm(out32 - out64) / np.linalg.norm(out64 - p["out_prior"])
    assert rel < 1e-5, rel


def test_forward_special_case_reduces_to_matmul_and_silu():
    """k = 1, route weight 1, all weight scales 1 and activation scale 1: the
    gate/up projection is a matmul of the decoded values and SwiGLU is
    torch's silu(gate) * up; the down projection then sees the per-row codes."""
    rng = np.random.default_rng(23)
    M, H, I, E = 3, 64, 32, 2
    aq = e4m3_encode((rng.standard_normal((M, H)) * 2).astype(np.float32))
    w13q = w4a8.e2m1_encode(rng.standard_normal((E, 2 * I, H)) * 2)
    w2q = w4a8.e2m1_encode(rng.standard_normal((E, H, I)) * 2)
    ids = np.array([[0], [1], [0]])
    out = w4a8.moe_forward_w4a8(aq, np.ones(M, np.float32), w13q, np.ones((E, 2 * I, H // 32), np.float32),
                                w2q, np.ones((E, H, I // 32), np.float32), ids, np.ones((M, 1), np.float32),
                                np.zeros((M, H), np.float32), round_bf16=False)
    for t in range(M):
        e = int(ids[t, 0])
        pre = torch.from_numpy(e4m3_decode(aq[t])) @ torch.from_numpy(w4a8.e2m1_decode(w13q[e])).T
        h = torch.nn.functional.silu(pre[:I]) * pre[I:]
        s = h.abs().max() / 448.0
        q = e4m3_decode(e4m3_encode((h / s).numpy()))
        y = torch.from_numpy(q) @ torch.from_numpy(w4a8.e2m1_decode(w2q[e])).T * s
        np.testing.assert_allclose(out[t], y.numpy(), rtol=1e-4, atol=1e-4 * float(y.abs().max()))


def test_forward_masked_routes_zero_scales_and_prior():
    p = _tiny_problem(24, M=3, H=64, I=32, E=3, k=2)
    # every route masked: out is the prior (rounded to BF16, already BF16 values)
    q = dict(p, topk_ids=np.full_like(p["topk_ids"], -1))
    np.testing.assert_array_equal(w4a8.moe_forward_w4a8(**q), p["out_prior"])
    # zero down-projection scales for one expert: its routes add nothing
    e0 = int(p["topk_ids"][0, 0])
    w2s = p["w2_s"].copy()
    w2s[e0] = 0
    q = dict(p, w2_s=w2s)
    only = dict(p, topk_ids=np.where(p["topk_ids"] == e0, -1, p["topk_ids"]))
    np.testing.assert_array_equal(w4a8.moe_forward_w4a8(**q), w4a8.moe_forward_w4a8(**only))


def test_forward_token_permutation_and_subset():
    p = _tiny_problem(25, M=4, H=64, I=32, E=3, k=2)
    full = w4a8.moe_forward_w4a8(**p)
    perm = np.array([2, 0, 3, 1])
    q = dict(p, a_q=p["a_q"][perm], a_s=p["a_s"][perm], topk_ids=p["topk_ids"][perm],
             topk_w=p["topk_w"][perm], out_prior=p["out_prior"][perm])
    np.testing.assert_array_equal(w4a8.moe_forward_w4a8(**q), full[perm])
    np.testing.assert_array_equal(w4a8.moe_forward_w4a8(**p, tokens=[3, 1]), full[[3, 1]])


def test_forward_expert_partitioned_is_bit_identical():
    """Experts computed in several threads, combined in the same fixed order,
    give exactly the single-threaded output and intermediate."""
    p = _tiny_problem(26, M=5, H=64, I=64, E=4, k=3, masked=((2, 1),))
    a, ia = w4a8.moe_forward_w4a8(**p, return_inter=True)
    b, ib = w4a8.moe_forward_w4a8(**p, return_inter=True, workers=3)
    np.testing.assert_array_equal(a, b)
    assert ia.keys() == ib.keys()
    for key in ia:
        np.testing.assert_array_equal(ia[key][0], ib[key][0])
        assert ia[key][1] == ib[key][1]


def test_forward_routed_scale_is_a_route_weight_factor():
    p = _tiny_problem(26, M=2, H=32, I=32, E=2, k=2)
    a = w4a8.moe_forward_w4a8(**p, routed_scale=2.0, round_bf16=False)
    b = w4a8.moe_forward_w4a8(**dict(p, topk_w=f32(p["topk_w"] * 2)), round_bf16=False)
    np.testing.assert_array_equal(a, b)


def test_forward_equals_block_fp8_forward_when_formats_coincide():
    """E2M1 values are E4M3 values, so weights whose K32 scales are constant
    over each 128x128 block, activations whose row scale is every group's
    scale, and I = 128 (one requant group per row) describe the same real
    numbers to both oracles.  They agree to FP32 accuracy despite different
    code: 32-wide against 128-wide blocks, the activation scale applied
    after the sum against inside each promotion."""
    from oracle import moe
    rng = np.random.default_rng(27)
    M, H, I, E, k = 5, 256, 128, 3, 2
    N = 2 * I
    aq = e4m3_encode((rng.standard_normal((M, H)) * 30).astype(np.float32))
    as_row = (rng.random(M) + 0.5).astype(np.float32)
    w13c = rng.integers(0, 16, size=(E, N, H)).astype(np.uint8)
    w2c = rng.integers(0, 16, size=(E, H, I)).astype(np.uint8)
    s13 = (rng.random((E, N // 128, H // 128)) * 0.01 + 0.001).astype(np.float32)
    s2 = (rng.random((E, H // 128, I // 128)) * 0.01 + 0.001).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int64)
    tw = rng.random((M, k)).astype(np.float32)
    prior = bf16_round((rng.standard_normal((M, H)) * 0.1).astype(np.float32))

    def k32(s):          # [E, R/128, C/128] -> one K32 scale per row and 32 columns
        return np.repeat(np.repeat(s, 128, axis=1), 4, axis=2)

    out4, inter4 = w4a8.moe_forward_w4a8(aq, as_row, w13c, k32(s13), w2c, k32(s2), ids, tw, prior,
                                         routed_scale=1.5, return_inter=True, round_bf16=False)
    out8, inter8 = moe.moe_forward(aq, np.repeat(as_row[:, None], H // 128, axis=1),
                                   e4m3_encode(w4a8.e2m1_decode(w13c)), s13,
                                   e4m3_encode(w4a8.e2m1_decode(w2c)), s2, ids, tw, prior,
                                   routed_scale=1.5, return_inter=True, round_bf16=False)
    n_diff = 0
    for key, (codes, scale) in inter4.items():
        c8, s8 = inter8[key]
        n_diff += int((codes != c8).sum())
        np.testing.assert_allclose(scale, s8[0], rtol=1e-6)
    assert n_diff <= 2
    rel = np.linalg.norm(out4.astype(np.float64) - out8) / np.linalg.norm(out8.astype(np.float64) - prior)
    assert rel < 1e-5, rel
