"""Oracle for the E2M1-K32 weight x FP8 activation expert computation.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy; float64
for exact sums, float32 where the method's arithmetic is FP32.

Page citations used below:

* [SM120-FP8] sglang-glm53-flash-sm120 pull request #13, description: the
  MoE experts whose weights are E2M1 codes with an FP32 scale for every 32
  elements of K ("K32") get an FP8-activation path; the K32 scales are
  applied in FP32, each activation row has one FP32 scale, and the weights
  stay in the form they were prepared in.  Its timed shape is E = 288,
  H = 4096, I = 1024 and top-8, and its checks include
  blocks only partly filled with rows, routes spread unevenly over the
  experts, experts whose weight scales are zero, and masked routes.
* E2M1 itself is the FP4 element type of the OCP Microscaling Formats (MX)
  specification; the page only names it.

The rest of the expert computation (SwiGLU, route weights, the reduction
onto a caller-owned BF16 output) is the block-FP8 path's, and is taken from
``oracle.moe`` unchanged.

Readings where the page is silent (numbered on from those of ``oracle.moe``
and listed in the design notes):

29. E2M1: 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; exponent
    field 0 is subnormal (m * 0.5); otherwise (1 + m/2) * 2**(e - 1).  The
    magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6; there is no NaN or infinity.
    Encoding rounds to nearest, ties to the even mantissa, saturates beyond 6
    (and infinities) to +-6, and keeps the sign of zero.
30. Storage packs two codes per byte, the even-indexed element in the low
    nibble.  Packing is storage only: everything below works on codes.
31. K32 weight quantisation: per output row and per 32 consecutive K
    elements, scale = f32(amax / 6) and codes = E2M1(f32(w / scale)); a block
    with amax 0 has scale 0 and zero codes.
32. Per-row activation quantisation: per token row over all K, scale =
    f32(amax / 448) and codes = E4M3(f32(x / scale)); a zero row has scale 0
    and zero codes.
33. GEMM: the dot over each 32-wide K block is exact and rounded once to
    FP32; the weight scale is applied per block in FP32 and the blocks are
    summed in order, acc = f32(acc + f32(dot * w_s)); the row's activation
    scale is constant along K and is applied once at the end,
    y = f32(acc * a_s).
34. The SwiGLU intermediate is requantised with the same per-row quantiser
    (reading 32) before the down projection.
"""

import numpy as np

from .moe import expert_routes, swiglu
from .numerics import E4M3_MAX, bf16_round, e4m3_decode, e4m3_encode, f32

K32 = 32          # the K extent of one weight scale block
E2M1_MAX = 6.0


# --------------------------------------------------------------------------
# E2M1 codec (reading 29) and nibble packing (reading 30)
# --------------------------------------------------------------------------

def e2m1_decode(codes):
    """Decode E2M1 codes (integers 0..15) to float64 values."""
    c = np.asarray(codes).astype(np.int32)
    assert ((c >= 0) & (c < 16)).all()
    e = (c >> 1) & 0x3
    m = c & 0x1
    # subnormal: m * 2**-1; normal: (2 + m) * 2**(e - 2)
    mag = np.ldexp(np.where(e == 0, m, 2 + m).astype(np.float64), np.where(e == 0, -1, e - 2))
    return np.where((c >> 3) == 1, -mag, mag)


def e2m1_encode(x):
    """Encode real values to E2M1 codes (uint8, 0..15).

    Within the binade [2**E, 2**(E+1)) the E2M1 spacing is 2**(E-1); below 1
    the subnormal spacing 0.5 applies, the same formula with E clamped to 0.
    r = |x| / 2**(E-1) is exact and ``np.round`` (halves to even) takes it to
    the nearest representable multiple; an even r is an even mantissa.  r
    lies in [2, 4] in a normal binade (4 carries into the next one) and in
    [0, 2] below 1.  NaN has no code and is rejected.
    """
    x = np.asarray(x, dtype=np.float64)
    assert not np.isnan(x).any()
    neg = np.signbit(x)
    a = np.minimum(np.abs(x), E2M1_MAX)     # saturate: beyond 6 (and inf) -> 6
    _, ex = np.frexp(a)                     # a = f * 2**ex, f in [0.5, 1)
    E = np.maximum(ex - 1, 0)               # binade exponent, subnormals share 0
    r = np.round(np.ldexp(a, 1 - E)).astype(np.int32)
    carry = r == 4
    E = E + carry
    r = np.where(carry, 2, r)
    normal = r >= 2
    e_field = np.where(normal, E + 1, 0)
    m_field = np.where(normal, r - 2, r)
    return ((neg.astype(np.int32) << 3) | (e_field << 1) | m_field).astype(np.uint8)


def pack_e2m1(codes):
    """codes uint8 [..., K] (K even) -> bytes uint8 [..., K/2]; element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    assert c.shape[-1] % 2 == 0 and (c < 16).all()
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed):
    """bytes uint8 [..., K/2] -> codes uint8 [..., K] (inverse of ``pack_e2m1``)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# --------------------------------------------------------------------------
# Quantisers (readings 31, 32)
# --------------------------------------------------------------------------

def quantize_weight_k32(w):
    """K32 weight quantisation ([SM120-FP8]; reading 31).

    w: float32 [..., rows, K] -> (codes uint8 [..., rows, K] (unpacked),
    scale float32 [..., rows, K/32]).
    """
    w = f32(w)
    K = w.shape[-1]
    assert K % K32 == 0
    g = w.reshape(w.shape[:-1] + (K // K32, K32))
    scale = f32(np.max(np.abs(g), axis=-1) / np.float32(E2M1_MAX))
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = e2m1_encode(f32(g / safe[..., None]))
    codes = np.where((scale > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(w.shape), scale


def dequantize_weight_k32(codes, scale):
    """float64 values of K32-quantised weights (codes [..., rows, K], scale [..., rows, K/32])."""
    return e2m1_decode(codes) * np.repeat(np.asarray(scale, dtype=np.float64), K32, axis=-1)


def quantize_act_per_row(x):
    """Per-row FP8 activation quantisation ([SM120-FP8]; reading 32).

    x: float32 [M, K] (BF16 values) -> (codes uint8 [M, K], scale float32 [M]).
    """
    x = f32(x)
    scale = f32(np.max(np.abs(x), axis=-1) / np.float32(E4M3_MAX))
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = e4m3_encode(f32(x / safe[:, None]))
    codes = np.where((scale > 0)[:, None], codes, np.uint8(0)).astype(np.uint8)
    return codes, scale


# --------------------------------------------------------------------------
# GEMM (reading 33)
# --------------------------------------------------------------------------

def k32_dots(xq, wq):
    """Exact per-32-block dot products, rounded once to FP32.

    xq: uint8 [n, K] E4M3 codes, wq: uint8 [J, K] E2M1 codes -> float32
    [n, J, K/32] with dots[i, j, kb] = f32(sum_{c<32} x[i, 32kb+c] * w[j, 32kb+c]).
    E4M3 values are multiples of 2**-9 and E2M1 values multiples of 2**-1, so
    every product is a multiple of 2**-10 of magnitude at most 448 * 6 < 2**12;
    any partial sum of 32 of them fits in 27 bits and float64 holds it exactly.
    """
    x = e4m3_decode(xq)
    w = e2m1_decode(wq)
    n, K = x.shape
    nkb = K // K32
    out = np.empty((n, w.shape[0], nkb), dtype=np.float32)
    for kb in range(nkb):
        sl = slice(kb * K32, (kb + 1) * K32)
        out[:, :, kb] = f32(x[:, sl] @ w[:, sl].T)
    return out


def gemm_w4a8(xq, xs, wq, ws):
    """One expert's projection ([SM120-FP8]; reading 33).

    xq [n, K] E4M3 codes, xs [n] f32 row scales, wq [J, K] E2M1 codes,
    ws [J, K/32] f32 -> y [n, J] f32 with acc = f32(acc + f32(dot * w_s))
    over K blocks in order, then y = f32(acc * a_s).
    """
    dots = k32_dots(xq, wq)
    ws = f32(ws)
    acc = np.zeros(dots.shape[:2], dtype=np.float32)
    for kb in range(dots.shape[2]):
        acc = f32(acc + f32(dots[:, :, kb] * ws[None, :, kb]))
    return f32(acc * f32(xs)[:, None])


# --------------------------------------------------------------------------
# Forward
# --------------------------------------------------------------------------

def moe_forward_w4a8(a_q, a_s, w13_q, w13_s, w2_q, w2_s, topk_ids, topk_w,
                     out_prior, routed_scale=1.0, tokens=None, return_inter=False,
                     round_bf16=True, workers=1):
    """Fused MoE expert forward with E2M1-K32 weights and per-row FP8
    activations, FP32 emulation ([SM120-FP8]; readings 29-34 and, for the
    steps shared with the block-FP8 path, 1, 6-8 of ``oracle.moe``).

    a_q [M,H] E4M3 codes, a_s [M] f32; w13_q [E,2I,H] E2M1 codes (unpacked,
    gate rows then up rows), w13_s [E,2I,H/32]; w2_q [E,H,I] E2M1 codes,
    w2_s [E,H,I/32]; topk_ids [M,k] int, topk_w [M,k] f32; out_prior [M,H]
    BF16 values as float32.

    Returns out [len(tokens), H] float32 holding BF16 values (the FP32
    accumulator with ``round_bf16=False``); with ``return_inter`` also
    {(t, j): (codes [I], scale)} of the requantised intermediate.  A token's
    routes are added in slot order in FP32 onto the prior value, then rounded
    once to BF16.  ``workers`` > 1 computes the experts' routes in that many
    threads and combines them in the same fixed order, so the output is
    bit-identical to ``workers=1``.
    """
    M, H = a_q.shape
    E, N, _ = w13_q.shape
    I = N // 2
    k = np.asarray(topk_ids).shape[1]
    if tokens is None:
        tokens = np.arange(M)
    tokens = np.asarray(tokens, dtype=np.int64)
    rs = np.float32(routed_scale)
    route_y = {}
    inter = {}

    def expert_part(e, ts, js):
        acc = gemm_w4a8(a_q[ts], np.asarray(a_s)[ts], w13_q[e], w13_s[e])
        h = swiglu(acc, I)
        qi, si = quantize_act_per_row(h)
        y = gemm_w4a8(qi, si, w2_q[e], w2_s[e])
        wr = f32(f32(np.asarray(topk_w)[ts, js]) * rs)
        return ts, js, f32(y * wr[:, None]), qi, si

    groups = sorted(expert_routes(topk_ids, E, tokens).items())
    if workers > 1:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(max_workers=workers) as pool:
            parts = list(pool.map(lambda g: expert_part(g[0], *g[1]), groups))
    else:
        parts = [expert_part(e, ts, js) for e, (ts, js) in groups]
    for ts, js, y, qi, si in parts:
        for n, (t, j) in enumerate(zip(ts, js)):
            route_y[(int(t), int(j))] = y[n]
            if return_inter:
                inter[(int(t), int(j))] = (qi[n], si[n])
    out = np.empty((tokens.size, H), dtype=np.float32)
    prior = f32(out_prior)
    for i, t in enumerate(tokens):
        acc = prior[t].copy()
        for j in range(k):
            y = route_y.get((int(t), j))
            if y is not None:
                acc = f32(acc + y)
        out[i] = bf16_round(acc) if round_bf16 else acc
    if return_inter:
        return out, inter
    return out


def moe_forward_w4a8_fp64(a_q, a_s, w13_q, w13_s, w2_q, w2_s, topk_ids, topk_w,
                          out_prior, routed_scale=1.0):
    """Route-by-route float64 evaluation of the same definition.

    Written independently of the emulation above: loops over routes and
    output columns, every weight dequantised element by element from its own
    K32 scale, no FP32 rounding anywhere except that the intermediate is
    still encoded to E4M3 codes (from float64 values) before the down
    projection.  Returns (out_f64 [M, H] before BF16 rounding,
    {(t, j): (codes, scale, h/scale)}).
    """
    M, H = a_q.shape
    E, N, _ = w13_q.shape
    I = N // 2
    k = np.asarray(topk_ids).shape[1]
    out = np.asarray(out_prior, dtype=np.float64).copy()
    inter = {}
    for t in range(M):
        x = e4m3_decode(a_q[t]) * float(a_s[t])
        for j in range(k):
            e = int(topk_ids[t, j])
            if not (0 <= e < E):
                continue
            pre = np.zeros(N)
            for n in range(N):
                w = e2m1_decode(w13_q[e, n]) * np.array([float(w13_s[e, n, c // K32]) for c in range(H)])
                pre[n] = float(np.dot(x, w))
            g, u = pre[:I], pre[I:]
            h = g / (1.0 + np.exp(-g)) * u
            s = np.max(np.abs(h)) / E4M3_MAX
            codes = e4m3_encode(h / s) if s > 0 else np.zeros(I, dtype=np.uint8)
            inter[(t, j)] = (codes, s, h / s if s > 0 else np.zeros(I))
            hq = e4m3_decode(codes) * s
            y = np.zeros(H)
            for hh in range(H):
                w = e2m1_decode(w2_q[e, hh]) * np.array([float(w2_s[e, hh, c // K32]) for c in range(I)])
                y[hh] = float(np.dot(hq, w))
            out[t] += y * float(topk_w[t, j]) * float(routed_scale)
    return out, inter
