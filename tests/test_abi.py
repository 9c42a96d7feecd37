"""The C ABI library loads and exports every symbol include/*.h declares;
host-only entry points and host-side argument validation (no GPU needed)."""

import ctypes
import glob
import os
import re

import pytest

from oracle import moe as oracle_moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_block_scale_gb300 import _lib
    from fp8_block_scale_gb300.build import build
    build()
    return _lib.load()


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//.*", "", src)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("moe_plan", "moe_prep_weights", "moe_requant_scales_ue8m0", "moe_fp8_block_scale_forward"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    from fp8_block_scale_gb300 import moe_status_string
    assert moe_status_string(0) == "MOE_OK"
    assert moe_status_string(2).startswith("MOE_ERR_SHAPE")
    assert "unknown" in moe_status_string(99)


@pytest.mark.parametrize("M,k,E,bm", [(16, 2, 8, 64), (1, 9, 257, 64), (8192, 8, 288, 128), (4096, 10, 512, 128),
                                      (3, 1, 1, 8)])
def test_plan_capacity_matches_oracle(lib, M, k, E, bm):
    from fp8_block_scale_gb300 import moe_plan_capacity
    assert moe_plan_capacity(M, k, E, bm) == oracle_moe.plan_capacity(M, k, E, bm)


def test_workspace_sizes(lib):
    from fp8_block_scale_gb300 import moe_forward_workspace_size, moe_plan_workspace_size
    ws = moe_forward_workspace_size(8192, 4096, 1024, 288, 8, 128, 102400)
    # BF16 route contributions + intermediate + activation rows in plan order (well-filled plan)
    assert ws >= 8192 * 8 * 4096 * 2 + 102400 * 1024 + 102400 * 8 * 4 + 102400 * 4096
    # a decode-sized plan keeps the activations where they are
    small = moe_forward_workspace_size(8, 7168, 256, 257, 9, 64, 4608)
    assert 72 * 7168 * 2 + 4608 * 256 <= small < 72 * 7168 * 2 + 4608 * 256 + 4608 * 7168
    assert moe_forward_workspace_size(8, 7168, 256, 0, 9, 64, 4608) == 0
    # sizes the vector path supports also hold its FP32 silu(gate) * up rows
    # by route ([R, I] floats); one token more than it takes does not
    at64 = moe_forward_workspace_size(64, 256, 256, 8, 2, 64, 64 * 2 + 8 * 63)
    at65 = moe_forward_workspace_size(65, 256, 256, 8, 2, 64, 64 * 2 + 8 * 63)
    # (65 tokens add two routes' rows elsewhere: 2 x 256 x 2 bytes, plus rounding)
    assert 128 * 256 * 4 - 2048 <= at64 - at65 <= 128 * 256 * 4
    assert moe_plan_workspace_size(8192, 8, 288) >= 8192 * 8 * 4 + 288 * 4


def _fake(n):
    return ctypes.c_void_p(n)


def test_forward_host_validation_without_gpu(lib):
    """Argument errors are reported on the host before any device call."""
    from fp8_block_scale_gb300._lib import MoeFwdArgs
    f = lib.moe_fp8_block_scale_forward
    assert f(None, None) == 1                                    # MOE_ERR_NULL
    a = MoeFwdArgs()
    a.M, a.H, a.I, a.E, a.top_k, a.block_m = 4, 256, 256, 8, 2, 64
    a.sorted_cap, a.blocks_cap = 640, 10
    a.H = 200
    assert f(ctypes.byref(a), None) == 2                         # H % 128
    a.H = 256
    a.block_m = 12
    assert f(ctypes.byref(a), None) == 2                         # block_m % 8
    a.block_m = 256
    assert f(ctypes.byref(a), None) == 2                         # block_m > 128
    a.block_m = 64
    for bad in (-1, 4):
        a.tile_mode = bad
        assert f(ctypes.byref(a), None) == 2                     # unknown tile mode
    a.tile_mode = 3                                              # the vector path ...
    a.M = 65
    assert f(ctypes.byref(a), None) == 2                         # ... takes at most 64 tokens
    a.M, a.I = 4, 1152
    assert f(ctypes.byref(a), None) == 2                         # ... and I <= 1024
    a.M, a.I, a.top_k = 64, 256, 17
    assert f(ctypes.byref(a), None) == 2                         # ... and M * top_k <= 1024 routes
    a.M, a.top_k, a.H = 4, 2, 8320
    assert f(ctypes.byref(a), None) == 2                         # ... and H <= 8192
    a.H = 256
    a.tile_mode = 2
    a.sorted_cap = 639
    assert f(ctypes.byref(a), None) == 4                         # capacity
    a.sorted_cap = 640
    assert f(ctypes.byref(a), None) == 1                         # null pointers
    for name in ("a", "a_scale", "w13", "w13_scale", "w2", "w2_scale", "topk_weights", "sorted_token_ids",
                 "expert_ids", "num_tokens_post_padded", "out", "workspace"):
        setattr(a, name, 4096)
    a.w13 = 4100                                                 # misaligned
    assert f(ctypes.byref(a), None) == 3
    a.w13 = 4096
    a.workspace_bytes = 10
    assert f(ctypes.byref(a), None) == 4                         # workspace too small
    a.M = 0
    assert f(ctypes.byref(a), None) == 0                         # nothing to do


def test_plan_and_prep_host_validation_without_gpu(lib):
    assert lib.moe_plan(None, 32, 4, 2, 8, 64, None, 0, None, 0, None, None, 0, None) == 1
    p = _fake(4096)
    assert lib.moe_plan(p, 16, 4, 2, 8, 64, p, 640, p, 10, p, p, 1 << 20, None) == 5      # id width
    assert lib.moe_plan(p, 32, 4, 2, 8, 60, p, 640, p, 10, p, p, 1 << 20, None) == 2      # block_m
    assert lib.moe_plan(p, 32, 4, 2, 4096, 64, p, 640, p, 10, p, p, 1 << 20, None) == 2   # E too large
    assert lib.moe_plan(p, 32, 4, 2, 8, 64, p, 64, p, 1, p, p, 1 << 20, None) == 4        # capacity
    assert lib.moe_prep_weights(p, p, 2, 250, 128, None) == 2
    assert lib.moe_prep_weights(_fake(4097), p, 2, 256, 128, None) == 3
    assert lib.moe_prep_weights(p, p, 2, 256, 128, None) == 2                             # overlap
    assert lib.moe_requant_scales_ue8m0(p, p, None, 1, 100, 128, None) == 2
    assert lib.moe_quantize_act_1x128(p, 4, 100, p, p, None) == 2
    assert lib.moe_quantize_act_1x128_ue8m0(p, 4, 100, p, p, None) == 2
    assert lib.moe_quantize_act_1x128_ue8m0(None, 4, 128, p, p, None) == 1
    assert lib.moe_quantize_weight_128x128(p, 1, 128, 64, p, p, None) == 2


def test_router_host_validation_without_gpu(lib):
    """moe_route_topk rejects bad arguments on the host, before any device call."""
    f = lib.moe_route_topk
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    p = ctypes.c_void_p(4096)
    assert f(p, 2, 4, 8, 2, 1.0, 1, p, 32, p, None) == 5          # unknown logit dtype
    assert f(p, 0, 4, 8, 2, 1.0, 1, p, 16, p, None) == 5          # id width
    assert f(p, 0, 4, 8, 9, 1.0, 1, p, 32, p, None) == 2          # top_k > E
    assert f(p, 0, 4, 64, 33, 1.0, 1, p, 32, p, None) == 2        # top_k > 32
    assert f(p, 0, 4, 2049, 2, 1.0, 1, p, 32, p, None) == 2       # E too large
    assert f(p, 0, -1, 8, 2, 1.0, 1, p, 32, p, None) == 2         # negative M
    assert f(None, 0, 4, 8, 2, 1.0, 1, p, 32, p, None) == 1       # null logits
    assert f(None, 0, 0, 8, 2, 1.0, 1, None, 32, None, None) == 0  # nothing to do


def test_w4a8_host_validation_without_gpu(lib):
    """moe_w4a8_forward and its quantisers reject bad arguments on the host."""
    from fp8_block_scale_gb300._lib import MoeW4A8Args
    f = lib.moe_w4a8_forward
    assert f(None, None) == 1                                    # MOE_ERR_NULL
    a = MoeW4A8Args()
    a.M, a.H, a.I, a.E, a.top_k, a.block_m = 4, 256, 128, 8, 2, 16
    a.sorted_cap, a.blocks_cap = 160, 10
    a.routed_scale = 1.0
    for field, bad in (("H", 240), ("H", 0), ("I", 48), ("I", 16), ("top_k", 65), ("top_k", 0), ("E", 0),
                       ("block_m", 12), ("block_m", 72), ("block_m", 0), ("M", -1)):
        good = getattr(a, field)
        setattr(a, field, bad)
        assert f(ctypes.byref(a), None) == 2, (field, bad)     # MOE_ERR_SHAPE
        setattr(a, field, good)
    a.block_m, a.H = 64, 4096
    assert f(ctypes.byref(a), None) == 2                         # block_m * H above 128 KiB
    a.block_m, a.H = 16, 256
    a.sorted_cap = 159
    assert f(ctypes.byref(a), None) == 4                         # capacity
    a.sorted_cap = 160
    assert f(ctypes.byref(a), None) == 1                         # null pointers
    for name in ("a", "a_scale", "w13", "w13_scale", "w2", "w2_scale", "topk_weights", "sorted_token_ids",
                 "expert_ids", "num_tokens_post_padded", "out", "workspace"):
        setattr(a, name, 4096)
    a.debug_q_inter = 4096
    assert f(ctypes.byref(a), None) == 1                         # debug codes without their scales
    a.debug_q_inter = None
    a.w2 = 4100
    assert f(ctypes.byref(a), None) == 3                         # misaligned
    a.w2 = 4096
    a.workspace_bytes = lib.moe_w4a8_workspace_size(4, 256, 128, 2) - 1
    assert f(ctypes.byref(a), None) == 4                         # workspace too small
    a.M = 0
    assert f(ctypes.byref(a), None) == 0                         # nothing to do

    p = _fake(4096)
    assert lib.moe_quantize_act_per_row(p, 4, 100, p, p, None) == 2
    assert lib.moe_quantize_act_per_row(p, -1, 128, p, p, None) == 2
    assert lib.moe_quantize_act_per_row(None, 4, 128, p, p, None) == 1
    assert lib.moe_quantize_act_per_row(_fake(4097), 4, 128, p, p, None) == 3
    assert lib.moe_quantize_act_per_row(None, 0, 128, None, None, None) == 0
    assert lib.moe_quantize_weight_k32(p, 4, 48, p, p, None) == 2
    assert lib.moe_quantize_weight_k32(p, 0, 64, p, p, None) == 2
    assert lib.moe_quantize_weight_k32(None, 4, 64, p, p, None) == 1
    assert lib.moe_quantize_weight_k32(p, 4, 64, _fake(4104), p, None) == 3


def test_w4a8_workspace_size(lib):
    """Route flags, SwiGLU rows (FP32), their codes, row scales and the FP32
    route contributions, each region rounded up to 256 bytes."""
    def r256(n):
        return -(-n // 256) * 256
    for M, H, I, k in ((3, 256, 128, 2), (1, 4096, 1024, 8), (37, 384, 96, 3), (0, 256, 128, 2)):
        R = M * k
        want = r256(4 * R) + r256(4 * R * I) + r256(R * I) + r256(4 * R) + r256(4 * R * H)
        assert lib.moe_w4a8_workspace_size(M, H, I, k) == want
    assert lib.moe_w4a8_workspace_size(-1, 256, 128, 2) == 0
    assert lib.moe_w4a8_workspace_size(4, 256, 128, 0) == 0


def test_selftest_host_validation_without_gpu(lib):
    """The failure-detection self-test checks its arguments on the host."""
    f = lib.moe_selftest_wait_timeout
    assert f(1000, None, _fake(256), None) == 1                  # MOE_ERR_NULL
    assert f(1000, _fake(256), None, None) == 1
    assert f(0, _fake(256), _fake(512), None) == 2               # limit below 1 us
    assert f(1000001, _fake(256), _fake(512), None) == 2         # limit above 1 s


@pytest.fixture(scope="module")
def debug_lib():
    from fp8_block_scale_gb300 import _lib
    from fp8_block_scale_gb300.build import build
    build(debug_bounds=True)
    return _lib.load(_lib.LIB_DEBUG_PATH)


def test_debug_bounds_switch_without_gpu(lib, debug_lib):
    """The normal build has no bounds records (reading them needs no device);
    the bounds-checking build says so and exports the same entry points."""
    n = ctypes.c_uint64(7)
    f = ctypes.c_char_p(b"x")
    line = ctypes.c_int32(3)
    assert lib.moe_debug_bounds_enabled() == 0
    assert lib.moe_debug_bounds_read(ctypes.byref(n), ctypes.byref(f), ctypes.byref(line), 1) == 0
    assert (n.value, f.value, line.value) == (0, None, 0)
    assert lib.moe_debug_bounds_read(None, None, None, 0) == 1
    # an out-of-range probe is refused on the host by the normal build
    p = _fake(4096)
    assert lib.moe_debug_bounds_selftest(p, 4, 4, p, None) == 2
    assert lib.moe_debug_bounds_selftest(p, 4, -1, p, None) == 2
    assert lib.moe_debug_bounds_selftest(None, 4, 0, p, None) == 1
    assert lib.moe_debug_bounds_selftest(p, 0, 0, p, None) == 2
    assert debug_lib.moe_debug_bounds_enabled() == 1
    missing = [name for name in _declared_functions() if not hasattr(debug_lib, name)]
    assert not missing, missing


def test_route_plan_host_validation_without_gpu(lib):
    """moe_route_plan rejects bad arguments on the host, before any device call."""
    f = lib.moe_route_plan
    p = _fake(4096)
    ok = dict(logits=p, dtype=0, M=4, E=64, k=4, scale=1.0, renorm=1, ids=p, bits=32, w=p, bm=64,
              s=p, cap=4096, e=p, bcap=64, ntpp=p)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["logits"], a["dtype"], a["M"], a["E"], a["k"], a["scale"], a["renorm"], a["ids"], a["bits"],
                 a["w"], a["bm"], a["s"], a["cap"], a["e"], a["bcap"], a["ntpp"], None)
    assert call(dtype=2) == 5                      # logit dtype
    assert call(bits=16) == 5                      # id width
    assert call(E=1025) == 2                       # more experts than the one-CTA plan takes
    assert call(M=129, k=8) == 2                   # 1032 routes > 1024
    assert call(k=65) == 2
    assert call(k=0) == 2
    assert call(bm=12) == 2
    assert call(M=-1) == 2
    assert call(s=None) == 1
    assert call(logits=None) == 1
    assert call(cap=10) == 4                       # plan capacity

