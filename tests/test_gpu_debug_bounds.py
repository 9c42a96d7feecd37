"""The bounds-checking build (libmoe_fp8_debug.so, -DMOE_DEBUG_BOUNDS) on
the GPU.  Every data-derived global index and tensor-copy coordinate of its
kernels is checked before the access; a failure is counted in a device-side
record and the access skipped.  The small parity cases of both forwards, in
each of their paths, run through it: results still match the oracle and no
check fails.  A self-test shows that a failing check is counted and stops
its access."""

import numpy as np
import pytest
import torch

from fp8_block_scale_gb300 import _lib as L
from fp8_block_scale_gb300.build import build
from fp8_block_scale_gb300.problem import DeviceProblem, W4A8Problem
import workloads as W
from tests import test_gpu_forward as F
from tests import test_gpu_w4a8 as F4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _debug_library():
    build(debug_bounds=True)
    with L.use_library(L.LIB_DEBUG_PATH):
        assert L.moe_debug_bounds_enabled()
        L.moe_debug_bounds_read(reset=True)
        yield


def _no_failures(label):
    n, f, line = L.moe_debug_bounds_read(reset=True)
    assert n == 0, f"{label}: {n} bounds checks failed, first at {f}:{line}"


def test_selftest_counts_a_failed_check_and_skips_the_access():
    data = torch.arange(10, 14, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_debug_bounds_selftest(data, 2, out)
    assert int(out.item()) == 12
    _no_failures("in-range probe")
    for probe in (4, -1, 1000):
        L.moe_debug_bounds_selftest(data, probe, out)
        assert int(out.item()) == -1
    n, f, line = L.moe_debug_bounds_read(reset=True)
    assert n == 3 and f == "api.cu" and line > 0, (n, f, line)
    _no_failures("after reset")


FP8_CASES = [(name, L.TILE_SINGLE, L.SCALES_FP32) for name in F.SMALL]
FP8_CASES += [(name, L.TILE_VECTOR, L.SCALES_FP32) for name in F.VECTOR_SMALL]
FP8_CASES += [(name, L.TILE_PAIR, L.SCALES_FP32) for name in ("ragged_bm128", "hot_many_blocks")]
FP8_CASES += [(name, L.TILE_SINGLE, L.SCALES_UE8M0) for name in ("ue8m0_both", "bs_masked_zero", "bs_ragged_bm8")]
_ALL_FP8 = {**F.SMALL, **F.BLOCK_SCALED}


@pytest.mark.parametrize("name,mode,scales", FP8_CASES,
                         ids=[f"{n}-{['auto', 'single', 'pair', 'vector'][m]}-{['fp32', 'ue8m0'][s]}"
                              for n, m, s in FP8_CASES])
def test_fp8_forward_under_bounds_checks(name, mode, scales):
    prob = DeviceProblem(_ALL_FP8[name])
    dq, ds = F._run(prob, tile_mode=mode, scale_mode=scales)
    _no_failures(name)
    F._check(prob, np.arange(prob.cfg.M), dq, ds, "debug-bounds")
    assert int(prob.status.item()) == 0


def test_plan_of_many_routes_under_bounds_checks():
    """More routes than the one-CTA plan takes: the three-launch plan."""
    cfg = W.MoEConfig("bounds_plan", M=700, H=256, I=128, E=40, top_k=4, block_m=16, routing="skewed",
                      n_hot=3, hot_frac=0.5)
    prob = DeviceProblem(cfg)
    dq, ds = F._run(prob)
    _no_failures(cfg.name)
    F._check(prob, np.arange(cfg.M), dq, ds, "debug-bounds")


W4_CASES = [(name, path) for name in F4.CASES for path in (L.W4A8_AUTO, L.W4A8_CUDA_CORES)]


@pytest.mark.parametrize("name,path", W4_CASES,
                         ids=[f"{n}-{'auto' if p == L.W4A8_AUTO else 'cuda_cores'}" for n, p in W4_CASES])
def test_w4a8_forward_under_bounds_checks(name, path):
    prob = W4A8Problem(F4.CASES[name])
    dq, ds = F4._run(prob, path=path)
    _no_failures(name)
    F4._check(prob, np.arange(prob.cfg.M), dq, ds)
    assert int(prob.status.item()) == 0


def test_noalloc_forward_under_bounds_checks():
    prob = DeviceProblem(W.CONFIGS["decode_m8"])
    prob.run_plan()
    L.moe_fp8_block_scale_forward_noalloc(prob.fwd_args())
    torch.cuda.synchronize()
    _no_failures("noalloc decode_m8")
    F._check(prob, np.arange(prob.cfg.M), label="debug-bounds noalloc")


@pytest.mark.parametrize("M,E,k,bm", [(1, 257, 9, 64), (113, 288, 9, 16), (1024, 1024, 1, 128)])
def test_route_plan_under_bounds_checks(M, E, k, bm):
    """Router and plan in one launch: no check fails, and the plan matches
    moe_plan on the ids it wrote."""
    rng = np.random.default_rng(M + E)
    logits = torch.from_numpy((rng.standard_normal((M, E)) * 2.0).astype(np.float32)).cuda()
    cap, bcap = L.moe_plan_capacity(M, k, E, bm)
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    s1 = torch.full((cap,), -3, dtype=torch.int32, device="cuda")
    e1 = torch.full((bcap,), -3, dtype=torch.int32, device="cuda")
    p1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_route_plan(logits, k, ids, w, bm, s1, e1, p1)
    _no_failures(f"route_plan m{M}")
    s2, e2, p2 = s1.clone().fill_(-3), e1.clone().fill_(-3), p1.clone()
    ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device="cuda")
    L.moe_plan(ids, E, bm, s2, e2, p2, ws)
    _no_failures(f"plan m{M}")
    assert torch.equal(s1, s2) and torch.equal(e1, e2) and int(p1.item()) == int(p2.item())
