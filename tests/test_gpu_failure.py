"""Failure detection on the GPU without a fault.

Every pipeline wait of the GEMM kernels is bounded; when one runs out the CTA
raises its abort flag, the other waits of the CTA give up at once, the CTA
reports MOE_DEV_TIMEOUT in *device_status and returns.  The self-test entry
point drives exactly that wait on an mbarrier nothing arrives at, with a
short limit, and the context must stay usable: a normal forward right after
it matches the oracle.
"""

import numpy as np
import pytest
import torch

import workloads as W
from fp8_block_scale_gb300 import _lib as L
from fp8_block_scale_gb300.problem import DeviceProblem
from oracle import moe as O
from oracle.inputs import MAX_ABS_TOL, REL_L2_TOL, oracle_inputs, out_metrics

pytestmark = pytest.mark.gpu

MOE_ERR_TIMEOUT = 8


@pytest.mark.parametrize("limit_us", [2000, 20000])
def test_bounded_wait_runs_out_and_the_context_stays_usable(limit_us):
    L.load()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert L.moe_selftest_wait_timeout(limit_us, status, elapsed) == MOE_ERR_TIMEOUT
    assert int(status.item()) & L.MOE_DEV_TIMEOUT
    waited = elapsed.cpu().numpy() * 1e-9
    print(f"limit {limit_us} us: waits gave up after {waited[0] * 1e3:.3f} ms and {waited[1] * 1e3:.3f} ms")
    # the barrier nobody arrives at: at least the limit, and well before the
    # pipelines' normal one-second bound
    assert limit_us * 1e-6 <= waited[0] < 0.5
    # the other warp stopped on the abort flag, not on its own one-second limit
    assert 0 < waited[1] < 0.5

    # the same context runs a normal forward
    cfg = W.CONFIGS["tiny"]
    prob = DeviceProblem(cfg)
    prob.run_plan()
    prob.run_forward(prob.fwd_args(tile_mode=L.TILE_SINGLE))
    torch.cuda.synchronize()
    inp, _ = oracle_inputs(cfg, prob.routing, np.arange(cfg.M))
    m = out_metrics(prob.out.float().cpu().numpy(), O.moe_forward(**inp, routed_scale=cfg.routed_scale))
    assert m["rel_l2"] <= REL_L2_TOL and m["max_rel"] <= MAX_ABS_TOL, m
    assert int(prob.status.item()) == 0
