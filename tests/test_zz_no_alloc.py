"""The allocation-free forward (moe_fp8_block_scale_forward_noalloc).

Some callers cannot allocate device memory: an engine that reserved all of
it for its own pool, a plug-in that only sees this C ABI, or a latency-bound
loop where an allocation may synchronise the device.  This entry point takes
the same arguments as the regular forward but uses a static device array as
scratch instead of the caller's workspace.  Its result must match the regular
forward's, call after call, within the forward's usual tolerances, and the
CPU oracle's within the forward's acceptance bar.  The cases take both
forward paths: the tensor-core tiles (ragged, decode_m8) and the vector path
(decode_m1, the single-token decode step such callers run most).
"""

import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from fp8_block_scale_gb300 import _lib as L
from fp8_block_scale_gb300.problem import DeviceProblem
from oracle import moe as O
from oracle.inputs import MAX_ABS_TOL, REL_L2_TOL, default_workers, oracle_inputs, out_metrics

pytestmark = pytest.mark.gpu

CASES = {
    "ragged": W.MoEConfig("ragged", M=37, H=384, I=256, E=5, top_k=3, block_m=64, out_init="normal0.1"),
    "decode_m8": W.CONFIGS["decode_m8"],
    "decode_m1": W.CONFIGS["decode_m1"],
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_forward_matches_workspace_forward_twice(name):
    lib = L.load()
    prob = DeviceProblem(CASES[name])
    prob.run_plan()
    ref = prob.out_prior.clone()
    prob.run_forward(prob.fwd_args(out=ref))
    torch.cuda.synchronize()
    ref_np = ref.float().cpu().numpy()
    cfg = CASES[name]
    inp, _ = oracle_inputs(cfg, prob.routing, np.arange(cfg.M))
    oracle_out = O.moe_forward(**inp, routed_scale=cfg.routed_scale, workers=default_workers())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        out = prob.out_prior.clone()
        args = prob.fwd_args(out=out)
        args.workspace = None           # ignored by the allocation-free entry point
        args.workspace_bytes = 0
        assert lib.moe_fp8_block_scale_forward_noalloc(ctypes.byref(args), stream) == 0
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        m = out_metrics(got, ref_np)
        assert m["rel_l2"] <= REL_L2_TOL and m["max_rel"] <= MAX_ABS_TOL, (call, m)
        m = out_metrics(got, oracle_out)
        assert m["rel_l2"] <= REL_L2_TOL and m["max_rel"] <= MAX_ABS_TOL, (call, "oracle", m)
        assert int(prob.status.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = L.load()
    cap_bytes = lib.moe_noalloc_scratch_bytes()
    assert cap_bytes == 32 << 20
    args = L.MoeFwdArgs()
    args.M, args.H, args.I, args.E, args.top_k, args.block_m = 8192, 4096, 1024, 288, 8, 128
    args.sorted_cap, args.blocks_cap = 102400, 800
    assert lib.moe_forward_workspace_size(8192, 4096, 1024, 288, 8, 128, 102400) > cap_bytes
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_fp8_block_scale_forward_noalloc(ctypes.byref(args), stream) == 4   # MOE_ERR_CAPACITY
