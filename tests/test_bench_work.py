"""The benchmark's algorithmic work model (CPU only): the FLOPs and bytes
every reported TFLOP/s figure and roofline fraction divides by, against
hand-computed closed forms."""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_decode_one_token_closed_form():
    # M = 1, H = 7168, I = 256, top-9 over 9 distinct experts of 257
    cfg = W.CONFIGS["decode_m1"]
    w = bench.work(cfg, np.arange(9)[None, :] * 7)
    assert (w["Rv"], w["U"]) == (9, 9)
    assert w["total"]["flop"] == 9 * 6 * 7168 * 256 == 99_090_432
    # per expert: 3*H*I code bytes + 4 * (2I/128 * H/128 + H/128 * I/128) scale bytes
    per_expert = 3 * 7168 * 256 + 4 * (4 * 56 + 56 * 2)
    assert per_expert == 5_506_368
    # + activations with their scales, out read and written, 8 bytes per route
    assert w["total"]["bytes"] == 9 * per_expert + (7168 + 4 * 56) + 4 * 7168 + 8 * 9 == 49_593_448


def test_prefill_8192_closed_form():
    cfg = W.CONFIGS["prefill_8192"]
    ids = np.arange(8192 * 8).reshape(8192, 8) % 288           # every expert touched
    w = bench.work(cfg, ids)
    assert (w["Rv"], w["U"]) == (65536, 288)
    assert w["total"]["flop"] == 65536 * 6 * 4096 * 1024 == 1_649_267_441_664
    per_expert = 3 * 4096 * 1024 + 4 * (16 * 32 + 32 * 8)
    acts = 8192 * (4096 + 4 * 32)
    assert w["total"]["bytes"] == 288 * per_expert + acts + 4 * 8192 * 4096 + 8 * 65536 == 3_794_108_416
    # the gate/up launch (the roofline's kernel): W13 codes and scales of every
    # touched expert, the activation rows with their scales, the intermediate
    # codes and scales it writes
    up_bytes = 288 * (2 * 1024 * 4096 + 4 * 16 * 32) + acts + 65536 * (1024 + 4 * 8)
    assert w["up"]["bytes"] == up_bytes == 2_520_317_952
    # the two GEMMs split the FLOPs 2 : 1
    assert w["up"]["flop"] == 2 * w["down"]["flop"]
    assert w["up"]["flop"] + w["down"]["flop"] == w["total"]["flop"]


def test_masked_and_out_of_range_ids_do_not_count():
    cfg = W.CONFIGS["tiny"]                                    # E = 8, top-2, M = 16
    ids = np.tile(np.array([[0, 1]]), (16, 1))
    ids[3] = [-1, 1]
    ids[4] = [8, 9]                                            # outside [0, E)
    w = bench.work(cfg, ids)
    assert w["Rv"] == 32 - 3 and w["U"] == 2
    assert w["total"]["flop"] == w["Rv"] * 6 * cfg.H * cfg.I
