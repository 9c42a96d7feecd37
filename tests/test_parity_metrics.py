"""Pins for the parity metrics every GPU test relies on (CPU only): a mistake
here would hide a real difference between the GPU path and the oracle.
Each check is a hand-worked case."""

import numpy as np

from oracle.inputs import bf16_ulps, code_diffs, out_metrics


def test_code_diffs_counts_and_adjacency():
    # identical codes, and +0 against -0
    assert code_diffs(np.array([0x38, 0x00]), np.array([0x38, 0x80])) == (0, 0)
    # one step inside a binade (1.0 -> 1.125) and across one (1.875 -> 2.0)
    assert code_diffs(np.array([0x38]), np.array([0x39])) == (1, 0)
    assert code_diffs(np.array([0x3F]), np.array([0x40])) == (1, 0)
    # the top of the range (416 -> 448) and the bottom (0 -> 2**-9, -0 -> 2**-9)
    assert code_diffs(np.array([0x7D]), np.array([0x7E])) == (1, 0)
    assert code_diffs(np.array([0x00]), np.array([0x01])) == (1, 0)
    assert code_diffs(np.array([0x80]), np.array([0x01])) == (1, 0)
    # two steps apart, a sign flip, and the two smallest values of opposite sign
    assert code_diffs(np.array([0x38]), np.array([0x3A])) == (1, 1)
    assert code_diffs(np.array([0x38]), np.array([0xB8])) == (1, 1)
    assert code_diffs(np.array([0x81]), np.array([0x01])) == (1, 1)
    # counts add up over an array
    got = np.array([0x38, 0x39, 0x3A, 0xB8, 0x00])
    ref = np.array([0x38, 0x38, 0x38, 0x38, 0x80])
    assert code_diffs(got, ref) == (3, 2)


def test_out_metrics_hand_example():
    ref = np.array([[3.0, -4.0], [0.0, 0.0]])
    got = ref + np.array([[0.0, 0.1], [0.0, 0.0]])
    prior = np.array([[3.0, -3.0], [0.0, 0.0]])
    m = out_metrics(got, ref, prior)
    assert np.isclose(m["rel_l2"], 0.1 / 5.0)            # |d| / |ref| = 0.1 / 5
    assert np.isclose(m["max_rel"], 0.1 / 4.0)           # max|d| / max|ref|
    assert np.isclose(m["rel_l2_delta"], 0.1 / 1.0)      # |d| / |ref - prior| = 0.1 / 1
    assert out_metrics(ref, ref)["rel_l2"] == 0.0


def test_bf16_ulps_steps():
    def bf(bits):
        return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)
    one, next_up = bf([0x3F80]), bf([0x3F81])              # 1.0 and 1.0078125
    assert bf16_ulps(one, next_up)[0] == 1
    assert bf16_ulps(bf([0x3F7F]), one)[0] == 1            # across a binade
    assert bf16_ulps(bf([0x0000]), bf([0x8000]))[0] == 0   # +0 and -0
    assert bf16_ulps(bf([0x0001]), bf([0x8001]))[0] == 2   # smallest values of opposite sign
    assert bf16_ulps(bf([0xBF80]), bf([0xBF81]))[0] == 1   # -1.0 and the next value below it
    assert bf16_ulps(bf([0xBF80]), one)[0] == 2 * 0x3F80   # -1 to 1: every value between
    a = bf([0x3F80, 0x4000, 0xC000])
    assert (bf16_ulps(a, a) == 0).all()
