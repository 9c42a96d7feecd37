"""Planted-mistake check of the oracle's CPU pins (not collected by pytest).

Each entry below is a plausible mistake in the oracle or in the parity
metrics the GPU tests use: a dropped term, a wrong sign, index or axis, a
swapped operand, a wrong constant or tie rule.
The script copies ``oracle/`` and ``tests/`` into a temporary directory,
plants one mistake at a time in the copy and runs the oracle pin tests
there; every mistake must make at least one pin fail.  The repository is
never modified.

    python tests/mutants.py            # all mistakes
    python tests/mutants.py -k ue8m0   # those whose name contains "ue8m0"
    python tests/mutants.py -j 8       # eight at a time (default: up to 4)

An entry whose anchor text no longer occurs in the oracle is reported as
stale (the oracle changed: update the entry).
"""

import argparse
import os
import queue
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_TESTS = ["tests/test_parity_metrics.py", "tests/test_oracle_numerics.py", "tests/test_oracle_moe.py",
             "tests/test_oracle_router.py", "tests/test_oracle_w4a8.py"]

# (file, name, text in the oracle, the mistaken text)
MUTANTS = [
    ('oracle/moe.py', 'routes_slot_lost',
     'groups[e][1].append(j)',
     'groups[e][1].append(0)'),
    ('oracle/moe.py', 'act_groups_transposed',
     'codes, scale = _quantize_groups(x.reshape(M, H // GROUP, GROUP))',
     'codes, scale = _quantize_groups(x.reshape(M, GROUP, H // GROUP).transpose(0, 2, 1))'),
    ('oracle/numerics.py', 'e4m3_negative_zero_lost',
     'neg = np.signbit(x)',
     'neg = x < 0'),
    ('oracle/moe.py', 'combine_bf16_route_unrounded',
     '                y = bf16_round(y)',
     '                y = y'),
    ('oracle/moe.py', 'combine_bf16_stepwise_unrounded',
     '                acc = bf16_round(acc)',
     '                acc = acc'),
    ('oracle/moe.py', 'act_ue8m0_not_rounded',
     'scale = ue8m0_round_up(f32(np.max(np.abs(g), axis=-1) / np.float32(E4M3_MAX)))',
     'scale = f32(np.max(np.abs(g), axis=-1) / np.float32(E4M3_MAX))'),
    ('oracle/numerics.py', 'e4m3_nan_code',
     'return np.where(nan, 0x7F, code).astype(np.uint8)',
     'return np.where(nan, 0x7E, code).astype(np.uint8)'),
    ('oracle/numerics.py', 'e4m3_decode_no_nan',
     'return np.where((e == 15) & (m == 7), np.nan, val)',
     'return val'),
    ('oracle/numerics.py', 'bf16_no_overflow',
     'r = np.where(r > bf16_max, np.inf, r)',
     'r = np.minimum(r, bf16_max)'),
    ('oracle/w4a8.py', 'e2m1_subnormal_scale',
     'mag = np.ldexp(np.where(e == 0, m, 2 + m).astype(np.float64), np.where(e == 0, -1, e - 2))',
     'mag = np.ldexp(np.where(e == 0, m, 2 + m).astype(np.float64), np.where(e == 0, 0, e - 2))'),
    ('oracle/moe.py', 'fp64_twin_routed_scale',
     'out[t] += y * float(topk_w[t, j]) * float(routed_scale)',
     'out[t] += y * float(topk_w[t, j])'),
    ('oracle/moe.py', 'fp64_twin_silu_sign',
     'h = g / (1.0 + np.exp(-g)) * u',
     'h = g / (1.0 + np.exp(g)) * u'),
    ('oracle/w4a8.py', 'w4_fp64_twin_route_weight',
     'out[t] += y * float(topk_w[t, j]) * float(routed_scale)',
     'out[t] += y * float(routed_scale)'),
    ('oracle/inputs.py', 'code_diffs_two_steps',
     'adjacent = same_sign & (np.abs(gi - ri) <= 1)',
     'adjacent = same_sign & (np.abs(gi - ri) <= 2)'),
    ('oracle/inputs.py', 'code_diffs_sign_ignored',
     'same_sign = (np.sign(g[diff]) == np.sign(r[diff])) | (g[diff] == 0) | (r[diff] == 0)',
     'same_sign = np.ones(int(diff.sum()), dtype=bool)'),
    ('oracle/inputs.py', 'out_metrics_max_over_norm',
     'mx = np.abs(d).max() / max(np.abs(ref).max(), 1e-30)',
     'mx = np.abs(d).max() / max(np.linalg.norm(ref), 1e-30)'),
    ('oracle/inputs.py', 'bf16_ulps_sign_order',
     'return np.where(bits & 0x8000, 0x8000 - bits, bits)',
     'return np.where(bits & 0x8000, bits - 0x8000, bits)'),
    ('oracle/moe.py', 'act_scale_240',
     'scale = f32(amax / np.float32(E4M3_MAX))',
     'scale = f32(amax / np.float32(240.0))'),
    ('oracle/moe.py', 'act_mul_not_div',
     'q = f32(x / safe[..., None])',
     'q = f32(x * safe[..., None])'),
    ('oracle/moe.py', 'act_no_zero_branch',
     'codes = np.where((scale > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)\n    return codes, scale',
     'return codes, scale'),
    ('oracle/moe.py', 'weight_block_transpose',
     'blocks = w.reshape(E, R // GROUP, GROUP, C // GROUP, GROUP).transpose(0, 1, 3, 2, 4)',
     'blocks = w.reshape(E, R // GROUP, GROUP, C // GROUP, GROUP).transpose(0, 1, 3, 4, 2)'),
    ('oracle/moe.py', 'cap_min_dropped',
     'cap = R + min(E, R) * (block_m - 1)',
     'cap = R + E * (block_m - 1)'),
    ('oracle/moe.py', 'plan_sentinel_R-1',
     'seg = np.full(nblk * block_m, R, dtype=np.int64)',
     'seg = np.full(nblk * block_m, R - 1, dtype=np.int64)'),
    ('oracle/moe.py', 'plan_descending',
     'seg[: routes.size] = routes',
     'seg[: routes.size] = routes[::-1]'),
    ('oracle/moe.py', 'plan_extra_block',
     'nblk = -(-routes.size // block_m)',
     'nblk = routes.size // block_m + 1'),
    ('oracle/moe.py', 'interleave_swap',
     'out[:, 16 * q: 16 * q + 8] = w13[:, 8 * q: 8 * q + 8]',
     'out[:, 16 * q: 16 * q + 8] = w13[:, I + 8 * q: I + 8 * q + 8]'),
    ('oracle/moe.py', 'ue8m0_floor',
     'p2 = np.where(f == 0.5, s, np.exp2(ex.astype(np.float64)))',
     'p2 = np.where(f == 0.5, s, np.exp2(ex.astype(np.float64) - 1))'),
    ('oracle/moe.py', 'ue8m0_ratio_inverted',
     'ratio = f32(safe_old / safe_new)',
     'ratio = f32(safe_new / safe_old)'),
    ('oracle/moe.py', 'ue8m0_exp_bias',
     'exp_byte = np.clip(ex - 1 + 127, 0, 254)',
     'exp_byte = np.clip(ex + 127, 0, 254)'),
    ('oracle/moe.py', 'silu_sign',
     'return f32(g64 / (1.0 + np.exp(-g64)))',
     'return f32(g64 / (1.0 + np.exp(g64)))'),
    ('oracle/moe.py', 'slice_dots_transposed',
     'out[:, :, kb] = f32(x[:, sl] @ w[:, sl].T)',
     'out[:, :, kb] = f32(x[:, sl] @ w[:, sl][::-1].T)'),
    ('oracle/moe.py', 'promote_scale_index',
     'sc = f32(a_s[:, kb][:, None] * w_s_rows[:, kb][None, :])',
     'sc = f32(a_s[:, kb][:, None] * w_s_rows[:, 0][None, :])'),
    ('oracle/moe.py', 'promote_act_scale_dropped',
     'sc = f32(a_s[:, kb][:, None] * w_s_rows[:, kb][None, :])',
     'sc = f32(w_s_rows[:, kb][None, :] + 0 * a_s[:, kb][:, None])'),
    ('oracle/moe.py', 'gemm1_scale_axis',
     'w_rows = np.repeat(f32(w13s_e), GROUP, axis=0)  # block scale per output row',
     'w_rows = np.repeat(f32(w13s_e), GROUP, axis=0)[::-1]'),
    ('oracle/moe.py', 'swiglu_swap',
     '    return f32(silu_f32(g) * u)',
     '    return f32(silu_f32(u) * g)'),
    ('oracle/moe.py', 'gemm2_scale_axis',
     '    w_rows = np.repeat(f32(w2s_e), GROUP, axis=0)\n    return promote(dots, f32(si), w_rows)',
     '    w_rows = np.repeat(f32(w2s_e), GROUP, axis=0)[::-1]\n    return promote(dots, f32(si), w_rows)'),
    ('oracle/moe.py', 'route_weight_dropped',
     '        wr = f32(f32(np.asarray(topk_w)[ts, js]) * rs)',
     '        wr = f32(np.ones(len(ts), np.float32) * rs)'),
    ('oracle/moe.py', 'routed_scale_dropped',
     '        wr = f32(f32(np.asarray(topk_w)[ts, js]) * rs)',
     '        wr = f32(f32(np.asarray(topk_w)[ts, js]))'),
    ('oracle/moe.py', 'prior_dropped',
     '        acc = bf16_round(prior[t]) if combine == "bf16_stepwise" else prior[t].copy()',
     '        acc = np.zeros_like(prior[t])'),
    ('oracle/moe.py', 'masked_not_skipped',
     '            if 0 <= e < E:\n                groups.setdefault(e, ([], []))',
     '            if True:\n                e = e % E\n                groups.setdefault(e, ([], []))'),
    ('oracle/numerics.py', 'e4m3_ties_away',
     'r = np.round(np.ldexp(a, 3 - E)).astype(np.int32)',
     'r = np.floor(np.ldexp(a, 3 - E) + 0.5).astype(np.int32)'),
    ('oracle/numerics.py', 'e4m3_subnormal_-7',
     'E = np.maximum(ex - 1, -6)',
     'E = np.maximum(ex - 1, -7)'),
    ('oracle/numerics.py', 'e4m3_no_sat',
     'a = np.minimum(a, E4M3_MAX)',
     'a = a'),
    ('oracle/numerics.py', 'e4m3_decode_bias',
     'np.where(e == 0, -9, e - 10)',
     'np.where(e == 0, -9, e - 11)'),
    ('oracle/numerics.py', 'bf16_truncate',
     'r = np.round(a / spacing) * spacing',
     'r = np.floor(a / spacing) * spacing'),
    ('oracle/w4a8.py', 'ties_away',
     'r = np.round(np.ldexp(a, 1 - E)).astype(np.int32)',
     'r = np.floor(np.ldexp(a, 1 - E) + 0.5).astype(np.int32)'),
    ('oracle/w4a8.py', 'bias2',
     'np.where(e == 0, -1, e - 2))',
     'np.where(e == 0, -1, e - 3))'),
    ('oracle/w4a8.py', 'no_sat',
     'a = np.minimum(np.abs(x), E2M1_MAX)',
     'a = np.abs(x)'),
    ('oracle/w4a8.py', 'nibble_swap',
     'return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)',
     'return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)'),
    ('oracle/w4a8.py', 'wmax4',
     'scale = f32(np.max(np.abs(g), axis=-1) / np.float32(E2M1_MAX))',
     'scale = f32(np.max(np.abs(g), axis=-1) / np.float32(4.0))'),
    ('oracle/w4a8.py', 'ws_index',
     'acc = f32(acc + f32(dots[:, :, kb] * ws[None, :, kb]))',
     'acc = f32(acc + f32(dots[:, :, kb] * ws[None, :, (kb + 1) % dots.shape[2]]))'),
    ('oracle/w4a8.py', 'no_xs',
     'return f32(acc * f32(xs)[:, None])',
     'return f32(acc)'),
    ('oracle/w4a8.py', 'act_448_to_240',
     'scale = f32(np.max(np.abs(x), axis=-1) / np.float32(E4M3_MAX))',
     'scale = f32(np.max(np.abs(x), axis=-1) / np.float32(240.0))'),
    ('oracle/w4a8.py', 'k16',
     'K32 = 32 ',
     'K32 = 16 '),
    ('oracle/w4a8.py', 'drop_route_w',
     'y = f32(y * wr[:, None])',
     'y = f32(y)'),
    ('oracle/w4a8.py', 'up_gate_swap',
     'h = swiglu(acc, I)',
     'h = swiglu(np.concatenate([acc[:, I:], acc[:, :I]], axis=1), I)'),
    ('oracle/w4a8.py', 'no_requant',
     'qi, si = quantize_act_per_row(h)',
     'qi, si = quantize_act_per_row(h); si = f32(si * 1.01)'),
    ('oracle/w4a8.py', 'w4_act_no_zero',
     'codes = np.where((scale > 0)[:, None], codes, np.uint8(0)).astype(np.uint8)\n    return codes, scale',
     'return codes, scale'),
    ('oracle/w4a8.py', 'w4_weight_no_zero',
     'codes = np.where((scale > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)\n    return codes.reshape(w.shape), scale',
     'return codes.reshape(w.shape), scale'),
    ('oracle/router.py', 'ties_descending_index',
     'order = np.lexsort((idx, -l[t]))',
     'order = np.lexsort((-idx, -l[t]))'),
    ('oracle/router.py', 'ascending_logits',
     'order = np.lexsort((idx, -l[t]))',
     'order = np.lexsort((idx, l[t]))'),
    ('oracle/router.py', 'renorm_flag_inverted',
     'den = num.sum(axis=1, keepdims=True) if renormalize else np.exp(l - m).sum(axis=1, keepdims=True)',
     'den = num.sum(axis=1, keepdims=True) if not renormalize else np.exp(l - m).sum(axis=1, keepdims=True)'),
    ('oracle/router.py', 'routed_scale_dropped',
     'return ids, num / den * routed_scale',
     'return ids, num / den'),
    ('oracle/router.py', 'no_max_shift',
     'num = np.exp(sel - m)',
     'num = np.exp(sel)'),
    ('oracle/router.py', 'off_by_one_k',
     'ids[t] = order[:top_k]',
     'ids[t] = order[1:top_k + 1] if top_k < E else order[:top_k]'),
]


def _run_one(copy, path, good, bad, env):
    """Plant one mistake in the given copy, run the pins there, restore."""
    target = os.path.join(copy, path)
    with open(target) as f:
        original = f.read()
    if good not in original:
        return None, f"anchor not found in {path}"
    with open(target, "w") as f:
        f.write(original.replace(good, bad, 1))
    try:
        r = subprocess.run([sys.executable, "-m", "pytest", *PIN_TESTS, "-q", "-x", "-p", "no:cacheprovider"],
                           cwd=copy, env=dict(env, PYTHONPATH=os.pathsep.join([copy, ROOT])),
                           capture_output=True, text=True)
    finally:
        with open(target, "w") as f:
            f.write(original)
    return r.returncode != 0, (r.stdout.strip().splitlines() or [""])[-1]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("-k", default="", help="only mistakes whose name contains this")
    ap.add_argument("-j", type=int, default=max(1, min(4, (os.cpu_count() or 2) // 2)),
                    help="mistakes checked at once, each in its own copy")
    args = ap.parse_args()
    todo = [m for m in MUTANTS if args.k in m[1]]
    tmp = tempfile.mkdtemp(prefix="oracle_mutants_")
    try:
        copies = queue.Queue()
        for i in range(args.j):
            copy = os.path.join(tmp, str(i))
            for d in ("oracle", "tests"):
                shutil.copytree(os.path.join(ROOT, d), os.path.join(copy, d),
                                ignore=shutil.ignore_patterns("__pycache__"))
            copies.put(copy)
        env = dict(os.environ)

        def check(m):
            path, name, good, bad = m
            copy = copies.get()
            try:
                return name, _run_one(copy, path, good, bad, env)
            finally:
                copies.put(copy)

        caught = missed = stale = 0
        with ThreadPoolExecutor(max_workers=args.j) as pool:
            for name, (ok, tail) in pool.map(check, todo):
                if ok is None:
                    stale += 1
                    print(f"{name:28s} STALE ({tail})", flush=True)
                    continue
                caught += ok
                missed += not ok
                print(f"{name:28s} {'caught' if ok else 'MISSED'}  {tail}", flush=True)
        print(f"{caught} caught, {missed} missed, {stale} stale")
        sys.exit(1 if missed or stale else 0)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


if __name__ == "__main__":
    main()
