"""ctypes binding of libmoe_fp8.so (the C ABI declared in include/moe_fp8.h).

Argument marshalling only: every function forwards device pointers, sizes
and the current torch stream to the C entry point of the same name and raises
``MoeError`` on a non-zero status.  There is no fallback: if the shared
library is missing, loading fails loudly.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_fp8.so")
LIB_DEBUG_PATH = os.path.join(_PKG, "libmoe_fp8_debug.so")  # the bounds-checking build

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_NULL", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_ALIGN", 4: "MOE_ERR_CAPACITY",
    5: "MOE_ERR_DTYPE", 6: "MOE_ERR_DEVICE", 7: "MOE_ERR_CUDA", 8: "MOE_ERR_TIMEOUT",
}
MOE_DEV_TIMEOUT = 0x1
MOE_DEV_BAD_EXPERT = 0x2
MOE_DEV_BAD_SCALE = 0x4


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class MoeFwdArgs(ctypes.Structure):
    """Mirror of ``struct moe_fwd_args``."""
    _fields_ = [
        ("a", ctypes.c_void_p),
        ("a_scale", ctypes.c_void_p),
        ("w13", ctypes.c_void_p),
        ("w13_scale", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("topk_weights", ctypes.c_void_p),
        ("sorted_token_ids", ctypes.c_void_p),
        ("expert_ids", ctypes.c_void_p),
        ("num_tokens_post_padded", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("device_status", ctypes.c_void_p),
        ("debug_q_inter", ctypes.c_void_p),
        ("debug_s_inter", ctypes.c_void_p),
        ("M", ctypes.c_int64),
        ("sorted_cap", ctypes.c_int64),
        ("blocks_cap", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_size_t),
        ("H", ctypes.c_int32),
        ("I", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("block_m", ctypes.c_int32),
        ("routed_scale", ctypes.c_float),
        ("profile_events", ctypes.POINTER(ctypes.c_void_p)),
        ("tile_mode", ctypes.c_int32),
        ("scale_mode", ctypes.c_int32),
    ]


TILE_AUTO, TILE_SINGLE, TILE_PAIR, TILE_VECTOR = 0, 1, 2, 3
W4A8_AUTO, W4A8_CUDA_CORES = 0, 1
SCALES_FP32, SCALES_UE8M0 = 0, 1


class MoeW4A8Args(ctypes.Structure):
    """Mirror of ``struct moe_w4a8_args`` (include/moe_w4a8.h)."""
    _fields_ = [
        ("a", ctypes.c_void_p),
        ("a_scale", ctypes.c_void_p),
        ("w13", ctypes.c_void_p),
        ("w13_scale", ctypes.c_void_p),
        ("w2", ctypes.c_void_p),
        ("w2_scale", ctypes.c_void_p),
        ("topk_weights", ctypes.c_void_p),
        ("sorted_token_ids", ctypes.c_void_p),
        ("expert_ids", ctypes.c_void_p),
        ("num_tokens_post_padded", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("device_status", ctypes.c_void_p),
        ("debug_q_inter", ctypes.c_void_p),
        ("debug_s_inter", ctypes.c_void_p),
        ("M", ctypes.c_int64),
        ("sorted_cap", ctypes.c_int64),
        ("blocks_cap", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_size_t),
        ("H", ctypes.c_int32),
        ("I", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("block_m", ctypes.c_int32),
        ("routed_scale", ctypes.c_float),
        ("path", ctypes.c_int32),
    ]


_libs = {}
_active = LIB_PATH

_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_plan_capacity": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]),
    "moe_plan_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int, ctypes.c_int]),
    "moe_plan": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_prep_weights": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p]),
    "moe_requant_scales_ue8m0": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "moe_route_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_void_p]),
    "moe_route_plan": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    "moe_quantize_act_1x128": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]),
    "moe_quantize_act_1x128_ue8m0": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                                    ctypes.c_void_p, ctypes.c_void_p]),
    "moe_quantize_weight_128x128": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_forward_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_int64]),
    "moe_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_fp8_block_scale_forward": (ctypes.c_int, [ctypes.POINTER(MoeFwdArgs), ctypes.c_void_p]),
    "moe_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p]),
    "moe_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "moe_fp8_block_scale_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(MoeFwdArgs), ctypes.c_void_p]),
    "moe_quantize_act_per_row": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                                ctypes.c_void_p, ctypes.c_void_p]),
    "moe_quantize_weight_k32": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_void_p, ctypes.c_void_p]),
    "moe_w4a8_workspace_size": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "moe_w4a8_forward": (ctypes.c_int, [ctypes.POINTER(MoeW4A8Args), ctypes.c_void_p]),
    "moe_debug_bounds_enabled": (ctypes.c_int, []),
    "moe_debug_bounds_selftest": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                 ctypes.c_void_p]),
    "moe_debug_bounds_read": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_char_p),
                                             ctypes.POINTER(ctypes.c_int32), ctypes.c_int]),
}


def load(path=None):
    """Load the library the wrappers call (libmoe_fp8.so unless ``use_library``
    selected another), built by ``fp8_block_scale_gb300.build.build()``."""
    path = _active if path is None else path
    lib = _libs.get(path)
    if lib is not None:
        return lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _libs[path] = lib
    return lib


class use_library:
    """Context manager: the wrappers call the library at `path` (for example
    LIB_DEBUG_PATH, the bounds-checking build) inside the block."""

    def __init__(self, path):
        self.path = path
        self.prev = None

    def __enter__(self):
        global _active
        load(self.path)
        self.prev, _active = _active, self.path
        return _libs[self.path]

    def __exit__(self, *exc):
        global _active
        _active = self.prev
        return False


def moe_debug_bounds_enabled():
    return bool(load().moe_debug_bounds_enabled())


def moe_debug_bounds_selftest(data, probe, out, stream=None):
    """Read data[probe] into out[0] through the bounds checks (int32 device tensors)."""
    _check("moe_debug_bounds_selftest", load().moe_debug_bounds_selftest(
        _ptr(data), data.numel(), int(probe), _ptr(out), _stream(stream)))


def moe_debug_bounds_read(reset=False):
    """(failures, first_file, first_line) of the active library's bounds
    checks since the last reset; waits for the device first."""
    n = ctypes.c_uint64()
    f = ctypes.c_char_p()
    line = ctypes.c_int32()
    _check("moe_debug_bounds_read", load().moe_debug_bounds_read(ctypes.byref(n), ctypes.byref(f),
                                                                 ctypes.byref(line), 1 if reset else 0))
    return n.value, (f.value.decode() if f.value else None), line.value


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != MOE_OK:
        raise MoeError(fn, status)


def moe_status_string(status):
    return load().moe_status_string(status).decode()


def moe_plan_capacity(M, top_k, E, block_m):
    cap = ctypes.c_int64()
    blocks = ctypes.c_int64()
    _check("moe_plan_capacity", load().moe_plan_capacity(M, top_k, E, block_m, ctypes.byref(cap), ctypes.byref(blocks)))
    return cap.value, blocks.value


def moe_plan_workspace_size(M, top_k, E):
    return load().moe_plan_workspace_size(M, top_k, E)


def moe_plan(topk_ids, E, block_m, sorted_token_ids, expert_ids, num_tokens_post_padded, workspace, stream=None):
    M, top_k = topk_ids.shape
    bits = {torch.int32: 32, torch.int64: 64}[topk_ids.dtype]
    _check("moe_plan", load().moe_plan(
        _ptr(topk_ids), bits, M, top_k, E, block_m, _ptr(sorted_token_ids), sorted_token_ids.numel(),
        _ptr(expert_ids), expert_ids.numel(), _ptr(num_tokens_post_padded), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def moe_prep_weights(w13, w13_interleaved, stream=None):
    E, N, H = w13.shape
    _check("moe_prep_weights", load().moe_prep_weights(_ptr(w13), _ptr(w13_interleaved), E, N, H, _stream(stream)))


def moe_requant_scales_ue8m0(w, scale, ue8m0_exp=None, stream=None):
    E, rows, cols = w.shape
    _check("moe_requant_scales_ue8m0", load().moe_requant_scales_ue8m0(
        _ptr(w), _ptr(scale), _ptr(ue8m0_exp), E, rows, cols, _stream(stream)))


LOGITS_F32, LOGITS_BF16 = 0, 1


def moe_route_topk(logits, top_k, topk_ids, topk_weights, routed_scale=1.0, renormalize=True, stream=None):
    """logits [M, E] float32 or bfloat16 -> topk_ids [M, top_k] (int32/int64), topk_weights [M, top_k] f32."""
    M, E = logits.shape
    dtype = {torch.float32: LOGITS_F32, torch.bfloat16: LOGITS_BF16}[logits.dtype]
    bits = {torch.int32: 32, torch.int64: 64}[topk_ids.dtype]
    _check("moe_route_topk", load().moe_route_topk(
        _ptr(logits), dtype, M, E, top_k, float(routed_scale), 1 if renormalize else 0, _ptr(topk_ids), bits,
        _ptr(topk_weights), _stream(stream)))


def moe_route_plan(logits, top_k, topk_ids, topk_weights, block_m, sorted_token_ids, expert_ids,
                   num_tokens_post_padded, routed_scale=1.0, renormalize=True, stream=None):
    """Router and plan in one launch (M * top_k <= 1024, E <= 1024): the
    outputs of moe_route_topk, then of moe_plan on those ids."""
    M, E = logits.shape
    dtype = {torch.float32: LOGITS_F32, torch.bfloat16: LOGITS_BF16}[logits.dtype]
    bits = {torch.int32: 32, torch.int64: 64}[topk_ids.dtype]
    _check("moe_route_plan", load().moe_route_plan(
        _ptr(logits), dtype, M, E, top_k, float(routed_scale), 1 if renormalize else 0, _ptr(topk_ids), bits,
        _ptr(topk_weights), block_m, _ptr(sorted_token_ids), sorted_token_ids.numel(), _ptr(expert_ids),
        expert_ids.numel(), _ptr(num_tokens_post_padded), _stream(stream)))


def moe_quantize_act_1x128(x_bf16, q, scale, stream=None):
    M, H = x_bf16.shape
    _check("moe_quantize_act_1x128", load().moe_quantize_act_1x128(
        _ptr(x_bf16), M, H, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_act_1x128_ue8m0(x_bf16, q, scale, stream=None):
    M, H = x_bf16.shape
    _check("moe_quantize_act_1x128_ue8m0", load().moe_quantize_act_1x128_ue8m0(
        _ptr(x_bf16), M, H, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_weight_128x128(w_bf16, q, scale, stream=None):
    E, rows, cols = w_bf16.shape
    _check("moe_quantize_weight_128x128", load().moe_quantize_weight_128x128(
        _ptr(w_bf16), E, rows, cols, _ptr(q), _ptr(scale), _stream(stream)))


def moe_forward_workspace_size(M, H, I, E, top_k, block_m, sorted_cap):
    return load().moe_forward_workspace_size(M, H, I, E, top_k, block_m, sorted_cap)


def moe_workspace_init(workspace, stream=None):
    _check("moe_workspace_init", load().moe_workspace_init(
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def make_fwd_args(a, a_scale, w13, w13_scale, w2, w2_scale, topk_weights, sorted_token_ids, expert_ids,
                  num_tokens_post_padded, out, workspace, top_k, block_m, routed_scale=1.0,
                  device_status=None, debug_q_inter=None, debug_s_inter=None):
    """Fill a ``moe_fwd_args`` from tensors (shapes give the sizes)."""
    M, H = a.shape
    E, N, _ = w13.shape
    args = MoeFwdArgs()
    args.a, args.a_scale = a.data_ptr(), a_scale.data_ptr()
    args.w13, args.w13_scale = w13.data_ptr(), w13_scale.data_ptr()
    args.w2, args.w2_scale = w2.data_ptr(), w2_scale.data_ptr()
    args.topk_weights = topk_weights.data_ptr()
    args.sorted_token_ids = sorted_token_ids.data_ptr()
    args.expert_ids = expert_ids.data_ptr()
    args.num_tokens_post_padded = num_tokens_post_padded.data_ptr()
    args.out = out.data_ptr()
    args.workspace = workspace.data_ptr()
    args.device_status = device_status.data_ptr() if device_status is not None else None
    args.debug_q_inter = debug_q_inter.data_ptr() if debug_q_inter is not None else None
    args.debug_s_inter = debug_s_inter.data_ptr() if debug_s_inter is not None else None
    args.M = M
    args.sorted_cap = sorted_token_ids.numel()
    args.blocks_cap = expert_ids.numel()
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    args.H, args.I, args.E = H, N // 2, E
    args.top_k, args.block_m = top_k, block_m
    args.routed_scale = routed_scale
    return args


PROFILE_EVENTS = 5  # before staging, after staging, after gate/up, after down, after combine


def set_profile_events(args, events):
    """Attach 5 recorded torch.cuda.Event objects (or None) to a moe_fwd_args."""
    if events is None:
        args.profile_events = None
        args._events_keepalive = None
        return
    if len(events) != PROFILE_EVENTS:
        raise ValueError(f"need {PROFILE_EVENTS} events")
    arr = (ctypes.c_void_p * PROFILE_EVENTS)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    args._events_keepalive = arr
    args.profile_events = ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p))


def moe_fp8_block_scale_forward(args, stream=None):
    _check("moe_fp8_block_scale_forward", load().moe_fp8_block_scale_forward(ctypes.byref(args), _stream(stream)))


def moe_selftest_wait_timeout(limit_us, device_status, elapsed_ns, stream=None):
    """Run the bounded-wait self-test; returns the raw status (MOE_ERR_TIMEOUT,
    8, is the expected outcome).  device_status: int32 [1], elapsed_ns:
    int64 [2] device tensors."""
    return load().moe_selftest_wait_timeout(int(limit_us), _ptr(device_status), _ptr(elapsed_ns), _stream(stream))


def moe_noalloc_scratch_bytes():
    return load().moe_noalloc_scratch_bytes()


def moe_fp8_block_scale_forward_noalloc(args, stream=None):
    """Forward without a caller workspace (static device scratch; see the header)."""
    _check("moe_fp8_block_scale_forward_noalloc",
           load().moe_fp8_block_scale_forward_noalloc(ctypes.byref(args), _stream(stream)))


# ---------------------------------------------------------------- E2M1-K32 weights x FP8 activations

def moe_quantize_act_per_row(x_bf16, q, scale, stream=None):
    M, K = x_bf16.shape
    _check("moe_quantize_act_per_row", load().moe_quantize_act_per_row(
        _ptr(x_bf16), M, K, _ptr(q), _ptr(scale), _stream(stream)))


def moe_quantize_weight_k32(w_bf16, q_packed, scale, stream=None):
    """w_bf16 [..., K] (leading dimensions folded into rows) -> q_packed [..., K/2], scale [..., K/32]."""
    K = w_bf16.shape[-1]
    _check("moe_quantize_weight_k32", load().moe_quantize_weight_k32(
        _ptr(w_bf16), w_bf16.numel() // K, K, _ptr(q_packed), _ptr(scale), _stream(stream)))


def moe_w4a8_workspace_size(M, H, I, top_k):
    return load().moe_w4a8_workspace_size(M, H, I, top_k)


def make_w4a8_args(a, a_scale, w13, w13_scale, w2, w2_scale, topk_weights, sorted_token_ids, expert_ids,
                   num_tokens_post_padded, out, workspace, top_k, block_m, routed_scale=1.0,
                   device_status=None, debug_q_inter=None, debug_s_inter=None):
    """Fill a ``moe_w4a8_args`` from tensors; w13 is [E, 2I, H/2] packed codes."""
    M, H = a.shape
    E, N, _ = w13.shape
    args = MoeW4A8Args()
    args.a, args.a_scale = a.data_ptr(), a_scale.data_ptr()
    args.w13, args.w13_scale = w13.data_ptr(), w13_scale.data_ptr()
    args.w2, args.w2_scale = w2.data_ptr(), w2_scale.data_ptr()
    args.topk_weights = topk_weights.data_ptr()
    args.sorted_token_ids = sorted_token_ids.data_ptr()
    args.expert_ids = expert_ids.data_ptr()
    args.num_tokens_post_padded = num_tokens_post_padded.data_ptr()
    args.out = out.data_ptr()
    args.workspace = workspace.data_ptr()
    args.device_status = device_status.data_ptr() if device_status is not None else None
    args.debug_q_inter = debug_q_inter.data_ptr() if debug_q_inter is not None else None
    args.debug_s_inter = debug_s_inter.data_ptr() if debug_s_inter is not None else None
    args.M = M
    args.sorted_cap = sorted_token_ids.numel()
    args.blocks_cap = expert_ids.numel()
    args.workspace_bytes = workspace.numel() * workspace.element_size()
    args.H, args.I, args.E = H, N // 2, E
    args.top_k, args.block_m = top_k, block_m
    args.routed_scale = routed_scale
    return args


def moe_w4a8_forward(args, stream=None):
    _check("moe_w4a8_forward", load().moe_w4a8_forward(ctypes.byref(args), _stream(stream)))
