"""Device buffers of one workload, prepared with the library's own kernels.

Raw BF16 activations and weights come from ``workloads``; they are quantised
on the GPU (moe_quantize_act_1x128 / moe_quantize_weight_128x128), optionally
requantised to UE8M0 scales (moe_requant_scales_ue8m0), interleaved
(moe_prep_weights), and the routing plan is built by moe_plan.  Nothing here
computes any step of the path itself.
"""

import torch

from . import _lib as L
import workloads as W


class DeviceProblem:
    """Quantised inputs, prepared weights, plan buffers and workspace of a workload.

    ``weights_from`` reuses the prepared weights of another problem with the
    same H, I, E, seed and weight options (a sweep over token counts).
    """

    def __init__(self, cfg: W.MoEConfig, device="cuda", chunk_experts=16, worst_case_plan=None,
                 weights_from=None):
        self.cfg = cfg
        self.device = device
        dev = torch.device(device)
        self.routing = W.make_routing(cfg)
        M, H, I, E, k, bm = cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.block_m
        N = 2 * I

        x = W.make_activations(cfg, device=dev)
        self.a = torch.empty(M, H, dtype=torch.uint8, device=dev)
        self.a_scale = torch.empty(M, H // 128, dtype=torch.float32, device=dev)
        if cfg.act_ue8m0:
            L.moe_quantize_act_1x128_ue8m0(x, self.a, self.a_scale)
        else:
            L.moe_quantize_act_1x128(x, self.a, self.a_scale)
        del x

        if weights_from is not None:
            src = weights_from
            assert (src.cfg.H, src.cfg.I, src.cfg.E, src.cfg.seed, src.cfg.ue8m0) == (H, I, E, cfg.seed, cfg.ue8m0)
            self.w13_logical, self.w13_scale, self.w2, self.w2_scale, self.w13 = (
                src.w13_logical, src.w13_scale, src.w2, src.w2_scale, src.w13)
        else:
            self._make_weights(cfg, dev, chunk_experts)
        self._make_rest(cfg, dev, worst_case_plan)

    def _make_weights(self, cfg, dev, chunk_experts):
        H, I, E = cfg.H, cfg.I, cfg.E
        N = 2 * I
        self.w13_logical = torch.empty(E, N, H, dtype=torch.uint8, device=dev)
        self.w13_scale = torch.empty(E, N // 128, H // 128, dtype=torch.float32, device=dev)
        self.w2 = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        self.w2_scale = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
        for e0 in range(0, E, chunk_experts):
            ex = list(range(e0, min(E, e0 + chunk_experts)))
            raw = W.make_weights(cfg, "w13", ex, device=dev)
            L.moe_quantize_weight_128x128(raw, self.w13_logical[e0:e0 + len(ex)], self.w13_scale[e0:e0 + len(ex)])
            raw = W.make_weights(cfg, "w2", ex, device=dev)
            L.moe_quantize_weight_128x128(raw, self.w2[e0:e0 + len(ex)], self.w2_scale[e0:e0 + len(ex)])
            del raw
        for e in self.routing.zero_scale_experts:
            self.w13_scale[e].zero_()
            self.w2_scale[e].zero_()
        if cfg.ue8m0:
            L.moe_requant_scales_ue8m0(self.w13_logical, self.w13_scale)
            L.moe_requant_scales_ue8m0(self.w2, self.w2_scale)
        self.w13 = torch.empty_like(self.w13_logical)
        L.moe_prep_weights(self.w13_logical, self.w13)

    def _make_rest(self, cfg, dev, worst_case_plan):
        M, H, I, E, k, bm = cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.block_m

        self.topk_ids = self.routing.topk_ids.to(dev)
        self.topk_weights = self.routing.topk_weights.to(dev)
        self.out_prior = W.make_out_prior(cfg, device=dev)
        self.out = self.out_prior.clone()

        cap, bcap = L.moe_plan_capacity(M, k, E, bm)
        if worst_case_plan is None:
            worst_case_plan = cfg.garbage_plan
        if worst_case_plan:  # E * (block_m - 1) padding bound, as a caller without min(E, R) would size it
            cap = -(-(M * k + E * (bm - 1)) // bm) * bm
            bcap = cap // bm
        if cfg.garbage_plan:
            self.sorted_ids = W.garbage_int32(cap, cfg.seed, device=dev)
            self.expert_ids = W.garbage_int32(bcap, cfg.seed + 1, device=dev)
        else:
            self.sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
            self.expert_ids = torch.empty(bcap, dtype=torch.int32, device=dev)
        self.ntpp = torch.zeros(1, dtype=torch.int32, device=dev)
        self.plan_ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device=dev)
        ws_bytes = L.moe_forward_workspace_size(M, H, I, E, k, bm, cap)
        self.workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        L.moe_workspace_init(self.workspace)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run_plan(self, stream=None):
        L.moe_plan(self.topk_ids, self.cfg.E, self.cfg.block_m, self.sorted_ids, self.expert_ids, self.ntpp,
                   self.plan_ws, stream)

    # how the forward applies the block scales unless a call says otherwise
    # (MOE_SCALES_UE8M0 needs power-of-two scales on both operands)
    scale_mode = L.SCALES_FP32

    def fwd_args(self, debug_q=None, debug_s=None, out=None, tile_mode=L.TILE_AUTO, scale_mode=None):
        if scale_mode is None:
            scale_mode = self.scale_mode
        args = L.make_fwd_args(self.a, self.a_scale, self.w13, self.w13_scale, self.w2, self.w2_scale,
                               self.topk_weights, self.sorted_ids, self.expert_ids, self.ntpp,
                               self.out if out is None else out, self.workspace, self.cfg.top_k, self.cfg.block_m,
                               self.cfg.routed_scale, self.status, debug_q, debug_s)
        args.tile_mode = tile_mode
        args.scale_mode = scale_mode
        return args

    def run_forward(self, args=None, stream=None):
        L.moe_fp8_block_scale_forward(self.fwd_args() if args is None else args, stream)


class W4A8Problem:
    """Device buffers of a workload for the E2M1-K32 weight x FP8 activation
    forward (include/moe_w4a8.h): activations quantised per row
    (moe_quantize_act_per_row), weights to packed E2M1 with K32 scales
    (moe_quantize_weight_k32), the plan from moe_plan."""

    def __init__(self, cfg: W.MoEConfig, device="cuda", chunk_experts=16):
        self.cfg = cfg
        dev = torch.device(device)
        self.routing = W.make_routing(cfg)
        M, H, I, E, k, bm = cfg.M, cfg.H, cfg.I, cfg.E, cfg.top_k, cfg.block_m
        N = 2 * I

        x = W.make_activations(cfg, device=dev)
        self.a = torch.empty(M, H, dtype=torch.uint8, device=dev)
        self.a_scale = torch.empty(M, dtype=torch.float32, device=dev)
        L.moe_quantize_act_per_row(x, self.a, self.a_scale)
        del x

        self.w13 = torch.empty(E, N, H // 2, dtype=torch.uint8, device=dev)
        self.w13_scale = torch.empty(E, N, H // 32, dtype=torch.float32, device=dev)
        self.w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=dev)
        self.w2_scale = torch.empty(E, H, I // 32, dtype=torch.float32, device=dev)
        for e0 in range(0, E, chunk_experts):
            ex = list(range(e0, min(E, e0 + chunk_experts)))
            e1 = e0 + len(ex)
            raw = W.make_weights(cfg, "w13", ex, device=dev)
            L.moe_quantize_weight_k32(raw, self.w13[e0:e1], self.w13_scale[e0:e1])
            raw = W.make_weights(cfg, "w2", ex, device=dev)
            L.moe_quantize_weight_k32(raw, self.w2[e0:e1], self.w2_scale[e0:e1])
            del raw
        for e in self.routing.zero_scale_experts:
            self.w13_scale[e].zero_()
            self.w2_scale[e].zero_()

        self.topk_ids = self.routing.topk_ids.to(dev)
        self.topk_weights = self.routing.topk_weights.to(dev)
        self.out_prior = W.make_out_prior(cfg, device=dev)
        self.out = self.out_prior.clone()
        cap, bcap = L.moe_plan_capacity(M, k, E, bm)
        if cfg.garbage_plan:
            self.sorted_ids = W.garbage_int32(cap, cfg.seed, device=dev)
            self.expert_ids = W.garbage_int32(bcap, cfg.seed + 1, device=dev)
        else:
            self.sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
            self.expert_ids = torch.empty(bcap, dtype=torch.int32, device=dev)
        self.ntpp = torch.zeros(1, dtype=torch.int32, device=dev)
        self.plan_ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device=dev)
        self.workspace = torch.empty(max(L.moe_w4a8_workspace_size(M, H, I, k), 256), dtype=torch.uint8,
                                     device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def run_plan(self, stream=None):
        L.moe_plan(self.topk_ids, self.cfg.E, self.cfg.block_m, self.sorted_ids, self.expert_ids, self.ntpp,
                   self.plan_ws, stream)

    def fwd_args(self, debug_q=None, debug_s=None, out=None, path=L.W4A8_AUTO):
        args = L.make_w4a8_args(self.a, self.a_scale, self.w13, self.w13_scale, self.w2, self.w2_scale,
                                self.topk_weights, self.sorted_ids, self.expert_ids, self.ntpp,
                                self.out if out is None else out, self.workspace, self.cfg.top_k,
                                self.cfg.block_m, self.cfg.routed_scale, self.status, debug_q, debug_s)
        args.path = path
        return args

    def run_forward(self, args=None, stream=None):
        L.moe_w4a8_forward(self.fwd_args() if args is None else args, stream)
