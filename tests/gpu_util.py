"""Helpers shared by the GPU parity tests: device copies of the seeded
workloads and oracle runs on the same inputs."""

import numpy as np
import torch

import workloads as WL
from oracle import quantize as Q, gemm, router, compare


def to_device(arr, dtype):
    """numpy float32 or bf16 bits (uint16) -> CUDA tensor of that dtype."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def as_f32(arr, dtype):
    return WL.bf16_bits_to_float32(arr) if dtype == "bf16" else np.asarray(arr, np.float32)


def f32_bits(v):
    return np.float32(v).view(np.uint32)


class Case:
    """One workload: host inputs, device inputs, packed device weight, oracle weight."""

    def __init__(self, w, with_oracle_w=True):
        import nvfp4_router_gate_gb300 as R
        self.w = w
        self.x = WL.make_x(w)
        self.W = WL.make_w(w)
        self.bias = WL.make_bias(w)
        self.x_dev = to_device(self.x, w.dtype)
        self.W_dev = to_device(self.W, w.dtype)
        self.bias_dev = None if self.bias is None else torch.from_numpy(self.bias).cuda()
        self.W_fp4, self.W_sf, self.w_gsa = R.nvfp4_pack_weight(self.W_dev)
        self.x32 = as_f32(self.x, w.dtype)
        if with_oracle_w:
            self.wq, self.ws, self.wg = Q.quantize(as_f32(self.W, w.dtype))

    def oracle_rows(self, rows):
        """Oracle logits/bounds for a subset of token rows (the gsa is the whole batch's)."""
        gsa = Q.global_scale(self.x32)
        xq, xs, _ = Q.quantize(self.x32[rows], gsa=gsa)
        L, B = gemm.logits(xq, xs, gsa, self.wq, self.ws, self.wg)
        return L, B

    def run(self, flags=0, k=None):
        import nvfp4_router_gate_gb300 as R
        k = k or self.w.k
        ids, wts = R.router_gate_topk(self.x_dev, self.W_fp4, self.W_sf, self.w_gsa, self.bias_dev, k,
                                      self.w.routed_scaling, self.w.raw, flags=flags)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), wts.cpu().numpy()

    def check(self, ids, wts, rows, k=None):
        k = k or self.w.k
        L, B = self.oracle_rows(rows)
        keys = router.selection_keys(L, self.bias, self.w.raw)
        res = compare.check_topk(ids[rows], wts[rows], L, B, keys, self.bias, self.w.routed_scaling,
                                 self.w.raw)
        return res
