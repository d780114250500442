"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on seeded synthetic inputs and fetch every intermediate; compare with
the oracle under the layer's tolerance."""
import numpy as np
import torch

import bit_moe_expert_histogram_gb300 as m
import synth


def d16(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def h16(t):
    return t.cpu().numpy().view(np.uint16)


def f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def close(g, r, what="", mre_bound=2e-3):
    """max|g-r| <= 1e-2*max|r| + 1e-3 and sum|g-r|/sum|r| <= mre_bound
    (2e-3: the layer's tolerance)."""
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    err = np.abs(g - r)
    mx = err.max() if err.size else 0.0
    bound = 1e-2 * np.abs(r).max() + 1e-3
    mre = err.sum() / max(np.abs(r).sum(), 1e-300)
    assert mx <= bound, "%s: max err %.4g > %.4g" % (what, mx, bound)
    assert mre <= mre_bound, "%s: mean rel err %.4g > %.3g" % (what, mre, mre_bound)
    return mx, mre


class Case:
    """One layer's inputs on the device plus caller-owned buffers."""

    def __init__(self, L, T, shape, tile_rows=128, dev="cuda"):
        self.L, self.T, self.S = L, T, shape
        self.dev = torch.device(dev)
        self.shape = m.make_shape(T, shape.H, shape.E, shape.K, shape.I, shape.n_shared, tile_rows)
        self.x = d16(L.x, self.dev)
        self.wr = d16(L.w_router, self.dev)
        self.bias = None if L.router_bias is None else torch.from_numpy(L.router_bias).to(self.dev)
        self.ex = m.ExpertWeights.from_numpy(L.q_gate_up, L.s_gate_up, L.b_gate_up, L.q_down,
                                             L.s_down, L.b_down, self.dev)
        self.sh = None
        if shape.n_shared:
            self.sh = m.ExpertWeights.from_numpy(L.sh_q_gate_up, L.sh_s_gate_up, L.sh_b_gate_up,
                                                 L.sh_q_down, L.sh_s_down, L.sh_b_down, self.dev)
        self.ws = m.alloc_workspace(self.shape, self.dev)
        K, H = shape.K, shape.H
        self.R = T * K
        self.Srows = self.R + T * shape.n_shared
        self.ids = torch.full((T, K), -7, dtype=torch.int32, device=self.dev)
        self.w = torch.zeros((T, K), dtype=torch.float32, device=self.dev)
        self.plan = m.PlanBuffers(self.shape, self.dev)
        self.y_slots = torch.zeros((self.Srows, H), dtype=torch.int16, device=self.dev)
        self.y = torch.zeros((T, H), dtype=torch.int16, device=self.dev)
        self.x_next = torch.zeros((T, H), dtype=torch.int16, device=self.dev)

    def set_x(self, x_bits):
        self.x.copy_(d16(x_bits, self.dev))

    def run_calls(self, x_next=False):
        m.moe_route(self.shape, self.x, self.wr, self.bias, self.ids, self.w, self.ws)
        m.moe_plan(self.shape, self.ids, self.plan, self.ws)
        m.moe_expert_ffn_w4(self.shape, self.x, self.ex, self.sh, self.plan, self.y_slots, self.ws)
        m.moe_combine(self.shape, self.y_slots, self.plan.row_pos, self.w, self.y,
                      self.x_next if x_next else None)
        st = m.moe_query_device_status(self.ws)
        assert st == 0, "device status %d" % st

    def run_layer(self, x_next=False):
        m.moe_layer_w4(self.shape, self.x, self.wr, self.bias, self.ex, self.sh, self.y, self.ws,
                       x_next=self.x_next if x_next else None, topk_ids=self.ids, topk_w=self.w)
        st = m.moe_query_device_status(self.ws)
        assert st == 0, "device status %d" % st

    def plan_np(self):
        p = self.plan
        nb = int(p.num_blocks.item())
        return dict(counts=p.counts.cpu().numpy(), offsets=p.offsets.cpu().numpy(),
                    sorted_rows=p.sorted_rows.cpu().numpy(), row_pos=p.row_pos.cpu().numpy(),
                    block_map=p.block_map.cpu().numpy().reshape(-1, 3)[:nb], num_blocks=nb)
