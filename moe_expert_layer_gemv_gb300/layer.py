"""A device-resident MoE layer: weights uploaded once, a workspace, and calls
into the C ABI (moe_expert_layer_gemv_gb300.abi).  Marshalling only."""
import torch

from . import abi


def _dev(t, device):
    return None if t is None else t.to(device, non_blocking=False).contiguous()


class MoeLayer:
    """Holds one layer's device weights (from inputs.make_inputs) and workspace."""

    def __init__(self, inp: dict, device="cuda", flags=0):
        s = inp["shape"]
        self.shape = s
        self.device = torch.device(device)
        self.dims = abi.dims_of(s, flags)
        self.router_w = _dev(inp["router_w"], device)
        self.gate_up = _dev(inp["gate_up"], device)
        self.down = _dev(inp["down"], device)
        self.gate_up_scales = _dev(inp["gate_up_scales"], device)
        self.down_scales = _dev(inp["down_scales"], device)
        self.experts = abi.expert_weights(self.gate_up, self.down, self.gate_up_scales,
                                          self.down_scales)
        self.shared = None
        if s.Is > 0:
            self.s_gate_up = _dev(inp["shared_gate_up"], device)
            self.s_down = _dev(inp["shared_down"], device)
            self.w_sg = _dev(inp["w_sg"], device)
            self.shared = abi.shared_weights(self.s_gate_up, self.s_down, self.w_sg)
        self.ws = abi.alloc_workspace(self.dims, device)

    def new_out(self):
        return torch.empty((self.shape.T, self.shape.d), dtype=torch.bfloat16, device=self.device)

    def forward(self, x, out=None, topk_ids=None, topk_weights=None, stream=None):
        out = self.new_out() if out is None else out
        abi.moe_layer_forward(self.dims, x, self.router_w, self.experts, self.shared, out,
                              topk_ids, topk_weights, self.ws, stream)
        return out

    def forward_timed(self, x, out, events, topk_ids=None, topk_weights=None, stream=None):
        abi.moe_layer_forward_timed(self.dims, x, self.router_w, self.experts, self.shared, out,
                                    topk_ids, topk_weights, self.ws, events, stream)
        return out

    def device_status(self) -> int:
        return abi.moe_read_device_status(self.ws)

    def layout(self) -> dict:
        """The routing and aligned layout the last forward left in the
        workspace (moe_workspace_views), copied to host numpy arrays."""
        s = self.shape
        v = abi.moe_workspace_views(self.dims)

        def take(name, n, dtype=torch.int32):
            off = v[name]
            return self.ws[off:off + 4 * n].view(dtype).cpu().numpy()

        npp = int(take("num_post_pad", 1)[0])
        return {"topk_ids": take("topk_ids", s.T * s.k).reshape(s.T, s.k),
                "topk_weights": take("topk_weights", s.T * s.k, torch.float32).reshape(s.T, s.k),
                "num_post_pad": npp, "sorted_ids": take("sorted_ids", npp),
                "block_expert_ids": take("block_expert_ids", npp // s.block),
                "expert_offsets": take("expert_offsets", s.E + 1)}
