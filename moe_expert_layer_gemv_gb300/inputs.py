"""Seeded synthetic inputs for the MoE expert layer.

This module holds no arithmetic of the method: it only draws random tensors of
the workloads' shapes and value distributions, so that the CUDA path and the
CPU oracle can be fed the same bytes.  Everything is drawn on the CPU from a
``torch.Generator`` seeded with ``manual_seed(seed)``, as fp32 normals scaled and
then cast to bf16 (round-to-nearest-even).  Draw order is fixed:
x, router_w, gate_up, down, w_sg, shared gate_up, shared down.

Workloads (the pages measure whole-model serving on private corpora and eval
suites; none is used here -- these synthetic tensors stand in for them):

* ``tiny``           T=4,    d=256,  E=8,   k=2,  I=128, no shared expert
* ``verify_t8``      T=8,    d=2048, E=256, k=8,  I=512, shared I=512
  (one target + seven draft positions: the block-length-eight DFlash profile of
  "Qwen3.6-35B-A3B for NInfer", CLI section)
* ``verify_t64``     T=64, same shapes (8 concurrent streams x 8 verify positions)
* ``verify_t64_skew``  as above, router rows of 16 hot experts scaled x4
* ``prefill_t4096``  T=4096, same shapes, 128-row align blocks
* ``int4_t32``       T=32, d=2048, E=512, k=10, I=512, shared I=1024, routed
  experts as symmetric int4 in groups of 32 along the reduction dim with one
  bf16 scale per group (512 routed experts, top-10, plus a shared expert:
  "veloGB10", The model; W4A16 routed experts: "Qwen3.8 Flash-Next - GB10
  UltraFast", How it works)

Two more routed-weight formats are drawn for the oracle's FP8 / NVFP4 paths
(the "NVFP4/FP8 families" of "veloGB10", README), by ``fmt`` on any shape:

* ``fp8``    E4M3 codes uint8 [E,2I,d] / [E,d,I]: normals of std
  FP8_VALUE_STD clamped to the format's +-448 and rounded by torch's
  float8_e4m3fn cast (never NaN), with |N(0, FP8_SCALE_STD)| bf16 scales per
  group of ``group`` along the reduction dim.
* ``nvfp4``  E2M1 codes, two per byte (even element in the low nibble), each
  nibble uniform over the 16 codes; E4M3 block scales per 16 elements drawn
  as uniform [1, 4) rounded by the float8_e4m3fn cast; one fp32 scale per
  expert matrix, 2^-8 times a uniform [0.5, 1) draw rounded to bf16 precision.
"""
from dataclasses import dataclass, field, replace

import torch

WEIGHT_STD = 0.02
INT4_SCALE_STD = 0.003
FP8_VALUE_STD = 64.0
FP8_SCALE_STD = 0.0003
E4M3_MAX = 448.0
SKEW_HOT = 16
SKEW_FACTOR = 4.0


@dataclass(frozen=True)
class LayerShape:
    T: int
    d: int
    E: int
    k: int
    I: int
    Is: int = 0                 # shared-expert intermediate; 0 = none
    renormalize: bool = True
    block: int = 16             # moe_align_block_size block B
    fmt: str = "bf16"           # "bf16" | "int4" | "fp8" | "nvfp4"
    group: int = 32             # scale group length along the reduction dim (nvfp4: 16)
    skew: bool = False
    name: str = field(default="", compare=False)

    @property
    def slots(self) -> int:
        return self.T * self.k


WORKLOADS = {
    "tiny": LayerShape(T=4, d=256, E=8, k=2, I=128, Is=0, block=16, name="tiny"),
    "verify_t8": LayerShape(T=8, d=2048, E=256, k=8, I=512, Is=512, block=16, name="verify_t8"),
    "verify_t64": LayerShape(T=64, d=2048, E=256, k=8, I=512, Is=512, block=16, name="verify_t64"),
    "verify_t64_skew": LayerShape(T=64, d=2048, E=256, k=8, I=512, Is=512, block=16, skew=True,
                                  name="verify_t64_skew"),
    "prefill_t4096": LayerShape(T=4096, d=2048, E=256, k=8, I=512, Is=512, block=128,
                                name="prefill_t4096"),
    "int4_t32": LayerShape(T=32, d=2048, E=512, k=10, I=512, Is=1024, block=16, fmt="int4",
                           group=32, name="int4_t32"),
}


def shape(name: str, **over) -> LayerShape:
    s = WORKLOADS[name]
    return replace(s, **over) if over else s


def _normal_bf16(g, size, std):
    return (torch.randn(size, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def _int4_pack(q: torch.Tensor) -> torch.Tensor:
    """Signed codes in [-8, 7] along the last dim -> uint8, two per byte,
    even element in the low nibble, stored offset-binary (code + 8)."""
    u = (q + 8).to(torch.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


def _int4_draw(g, rows_shape, cols, group):
    q = torch.randint(-8, 8, tuple(rows_shape) + (cols,), generator=g, dtype=torch.int16)
    scales = (torch.randn(tuple(rows_shape) + (cols // group,), generator=g,
                          dtype=torch.float32).abs() * INT4_SCALE_STD).to(torch.bfloat16)
    return _int4_pack(q), scales


def _fp8_draw(g, rows_shape, cols, group):
    v = torch.randn(tuple(rows_shape) + (cols,), generator=g, dtype=torch.float32) * FP8_VALUE_STD
    codes = v.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)
    scales = (torch.randn(tuple(rows_shape) + (cols // group,), generator=g,
                          dtype=torch.float32).abs() * FP8_SCALE_STD).to(torch.bfloat16)
    return codes.contiguous(), scales


def _nvfp4_draw(g, rows_shape, cols, group, n_experts):
    nib = torch.randint(0, 16, tuple(rows_shape) + (cols,), generator=g, dtype=torch.int16)
    codes = (nib[..., 0::2] | (nib[..., 1::2] << 4)).to(torch.uint8).contiguous()
    bs = 1.0 + 3.0 * torch.rand(tuple(rows_shape) + (cols // group,), generator=g,
                                dtype=torch.float32)
    scales = bs.to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    glob = ((0.5 + 0.5 * torch.rand((n_experts,), generator=g, dtype=torch.float32))
            .to(torch.bfloat16).to(torch.float32) * 2.0 ** -8)
    return codes, scales, glob


def make_inputs(s: LayerShape, seed: int = 0) -> dict:
    """Draw one layer's inputs on the CPU.  Returns torch CPU tensors:
    x bf16[T,d], router_w bf16[E,d], gate_up / down (bf16 [E,2I,d] / [E,d,I], or
    int4 codes uint8 [E,2I,d/2] / [E,d,I/2] with bf16 scales [E,2I,d/g] /
    [E,d,I/g], or fp8 codes uint8 [E,2I,d] / [E,d,I] with bf16 scales, or
    nvfp4 codes uint8 [E,2I,d/2] / [E,d,I/2] with E4M3 scales uint8 [E,2I,d/g]
    / [E,d,I/g] and fp32 gate_up_global / down_global [E]), and when Is > 0:
    w_sg bf16[d], shared_gate_up bf16[2Is,d], shared_down bf16[d,Is]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {"shape": s, "seed": seed}
    out["x"] = torch.randn((s.T, s.d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    wr = torch.randn((s.E, s.d), generator=g, dtype=torch.float32) * WEIGHT_STD
    if s.skew:
        gh = torch.Generator(device="cpu")
        gh.manual_seed(seed + 1000)
        hot = torch.randperm(s.E, generator=gh)[:SKEW_HOT]
        wr[hot] *= SKEW_FACTOR
        out["hot_experts"] = hot
    out["router_w"] = wr.to(torch.bfloat16)
    if s.fmt == "bf16":
        out["gate_up"] = _normal_bf16(g, (s.E, 2 * s.I, s.d), WEIGHT_STD)
        out["down"] = _normal_bf16(g, (s.E, s.d, s.I), WEIGHT_STD)
        out["gate_up_scales"] = None
        out["down_scales"] = None
    elif s.fmt == "int4":
        out["gate_up"], out["gate_up_scales"] = _int4_draw(g, (s.E, 2 * s.I), s.d, s.group)
        out["down"], out["down_scales"] = _int4_draw(g, (s.E, s.d), s.I, s.group)
    elif s.fmt == "fp8":
        out["gate_up"], out["gate_up_scales"] = _fp8_draw(g, (s.E, 2 * s.I), s.d, s.group)
        out["down"], out["down_scales"] = _fp8_draw(g, (s.E, s.d), s.I, s.group)
    elif s.fmt == "nvfp4":
        (out["gate_up"], out["gate_up_scales"],
         out["gate_up_global"]) = _nvfp4_draw(g, (s.E, 2 * s.I), s.d, s.group, s.E)
        (out["down"], out["down_scales"],
         out["down_global"]) = _nvfp4_draw(g, (s.E, s.d), s.I, s.group, s.E)
    else:
        raise ValueError(f"unknown weight format {s.fmt!r}")
    if s.Is > 0:
        out["w_sg"] = _normal_bf16(g, (s.d,), WEIGHT_STD)
        out["shared_gate_up"] = _normal_bf16(g, (2 * s.Is, s.d), WEIGHT_STD)
        out["shared_down"] = _normal_bf16(g, (s.d, s.Is), WEIGHT_STD)
    return out


def make_x(s: LayerShape, seed: int) -> torch.Tensor:
    """Only the token batch of make_inputs(s, seed) (x is its first draw)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randn((s.T, s.d), generator=g, dtype=torch.float32).to(torch.bfloat16)


def bits(t: torch.Tensor):
    """Raw bit pattern of a bf16 CPU tensor as a numpy uint16 array."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")
