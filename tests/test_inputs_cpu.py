"""The seeded input recipe: shapes, dtypes, value distributions, the int4
packing, the skewed-routing variant and determinism -- what the parity tests,
the smoke check and the bench all feed both the CUDA path and the oracle."""
import math

import numpy as np
import pytest
import torch

from moe_expert_layer_gemv_gb300 import inputs as I


def test_workload_table():
    s = I.shape("verify_t8")
    assert (s.T, s.d, s.E, s.k, s.I, s.Is, s.block, s.fmt) == (8, 2048, 256, 8, 512, 512, 16, "bf16")
    s = I.shape("int4_t32")
    assert (s.T, s.d, s.E, s.k, s.I, s.Is, s.fmt, s.group) == (32, 2048, 512, 10, 512, 1024, "int4", 32)
    assert I.shape("prefill_t4096").block == 128 and I.shape("prefill_t4096").T == 4096
    assert I.shape("verify_t64_skew").skew and not I.shape("verify_t64").skew
    assert I.shape("tiny").Is == 0
    assert I.shape("verify_t8", T=3).T == 3  # overrides keep the rest


def test_bf16_shapes_and_distributions():
    s = I.shape("verify_t8", E=16)
    inp = I.make_inputs(s, 0)
    assert inp["x"].shape == (8, 2048) and inp["x"].dtype == torch.bfloat16
    assert inp["router_w"].shape == (16, 2048)
    assert inp["gate_up"].shape == (16, 1024, 2048) and inp["down"].shape == (16, 2048, 512)
    assert inp["w_sg"].shape == (2048,)
    assert inp["shared_gate_up"].shape == (1024, 2048) and inp["shared_down"].shape == (2048, 512)
    x = inp["x"].float()
    assert abs(x.mean().item()) < 0.05 and abs(x.std().item() - 1.0) < 0.05
    for key in ("router_w", "gate_up", "down", "shared_gate_up", "shared_down"):
        w = inp[key].float()
        assert abs(w.mean().item()) < 1e-3, key
        assert abs(w.std().item() / 0.02 - 1.0) < 0.03, key


def test_int4_codes_scales_and_packing():
    s = I.shape("int4_t32", E=4)
    inp = I.make_inputs(s, 0)
    gu, gus = inp["gate_up"], inp["gate_up_scales"]
    assert gu.dtype == torch.uint8 and gu.shape == (4, 1024, 1024)
    assert gus.dtype == torch.bfloat16 and gus.shape == (4, 1024, 64)
    assert inp["down"].shape == (4, 2048, 256) and inp["down_scales"].shape == (4, 2048, 16)
    lo = (gu & 0xF).to(torch.int64) - 8
    hi = (gu >> 4).to(torch.int64) - 8
    codes = torch.cat([lo.flatten(), hi.flatten()])
    assert codes.min().item() == -8 and codes.max().item() == 7
    freq = torch.bincount(codes + 8, minlength=16).double() / codes.numel()
    assert (freq - 1 / 16).abs().max().item() < 2e-3  # uniform over [-8, 7]
    sc = gus.float()
    assert sc.min().item() >= 0.0
    # |N(0, s)| has mean s * sqrt(2 / pi)
    assert abs(sc.mean().item() / (0.003 * math.sqrt(2 / math.pi)) - 1.0) < 0.02
    # the shared expert stays bf16 ~ N(0, 0.02)
    assert inp["shared_gate_up"].dtype == torch.bfloat16 and inp["shared_gate_up"].shape == (2048, 2048)


def test_int4_pack_even_element_in_low_nibble():
    q = torch.tensor([[-8, 7, 0, -1, 3, -5]], dtype=torch.int16)
    p = I._int4_pack(q)
    assert p.tolist() == [[0x0 | (0xF << 4), 0x8 | (0x7 << 4), 0xB | (0x3 << 4)]]


def test_skewed_router_rows():
    s = I.shape("verify_t64_skew", E=64)
    inp = I.make_inputs(s, 3)
    g = torch.Generator().manual_seed(3 + 1000)
    hot = torch.randperm(64, generator=g)[:16]
    assert torch.equal(inp["hot_experts"], hot)
    wr = inp["router_w"].float()
    mask = torch.zeros(64, dtype=torch.bool)
    mask[hot] = True
    assert abs(wr[mask].std().item() / 0.08 - 1.0) < 0.03
    assert abs(wr[~mask].std().item() / 0.02 - 1.0) < 0.03
    # the skew leaves every other draw unchanged
    plain = I.make_inputs(I.shape("verify_t64", E=64), 3)
    assert torch.equal(plain["x"], inp["x"]) and torch.equal(plain["gate_up"], inp["gate_up"])
    assert torch.equal(plain["router_w"][~mask], inp["router_w"][~mask])


def test_determinism_and_token_batches():
    s = I.shape("tiny")
    a, b = I.make_inputs(s, 7), I.make_inputs(s, 7)
    for key in ("x", "router_w", "gate_up", "down"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["x"], I.make_inputs(s, 8)["x"])
    assert torch.equal(I.make_x(s, 7), a["x"])


def test_bits_round_trip():
    t = torch.tensor([1.0, -2.5, 0.0, float("inf")], dtype=torch.bfloat16)
    b = I.bits(t)
    assert b.dtype == np.uint16 and b.tolist() == [0x3F80, 0xC020, 0x0000, 0x7F80]


def test_fp8_codes_scales_and_ranges():
    s = I.shape("int4_t32", T=4, d=256, E=4, k=2, I=64, Is=32, fmt="fp8", group=32)
    a = I.make_inputs(s, seed=2)
    gu, dn = a["gate_up"], a["down"]
    assert gu.shape == (s.E, 2 * s.I, s.d) and gu.dtype == torch.uint8
    assert dn.shape == (s.E, s.d, s.I) and dn.dtype == torch.uint8
    assert a["gate_up_scales"].shape == (s.E, 2 * s.I, s.d // 32)
    assert a["down_scales"].shape == (s.E, s.d, s.I // 32)
    for c in (gu, dn):
        assert not bool(((c & 0x7F) == 0x7F).any())  # no NaN pattern
        v = c.view(torch.float8_e4m3fn).to(torch.float32)
        assert float(v.abs().max()) <= I.E4M3_MAX
        assert abs(float(v.std()) / I.FP8_VALUE_STD - 1.0) < 0.05
    sc = a["gate_up_scales"].to(torch.float32)
    assert float(sc.min()) >= 0.0 and abs(float(sc.mean()) / (I.FP8_SCALE_STD * math.sqrt(2 / math.pi)) - 1) < 0.1


def test_nvfp4_codes_scales_globals():
    s = I.shape("int4_t32", T=4, d=256, E=4, k=2, I=64, Is=32, fmt="nvfp4", group=16)
    a = I.make_inputs(s, seed=3)
    assert a["gate_up"].shape == (s.E, 2 * s.I, s.d // 2)
    assert a["down"].shape == (s.E, s.d, s.I // 2)
    assert a["gate_up_scales"].shape == (s.E, 2 * s.I, s.d // 16)
    assert a["down_scales"].shape == (s.E, s.d, s.I // 16)
    nib = torch.cat([a["gate_up"] & 15, a["gate_up"] >> 4]).to(torch.int64)
    counts = torch.bincount(nib.flatten(), minlength=16).to(torch.float64)
    assert float(counts.min()) > 0.9 * float(counts.mean())  # all 16 codes, near uniform
    for sc in (a["gate_up_scales"], a["down_scales"]):
        v = sc.view(torch.float8_e4m3fn).to(torch.float32)
        assert float(v.min()) >= 1.0 and float(v.max()) <= 4.0
    for gl in (a["gate_up_global"], a["down_global"]):
        assert gl.shape == (s.E,) and gl.dtype == torch.float32
        assert float(gl.min()) >= 2.0 ** -9 and float(gl.max()) <= 2.0 ** -8


def test_quantised_formats_are_deterministic():
    for fmt, g in (("fp8", 32), ("nvfp4", 16)):
        s = I.shape("int4_t32", T=2, d=256, E=3, k=2, I=64, Is=0, fmt=fmt, group=g)
        a, b, c = I.make_inputs(s, 5), I.make_inputs(s, 5), I.make_inputs(s, 6)
        assert torch.equal(a["gate_up"], b["gate_up"]) and torch.equal(a["down_scales"], b["down_scales"])
        assert not torch.equal(a["gate_up"], c["gate_up"])
