"""Pins for the fp64 CPU oracle, each against something other than the oracle
itself: exact bit-level facts, closed forms, brute force on tiny inputs,
independent library routines (numpy, scipy, torch fp64) and invariants.

A plausible slip in the oracle -- a swapped gate/up half, a dropped shared
term, a wrong nibble, an unstable align, an off-by-one margin, a missing
renormalisation -- fails at least one test here.
"""
import itertools
import math
import struct

import numpy as np
import pytest
import scipy.special
import torch
import torch.nn.functional as F

import oracle
from moe_expert_layer_gemv_gb300 import inputs as I


def f32_bits_to_bf16(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0] >> 16


# ----------------------------------------------------------------------------- decode


def test_bf16_decode_exact_values():
    cases = {0x3F80: 1.0, 0xC000: -2.0, 0x0000: 0.0, 0x3E80: 0.25, 0x4049: 3.140625,
             0x0001: 2.0 ** -133, 0x7F7F: 3.3895313892515355e38}
    got = oracle.decode_bf16(np.array(list(cases), np.uint16))
    assert list(got) == list(cases.values())
    assert math.isinf(oracle.decode_bf16(np.array([0x7F80], np.uint16))[0])


def test_bf16_decode_matches_torch_widening():
    rng = np.random.default_rng(0)
    b = rng.integers(0, 1 << 16, size=20000, dtype=np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]  # drop inf/nan patterns
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.decode_bf16(b), ref)


def test_int4_dequant_hand_example():
    # byte 0x8F: low nibble 0xF -> u=15 -> code 7; high nibble 0x8 -> code 0.
    # byte 0x01: low 1 -> code -7; high 0 -> code -8.   scale 0.5 (bf16 0x3F00)
    codes = np.array([[0x8F, 0x01]], np.uint8)
    scales = np.array([[0x3F00]], np.uint16)
    got = oracle.dequant_int4(codes, scales, cols=4, group=4)
    assert got.tolist() == [[3.5, 0.0, -3.5, -4.0]]


def test_int4_dequant_matches_independent_unpack():
    s = I.shape("int4_t32", E=3, d=256, I=64, T=2, Is=0)
    inp = I.make_inputs(s, seed=3)
    codes = inp["gate_up"].numpy()
    scales = inp["gate_up_scales"]
    lo = (codes & 15).astype(np.int64) - 8
    hi = (codes >> 4).astype(np.int64) - 8
    q = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (codes.shape[-1] * 2,))
    sc = scales.to(torch.float64).numpy()
    ref = q * np.repeat(sc, s.group, axis=-1)
    got = oracle.dequant_int4(codes, I.bits(scales), cols=s.d, group=s.group)
    assert np.array_equal(got, ref)
    assert q.min() >= -8 and q.max() <= 7


# ----------------------------------------------------------------------------- routing


def test_router_logits_match_blas():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 96))
    wr = rng.standard_normal((7, 96))
    got = oracle.router_logits(x, wr)
    np.testing.assert_allclose(got, x @ wr.T, rtol=1e-12, atol=1e-12)


def _brute_force_topk(L, k):
    """All k-subsets in lexicographic order; keep the first with the largest
    (exact, integer) sum -> max-sum set with ties to lower ids; order it by
    value descending, equal values by id ascending."""
    best, best_sum = None, None
    for sub in itertools.combinations(range(len(L)), k):
        ssum = sum(L[i] for i in sub)
        if best_sum is None or ssum > best_sum:
            best, best_sum = sub, ssum
    return sorted(best, key=lambda e: (-L[e], e))


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(2, 8))
    k = int(rng.integers(1, E + 1))
    L = rng.integers(-2, 3, size=E).astype(np.float64)  # small integers: many exact ties
    ids, w, margin, p = oracle.topk(L[None, :], k, renormalize=True)
    assert ids[0].tolist() == _brute_force_topk(L.tolist(), k)
    sm = scipy.special.softmax(L)
    np.testing.assert_allclose(p[0], sm, rtol=1e-14)
    ref_w = sm[ids[0]] / sm[ids[0]].sum()
    np.testing.assert_allclose(w[0], ref_w, rtol=1e-14)
    srt = np.sort(L)[::-1]
    if k < E:
        assert margin[0] == srt[k - 1] - srt[k]
    else:
        assert math.isinf(margin[0])


def test_topk_zero_router_picks_lowest_ids_uniform_weights():
    ids, w, margin, _ = oracle.topk(np.zeros((3, 10)), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3
    assert np.all(w == 0.25)
    assert np.all(margin == 0.0)


def test_topk_k_equals_E_is_softmax_and_no_renorm_is_p():
    rng = np.random.default_rng(7)
    L = rng.standard_normal((4, 6))
    ids, w, margin, _ = oracle.topk(L, 6)
    for t in range(4):
        np.testing.assert_allclose(w[t], scipy.special.softmax(L[t])[ids[t]], rtol=1e-14)
    assert np.all(np.isinf(margin))
    ids2, w2, _, _ = oracle.topk(L, 2, renormalize=False)
    for t in range(4):
        np.testing.assert_allclose(w2[t], scipy.special.softmax(L[t])[ids2[t]], rtol=1e-14)


def test_topk_weights_sum_to_one_and_ids_distinct():
    rng = np.random.default_rng(11)
    L = rng.standard_normal((64, 256))
    ids, w, _, _ = oracle.topk(L, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    # every chosen logit >= every unchosen logit
    for t in range(64):
        chosen = L[t, ids[t]]
        rest = np.delete(L[t], ids[t])
        assert chosen.min() >= rest.max()
        assert np.all(np.diff(chosen) <= 0)


def test_weights_for_ids_matches_selection_on_own_ids():
    rng = np.random.default_rng(5)
    L = rng.standard_normal((6, 12))
    ids, w, _, _ = oracle.topk(L, 3)
    assert np.array_equal(oracle.weights_for_ids(L, ids), w)
    other = np.array([[0, 5, 7]] * 6, np.int32)
    w2 = oracle.weights_for_ids(L, other)
    sm = scipy.special.softmax(L, axis=1)
    ref = np.take_along_axis(sm, other, 1)
    np.testing.assert_allclose(w2, ref / ref.sum(1, keepdims=True), rtol=1e-14)


# ----------------------------------------------------------------------------- align


def _reference_align(ids, E, B):
    """Stable library sort, then pad each expert's run to a multiple of B."""
    S = len(ids)
    order = sorted(range(S), key=lambda s: ids[s])  # Python's sort is stable
    sorted_ids, blocks, offs = [], [], []
    pos = 0
    for e in range(E):
        run = [s for s in order if ids[s] == e]
        offs.append(len(sorted_ids))
        if not run:
            continue
        padded = -(-len(run) // B) * B
        sorted_ids += run + [S] * (padded - len(run))
        blocks += [e] * (padded // B)
    offs.append(len(sorted_ids))
    return sorted_ids, blocks, offs


@pytest.mark.parametrize("S,E,B,seed", [(8, 8, 16, 0), (64, 256, 16, 1), (512, 256, 16, 2),
                                        (37, 5, 4, 3), (1, 3, 1, 4), (0, 4, 8, 5),
                                        (300, 17, 128, 6), (320, 512, 16, 7)])
def test_align_matches_stable_sort(S, E, B, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=S).astype(np.int32)
    got = oracle.align(ids, E, B)
    ref_sorted, ref_blocks, ref_offs = _reference_align(ids.tolist(), E, B)
    assert got["sorted_ids"].tolist() == ref_sorted
    assert got["block_expert_ids"].tolist() == ref_blocks
    assert got["expert_offsets"].tolist() == ref_offs
    assert got["num_post_pad"] == len(ref_sorted)
    # invariants
    c = got["counts"]
    assert c.sum() == S
    real = got["sorted_ids"][got["sorted_ids"] < S]
    assert sorted(real.tolist()) == list(range(S))
    assert got["num_post_pad"] % B == 0
    assert got["num_post_pad"] == int(sum(-(-int(v) // B) * B for v in c))
    assert np.all(np.diff(got["block_expert_ids"]) >= 0)
    assert got["num_post_pad"] <= oracle.align_capacity(S, E, B)


def test_align_all_to_one_expert():
    ids = np.full(33, 2, np.int32)
    got = oracle.align(ids, 4, 16)
    assert got["num_post_pad"] == 48
    assert got["sorted_ids"].tolist() == list(range(33)) + [33] * 15
    assert got["block_expert_ids"].tolist() == [2, 2, 2]
    assert got["expert_offsets"].tolist() == [0, 0, 0, 48, 48]


# ----------------------------------------------------------------------------- expert + combine


def test_swiglu_expert_matches_torch_fp64():
    rng = np.random.default_rng(2)
    d, Ie = 48, 20
    x = rng.standard_normal(d)
    wgu = rng.standard_normal((2 * Ie, d)) * 0.2
    wd = rng.standard_normal((d, Ie)) * 0.2
    got = oracle.swiglu_expert(x, wgu, wd)
    xt = torch.from_numpy(x)
    g = F.linear(xt, torch.from_numpy(wgu[:Ie]))
    u = F.linear(xt, torch.from_numpy(wgu[Ie:]))
    ref = F.linear(F.silu(g) * u, torch.from_numpy(wd)).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_swiglu_closed_form():
    # x = e0; gate row 0 = [2,0], up row = [3,0] -> h = silu(2)*3; Wd = [[1],[0.5]]
    y = oracle.swiglu_expert(np.array([1.0, 0.0]), np.array([[2.0, 0.0], [3.0, 0.0]]),
                             np.array([[1.0], [0.5]]))
    h = 2.0 / (1.0 + math.exp(-2.0)) * 3.0
    assert y.tolist() == [h, 0.5 * h]


def test_combine_identity_expert_reproduces_input():
    rng = np.random.default_rng(4)
    T, k, d = 6, 3, 40
    x = rng.standard_normal((T, d))
    w = rng.random((T, k))
    w /= w.sum(1, keepdims=True)
    y = np.repeat(x, k, axis=0)  # identity expert: y_tj = x_t
    out = oracle.combine(w, y)
    np.testing.assert_allclose(out, x, rtol=0, atol=1e-15 * np.abs(x).max() * 4)


def test_combine_shared_gate_zero_is_half():
    rng = np.random.default_rng(6)
    T, k, d = 3, 2, 8
    w = rng.random((T, k))
    y = rng.standard_normal((T * k, d))
    ys = rng.standard_normal((T, d))
    out = oracle.combine(w, y, np.zeros(T), ys)
    routed = oracle.combine(w, y)
    assert np.array_equal(out, routed + 0.5 * ys)


# ----------------------------------------------------------------------------- full layer


def _oracle_args(inp):
    s = inp["shape"]
    fmt = {"bf16": oracle.BF16, "int4": oracle.INT4, "fp8": oracle.FP8, "nvfp4": oracle.NVFP4}[s.fmt]
    conv = (lambda t: I.bits(t)) if s.fmt == "bf16" else (lambda t: t.numpy())
    sconv = (lambda t: t.numpy()) if s.fmt == "nvfp4" else I.bits  # E4M3 bytes, else bf16 bits
    ex = {"format": fmt, "group": s.group, "gate_up": conv(inp["gate_up"]), "down": conv(inp["down"]),
          "gate_up_scales": None if inp["gate_up_scales"] is None else sconv(inp["gate_up_scales"]),
          "down_scales": None if inp["down_scales"] is None else sconv(inp["down_scales"])}
    if s.fmt == "nvfp4":
        ex["gate_up_global"] = inp["gate_up_global"].numpy()
        ex["down_global"] = inp["down_global"].numpy()
    sh = None
    if s.Is > 0:
        sh = {"gate_up": I.bits(inp["shared_gate_up"]), "down": I.bits(inp["shared_down"]),
              "gate_w": I.bits(inp["w_sg"])}
    dims = {"T": s.T, "d": s.d, "E": s.E, "k": s.k, "I": s.I, "Is": s.Is,
            "renormalize": int(s.renormalize)}
    return I.bits(inp["x"]), I.bits(inp["router_w"]), ex, sh, dims


def _torch_dense_mixture(inp):
    """Dense restatement: every expert on every token, gate weight zero outside
    the top-k (softmax over E, renormalised over the selected set)."""
    s = inp["shape"]
    f = lambda t: t.to(torch.float64)
    x = f(inp["x"])
    logits = x @ f(inp["router_w"]).T
    p = torch.softmax(logits, dim=-1)
    top = torch.topk(logits, s.k, dim=-1)
    gate = torch.zeros_like(p)
    sel = torch.gather(p, 1, top.indices)
    gate.scatter_(1, top.indices, sel / sel.sum(1, keepdim=True) if s.renormalize else sel)
    gu = f(inp["gate_up"])
    dn = f(inp["down"])
    g = torch.einsum("td,eid->tei", x, gu[:, : s.I])
    u = torch.einsum("td,eid->tei", x, gu[:, s.I:])
    y = torch.einsum("tei,edi->ted", F.silu(g) * u, dn)
    out = torch.einsum("te,ted->td", gate, y)
    if s.Is > 0:
        sgu = f(inp["shared_gate_up"])
        h = F.silu(x @ sgu[: s.Is].T) * (x @ sgu[s.Is:].T)
        out = out + torch.sigmoid(x @ f(inp["w_sg"]))[:, None] * (h @ f(inp["shared_down"]).T)
    return out.numpy(), top.indices.numpy()


@pytest.mark.parametrize("name,over,seed", [
    ("tiny", {}, 0),
    ("tiny", {}, 1),
    ("verify_t8", {"d": 128, "E": 16, "I": 24, "Is": 40, "T": 5}, 0),
    ("verify_t8", {"d": 64, "E": 6, "k": 6, "I": 16, "Is": 8, "T": 3}, 2),
])
def test_layer_equals_dense_mixture(name, over, seed):
    inp = I.make_inputs(I.shape(name, **over), seed=seed)
    res = oracle.layer(*_oracle_args(inp))
    ref, ref_ids = _torch_dense_mixture(inp)
    s = inp["shape"]
    # torch.topk's order among exact ties is unspecified; seeds avoid ties
    assert np.array_equal(np.sort(res["ids"], 1), np.sort(ref_ids, 1))
    scale = np.linalg.norm(ref)
    assert np.linalg.norm(res["out"] - ref) <= 1e-12 * scale
    assert np.all(np.abs(res["w"].sum(1) - 1.0) <= 1e-12)
    assert res["out"].shape == (s.T, s.d)


def test_layer_single_expert_is_dense_swiglu():
    s = I.LayerShape(T=3, d=64, E=1, k=1, I=32)
    inp = I.make_inputs(s, seed=9)
    res = oracle.layer(*_oracle_args(inp))
    x = inp["x"].to(torch.float64)
    gu = inp["gate_up"][0].to(torch.float64)
    dn = inp["down"][0].to(torch.float64)
    ref = F.linear(F.silu(F.linear(x, gu[:32])) * F.linear(x, gu[32:]), dn).numpy()
    np.testing.assert_allclose(res["out"], ref, rtol=1e-12, atol=1e-14)
    assert np.all(res["w"] == 1.0) and np.all(res["ids"] == 0)


def test_layer_closed_form_with_shared_expert():
    """tests/golden/closed_form_layer.json: a hand-chosen one-token layer whose
    output has a closed form in exp() (computed here, not stored)."""
    import json
    import os

    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_form_layer.json")))
    bf = lambda a: np.array([f32_bits_to_bf16(v) for v in np.ravel(a)], np.uint16).reshape(
        np.shape(a))
    dm = g["dims"]
    sh = {"gate_up": bf(g["shared_gate_up"]), "down": bf(g["shared_down"]), "gate_w": bf(g["w_sg"])}
    res = oracle.layer(bf(g["x"]), bf(g["router_w"]),
                       {"format": oracle.BF16, "gate_up": bf(g["gate_up"]), "down": bf(g["down"])},
                       sh, dm)
    h = 2.0 / (1.0 + math.exp(-2.0)) * 3.0   # expert 0: g = 2, u = 3
    hs = 1.0 / (1.0 + math.exp(-1.0))        # shared: g = u = 1, sigmoid gate at 0 = 1/2
    assert res["ids"].tolist() == [[0]]
    assert res["w"].tolist() == [[1.0]]
    np.testing.assert_allclose(res["out"][0], [h + 0.5 * hs, 0.5 * h + 0.5 * hs], rtol=1e-15)
    assert res["sg"][0] == 0.0


def test_layer_down_linearity_and_token_subset():
    s = I.shape("tiny")
    inp = I.make_inputs(s, seed=4)
    args = list(_oracle_args(inp))
    base = oracle.layer(*args)
    dn2 = (inp["down"].to(torch.float32) * 2).to(torch.bfloat16)  # exact doubling
    args2 = list(args)
    args2[2] = dict(args[2], down=I.bits(dn2))
    dbl = oracle.layer(*args2)
    assert np.array_equal(dbl["out"], 2 * base["out"])
    sub = oracle.layer(*args, tokens=np.array([3, 1], np.int32))
    assert np.array_equal(sub["out"], base["out"][[3, 1]])
    assert np.array_equal(sub["ids"], base["ids"][[3, 1]])


def test_layer_ids_override():
    s = I.shape("tiny")
    inp = I.make_inputs(s, seed=5)
    args = _oracle_args(inp)
    base = oracle.layer(*args)
    same = oracle.layer(*args, ids_override=base["ids"])
    assert np.array_equal(same["out"], base["out"])
    flipped = base["ids"][:, ::-1].copy()  # same set, other order: same sum up to rounding
    fl = oracle.layer(*args, ids_override=flipped)
    np.testing.assert_allclose(fl["out"], base["out"], rtol=1e-13, atol=1e-15)
    other = np.array([[6, 7]] * s.T, np.int32)
    ot = oracle.layer(*args, ids_override=other)
    assert np.array_equal(ot["ids"], other)
    assert not np.allclose(ot["out"], base["out"])


def test_layer_int4_equals_dequantised_f64():
    s = I.shape("int4_t32", T=4, d=128, E=6, k=3, I=64, Is=32)
    inp = I.make_inputs(s, seed=8)
    x, wr, ex, sh, dims = _oracle_args(inp)
    q = oracle.layer(x, wr, ex, sh, dims)
    # independent unpack (numpy) -> the fp64 test format
    def deq(codes, scales, cols):
        lo = (codes & 15).astype(np.int64) - 8
        hi = (codes >> 4).astype(np.int64) - 8
        v = np.stack([lo, hi], -1).reshape(codes.shape[:-1] + (cols,))
        return v * np.repeat(scales.to(torch.float64).numpy(), s.group, -1)
    ex64 = {"format": oracle.F64, "gate_up": deq(inp["gate_up"].numpy(), inp["gate_up_scales"], s.d),
            "down": deq(inp["down"].numpy(), inp["down_scales"], s.I)}
    f = oracle.layer(x, wr, ex64, sh, dims)
    assert np.array_equal(q["out"], f["out"])


def test_margin_is_kth_minus_next_logit():
    inp = I.make_inputs(I.shape("tiny"), seed=0)
    res = oracle.layer(*_oracle_args(inp))
    L = inp["x"].to(torch.float64) @ inp["router_w"].to(torch.float64).T
    srt = torch.sort(L, dim=1, descending=True).values
    np.testing.assert_allclose(res["margin"], (srt[:, 1] - srt[:, 2]).numpy(), rtol=1e-12)


# ----------------------------------------------------------------------------- fp8 / nvfp4
# Block-scaled weight formats ("veloGB10": the NVFP4/FP8 weight families it
# serves).  The element decodes are pinned against torch's float8_e4m3fn and
# against the E2M1 value table of the format's definition; the layer in each
# format against the same layer on independently dequantised fp64 weights.

E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e4m3_decode_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    got = [oracle.e4m3_to_f64(b) for b in range(256)]
    for b in range(256):
        if math.isnan(ref[b]):
            assert math.isnan(got[b]) and (b & 0x7F) == 0x7F, hex(b)
        else:
            assert got[b] == ref[b] and math.copysign(1, got[b]) == math.copysign(1, ref[b]), hex(b)
    # the format's landmarks: smallest subnormal, smallest normal, one, largest
    assert got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6
    assert got[0x38] == 1.0 and got[0x7E] == 448.0


def test_e2m1_decode_is_the_format_table():
    got = [oracle.e2m1_to_f64(c) for c in range(16)]
    assert got[:8] == E2M1_MAGNITUDES
    assert got[8:] == [-m for m in E2M1_MAGNITUDES]
    assert math.copysign(1, got[8]) == -1.0  # code 8 is -0


def _fp8_codes(rng, shape):
    """Random E4M3 bytes without the two NaN patterns."""
    c = rng.integers(0, 254, size=shape, dtype=np.int64)
    c = np.where(c >= 0x7F, c + 1, c)  # skip 0x7F
    return np.where(c >= 0xFF, 0xFE, c).astype(np.uint8)


def _bf16_scales(rng, shape):
    return I.bits(torch.from_numpy(np.abs(rng.normal(0.0, 0.01, size=shape)).astype(np.float32))
                  .to(torch.bfloat16))


def _e4m3_scales(rng, shape):
    """Positive E4M3 block scales (exponent field 1..14)."""
    e = rng.integers(1, 15, size=shape)
    m = rng.integers(0, 8, size=shape)
    return ((e << 3) | m).astype(np.uint8)


def _deq_fp8(codes, scales_bits, group):
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    sc = torch.from_numpy(scales_bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64)
    return v * np.repeat(sc.numpy(), group, axis=-1)


def _deq_nvfp4(codes, scales, glob, group, cols):
    table = np.array(E2M1_MAGNITUDES + [-m for m in E2M1_MAGNITUDES])
    lo = table[codes & 15]
    hi = table[codes >> 4]
    v = np.stack([lo, hi], -1).reshape(codes.shape[:-1] + (cols,))
    sc = torch.from_numpy(scales).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return v * np.repeat(sc, group, axis=-1) * glob.astype(np.float64).reshape(
        (-1,) + (1,) * (codes.ndim - 1))


def test_fp8_dequant_matches_independent_decode():
    rng = np.random.default_rng(11)
    codes = _fp8_codes(rng, (5, 96))
    scales = _bf16_scales(rng, (5, 3))
    got = oracle.dequant_fp8(codes, scales, cols=96, group=32)
    assert np.array_equal(got, _deq_fp8(codes, scales, 32))


def test_nvfp4_dequant_matches_independent_decode():
    rng = np.random.default_rng(12)
    codes = rng.integers(0, 256, size=(4, 32), dtype=np.int64).astype(np.uint8)  # 64 elements/row
    scales = _e4m3_scales(rng, (4, 4))
    glob = np.float32(0.0625)
    got = oracle.dequant_nvfp4(codes, scales, glob, cols=64, group=16)
    ref = _deq_nvfp4(codes[None], scales[None], np.array([glob]), 16, 64)[0]
    assert np.array_equal(got, ref)
    # hand example: byte 0x2F -> low nibble 0xF = -6, high 0x2 = 1.0; scale 0x38 = 1.0
    one = oracle.dequant_nvfp4(np.array([[0x2F]], np.uint8), np.array([[0x38]], np.uint8),
                               np.float32(2.0), cols=2, group=2)
    assert one.tolist() == [[-12.0, 2.0]]


def _quant_layer_inputs(seed):
    s = I.shape("verify_t8", T=4, d=128, E=6, k=3, I=64, Is=32)
    return s, I.make_inputs(s, seed=seed)


def test_layer_fp8_equals_dequantised_f64():
    s, inp = _quant_layer_inputs(13)
    x, wr, _, sh, dims = _oracle_args(inp)
    rng = np.random.default_rng(13)
    g = 32
    gu = _fp8_codes(rng, (s.E, 2 * s.I, s.d))
    dn = _fp8_codes(rng, (s.E, s.d, s.I))
    gus = _bf16_scales(rng, (s.E, 2 * s.I, s.d // g))
    dns = _bf16_scales(rng, (s.E, s.d, s.I // g))
    q = oracle.layer(x, wr, {"format": oracle.FP8, "group": g, "gate_up": gu, "down": dn,
                             "gate_up_scales": gus, "down_scales": dns}, sh, dims)
    f = oracle.layer(x, wr, {"format": oracle.F64, "gate_up": _deq_fp8(gu, gus, g),
                             "down": _deq_fp8(dn, dns, g)}, sh, dims)
    assert np.array_equal(q["ids"], f["ids"])
    assert np.array_equal(q["out"], f["out"])


def test_layer_nvfp4_equals_dequantised_f64():
    s, inp = _quant_layer_inputs(14)
    x, wr, _, sh, dims = _oracle_args(inp)
    rng = np.random.default_rng(14)
    g = 16
    gu = rng.integers(0, 256, size=(s.E, 2 * s.I, s.d // 2), dtype=np.int64).astype(np.uint8)
    dn = rng.integers(0, 256, size=(s.E, s.d, s.I // 2), dtype=np.int64).astype(np.uint8)
    gus = _e4m3_scales(rng, (s.E, 2 * s.I, s.d // g))
    dns = _e4m3_scales(rng, (s.E, s.d, s.I // g))
    gug = (2.0 ** rng.integers(-12, -6, size=s.E)).astype(np.float32)
    dng = (2.0 ** rng.integers(-12, -6, size=s.E)).astype(np.float32)
    ex = {"format": oracle.NVFP4, "group": g, "gate_up": gu, "down": dn, "gate_up_scales": gus,
          "down_scales": dns, "gate_up_global": gug, "down_global": dng}
    q = oracle.layer(x, wr, ex, sh, dims)
    f = oracle.layer(x, wr, {"format": oracle.F64, "gate_up": _deq_nvfp4(gu, gus, gug, g, s.d),
                             "down": _deq_nvfp4(dn, dns, dng, g, s.I)}, sh, dims)
    assert np.array_equal(q["ids"], f["ids"])
    assert np.array_equal(q["out"], f["out"])
    # the per-expert scale is required
    with pytest.raises(ValueError):
        oracle.layer(x, wr, dict(ex, gate_up_global=None), sh, dims)


@pytest.mark.parametrize("fmt,group", [("fp8", 32), ("nvfp4", 16)])
def test_layer_on_drawn_quantised_weights_equals_dequantised_f64(fmt, group):
    """The same pin on the input recipe's own FP8 / NVFP4 draws."""
    s = I.shape("int4_t32", T=5, d=256, E=6, k=3, I=64, Is=32, fmt=fmt, group=group)
    inp = I.make_inputs(s, seed=15)
    x, wr, ex, sh, dims = _oracle_args(inp)
    q = oracle.layer(x, wr, ex, sh, dims)
    if fmt == "fp8":
        f64 = {"gate_up": _deq_fp8(ex["gate_up"], ex["gate_up_scales"], group),
               "down": _deq_fp8(ex["down"], ex["down_scales"], group)}
    else:
        f64 = {"gate_up": _deq_nvfp4(ex["gate_up"], ex["gate_up_scales"], ex["gate_up_global"],
                                     group, s.d),
               "down": _deq_nvfp4(ex["down"], ex["down_scales"], ex["down_global"], group, s.I)}
    f = oracle.layer(x, wr, dict(f64, format=oracle.F64), sh, dims)
    assert np.array_equal(q["ids"], f["ids"])
    assert np.array_equal(q["out"], f["out"])
    assert np.isfinite(q["out"]).all()
