"""Shared helpers of the test suite: feeding the same seeded inputs to the CUDA
path (through the C ABI) and to the fp64 oracle, and the parity criteria.

Parity criteria (the layer's stated pass bar):
  * expert ids, and the aligned sort/pad layout, bit-exact on every token whose
    oracle k-th vs (k+1)-th router-logit margin exceeds 1e-4; near-tie tokens
    are counted separately, their GPU choice must still be a valid top-k within
    the margin, and the oracle output is recomputed with the GPU's ids;
  * output rel-L2 error <= 5e-3 and max-abs error <= 2e-2 * rms(out) against
    the fp64 oracle, for the bf16 output.
"""
import functools

import numpy as np
import torch

import oracle
from moe_expert_layer_gemv_gb300 import inputs as I

# Parity figures of every layer comparison in this session, printed by the
# terminal summary (conftest.py): name, rel-L2, max-abs/rms beyond rounding,
# literal max-abs/rms, near-tie tokens, tokens whose ids differ.
PARITY_LOG = []

NEAR_TIE = 1e-4
REL_L2_TOL = 5e-3
MAX_ABS_TOL = 2e-2  # times rms(oracle out)
WEIGHT_RTOL = 2e-5  # fp32 softmax weights vs fp64


@functools.lru_cache(maxsize=3)
def _cached_inputs(name, seed, over):
    return I.make_inputs(I.shape(name, **dict(over)), seed)


def inputs(name, seed=0, **over):
    """I.make_inputs(I.shape(name, **over), seed), the last few kept: drawing a
    full-size layer's weights takes seconds.  Callers must not modify the
    returned tensors (make a new dict to change one)."""
    return _cached_inputs(name, seed, tuple(sorted(over.items())))


def oracle_args(inp):
    s = inp["shape"]
    fmt = oracle.BF16 if s.fmt == "bf16" else oracle.INT4
    conv = I.bits if s.fmt == "bf16" else (lambda t: t.numpy())
    ex = {"format": fmt, "group": s.group, "gate_up": conv(inp["gate_up"]), "down": conv(inp["down"]),
          "gate_up_scales": None if inp["gate_up_scales"] is None else I.bits(inp["gate_up_scales"]),
          "down_scales": None if inp["down_scales"] is None else I.bits(inp["down_scales"])}
    sh = None
    if s.Is > 0:
        sh = {"gate_up": I.bits(inp["shared_gate_up"]), "down": I.bits(inp["shared_down"]),
              "gate_w": I.bits(inp["w_sg"])}
    dims = {"T": s.T, "d": s.d, "E": s.E, "k": s.k, "I": s.I, "Is": s.Is,
            "renormalize": int(s.renormalize)}
    return I.bits(inp["x"]), I.bits(inp["router_w"]), ex, sh, dims


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def bf16_half_ulp(x):
    """Half a bf16 unit in the last place at each |x| (8 significant bits):
    the largest error of rounding x to the nearest bf16."""
    x = np.asarray(x, np.float64)
    _, p = np.frexp(x)  # |x| = m 2^p, m in [0.5, 1): ulp = 2^(p - 8)
    return np.where(x != 0, np.ldexp(1.0, p - 9), 0.0)


def compare_out(gpu_out, ref_out, name=None):
    """Returns (rel_l2, max_abs / rms beyond rounding, literal max_abs / rms)
    and asserts the pass bar; `name` logs the figures for the summary.

    The output is bf16, so even the correctly rounded exact result is off by
    up to half a bf16 ulp, which at a 6-sigma element lying just above a power
    of two is ~2.3% of rms: more than the 2e-2 rms bound itself.  The bound is
    therefore applied to the error of the computation, the rounding to the
    output type allowed on top: |out - exact| <= 2e-2 rms + half_ulp(exact).
    rel-L2 is taken as is (rounding alone contributes ~1.7e-3)."""
    g = np.asarray(gpu_out, np.float64)
    r = np.asarray(ref_out, np.float64)
    assert g.shape == r.shape
    assert np.all(np.isfinite(g))
    rms = float(np.sqrt(np.mean(r * r)))
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    err = np.abs(g - r)
    mx = float((err - bf16_half_ulp(r)).max() / max(rms, 1e-300)) if g.size else 0.0
    literal = float(err.max() / max(rms, 1e-300)) if g.size else 0.0
    if name is not None:
        PARITY_LOG.append({"name": name, "rel": rel, "max": mx, "literal": literal})
    assert rel <= REL_L2_TOL, f"rel-L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_TOL, f"max-abs/rms beyond bf16 rounding {mx:.3e} > {MAX_ABS_TOL} (raw {literal:.3e})"
    return rel, mx, literal


def oracle_routing(inp):
    """The oracle's own routing of the inputs: fp64 router logits, top-k ids,
    weights and the k-th vs (k+1)-th logit margin of every token."""
    s = inp["shape"]
    L = oracle.router_logits(oracle.decode_bf16(I.bits(inp["x"])),
                             oracle.decode_bf16(I.bits(inp["router_w"])))
    ids, w, margin, _ = oracle.topk(L, s.k, s.renormalize)
    return {"ids": ids, "w": w, "margin": margin, "logits": L}


def check_layout(lay, ids, E, B):
    """The aligned layout a layer call left in its workspace, bit for bit
    against the oracle's moe_align_block_size of the call's own ids."""
    ref = oracle.align(np.asarray(ids).reshape(-1), E, B)
    assert np.array_equal(lay["topk_ids"], ids)
    assert lay["num_post_pad"] == ref["num_post_pad"]
    assert np.array_equal(lay["sorted_ids"], ref["sorted_ids"])
    assert np.array_equal(lay["block_expert_ids"], ref["block_expert_ids"])
    assert np.array_equal(lay["expert_offsets"], ref["expert_offsets"])
    return ref


def check_routing(gpu_ids, gpu_w, ref, logits64=None):
    """ids bit-exact off near-ties; near-ties must be valid; weights close.
    `ref` is an oracle.layer result for the same tokens (own routing)."""
    ids = np.asarray(gpu_ids)
    margin = ref["margin"]
    far = margin > NEAR_TIE
    mism = np.any(ids != ref["ids"], axis=1)
    assert not np.any(mism & far), f"ids differ on {int(np.sum(mism & far))} tokens with margin > 1e-4"
    for t in np.nonzero(mism)[0]:
        assert len(set(ids[t].tolist())) == ids.shape[1]
        if logits64 is not None:
            kth = np.sort(logits64[t])[::-1][ids.shape[1] - 1]
            assert np.all(logits64[t][ids[t]] >= kth - NEAR_TIE)
    return int(np.sum(~far)), int(np.sum(mism))
