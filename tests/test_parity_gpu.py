"""GPU parity of the CUDA path (called through the C ABI) against the fp64
oracle on the same seeded inputs: the whole layer on every workload shape,
each stage on its own, and the edge cases (T=1, T=0, ties, k=E, one expert
holding all tokens, several align block sizes, ragged tiles, bad ids)."""
import dataclasses
import time

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_gemv_gb300 import abi, build
from moe_expert_layer_gemv_gb300 import inputs as I
from moe_expert_layer_gemv_gb300.layer import MoeLayer

from _common import (NEAR_TIE, PARITY_LOG, WEIGHT_RTOL, bf16_to_f64, check_layout, check_routing,
                     compare_out, inputs, oracle_args, oracle_routing)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    abi.load()


def run_layer(inp, flags=0):
    s = inp["shape"]
    layer = MoeLayer(inp, "cuda", flags)
    x = inp["x"].cuda()
    ids = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
    w = torch.empty((s.T, s.k), dtype=torch.float32, device="cuda")
    out = layer.forward(x, topk_ids=ids, topk_weights=w)
    torch.cuda.synchronize()
    assert layer.device_status() == abi.MOE_OK
    return layer, out, ids.cpu().numpy(), w.cpu().numpy()


def logits64(inp):
    return (inp["x"].to(torch.float64) @ inp["router_w"].to(torch.float64).T).numpy()


def layer_parity(inp, name=None, flags=0):
    """Full-layer check of every token: routing against the oracle's (ids
    bit-exact off near-ties), the aligned layout the call left in its
    workspace bit for bit against the oracle's align of the call's ids, and the
    output against the oracle fed the call's ids (which covers near-ties)."""
    s = inp["shape"]
    layer, out, ids, w = run_layer(inp, flags)
    ref = oracle_routing(inp)
    n_near, n_mism = check_routing(ids, w, ref, ref["logits"])
    lay = layer.layout()
    check_layout(lay, ids, s.E, s.block)
    assert np.array_equal(lay["topk_weights"], w)
    ov = oracle.layer(*oracle_args(inp), ids_override=ids)
    np.testing.assert_allclose(w, ov["w"], rtol=WEIGHT_RTOL, atol=1e-7)
    name = name or f"{s.name} T={s.T} d={s.d} E={s.E} k={s.k} I={s.I} Is={s.Is} B={s.block}"
    rel, mx, lit = compare_out(bf16_to_f64(out), ov["out"], name)
    PARITY_LOG[-1].update(near=n_near, mism=n_mism)
    return {"rel": rel, "max": mx, "literal": lit, "near": n_near, "mism": n_mism,
            "layer": layer, "ids": ids, "out": out}


@pytest.mark.parametrize("name,seed", [("tiny", 0), ("tiny", 1), ("tiny", 2),
                                       ("verify_t8", 0), ("verify_t8", 1), ("verify_t8", 2),
                                       ("verify_t64", 0), ("verify_t64_skew", 0),
                                       ("int4_t32", 0), ("int4_t32", 1)])
def test_layer_parity_workloads(name, seed):
    layer_parity(inputs(name, seed), f"{name} seed {seed}")


def test_layer_parity_prefill_full():
    """The T=4096 prefill layer on the tensor-core path, every token against
    the oracle: all ~380 padded 128-row M blocks of the routed experts and all
    32 M blocks of the shared expert hold checked rows, and the multi-CTA
    align's layout is compared bit for bit."""
    layer_parity(inputs("prefill_t4096", 0), "prefill_t4096 seed 0 (all tokens)")


@pytest.mark.parametrize("over,seed", [
    ({"T": 5, "d": 264, "E": 12, "k": 3, "I": 40, "Is": 24}, 3),     # ragged everything
    ({"T": 1}, 4),                                                   # single token
    ({"T": 33, "d": 1032, "E": 70, "k": 5, "I": 200, "Is": 56, "block": 64}, 5),
    ({"T": 17, "d": 512, "E": 8, "k": 8, "I": 64, "Is": 0}, 6),      # k == E
    ({"T": 130, "d": 256, "E": 32, "k": 4, "I": 72, "Is": 40, "block": 128}, 7),  # T > fused top-k
    # rows so short that the expert stages' rings cannot hold the shared-memory
    # plan of 2048 slots over 512 experts: the routing kernel's last token tile
    # (of 16) runs the align and the workspace plan
    ({"T": 128, "d": 64, "E": 512, "k": 16, "I": 16, "Is": 16}, 8),
])
def test_layer_parity_ragged_and_edges(over, seed):
    layer_parity(I.make_inputs(I.shape("verify_t8", **over), seed))


def test_layer_int4_ragged():
    layer_parity(I.make_inputs(I.shape("int4_t32", T=7, d=512, E=20, k=4, I=256, Is=72), 9))


def test_zero_router_ties_pick_lowest_ids():
    inp = I.make_inputs(I.shape("verify_t8", T=6, d=256, E=16, k=4, I=32, Is=16), 1)
    inp["router_w"] = torch.zeros_like(inp["router_w"])
    layer, out, ids, w = run_layer(inp)
    assert ids.tolist() == [[0, 1, 2, 3]] * 6
    assert np.all(w == np.float32(0.25))
    ov = oracle.layer(*oracle_args(inp), ids_override=ids)
    compare_out(bf16_to_f64(out), ov["out"])


def test_one_expert_holds_every_token():
    # x > 0 and router row 3 = +1, others 0: every token's top-1 is expert 3.
    s = I.shape("verify_t8", T=64, d=256, E=8, k=1, I=48, Is=24)
    inp = I.make_inputs(s, 2)
    inp["x"] = inp["x"].abs()
    wr = torch.zeros((s.E, s.d), dtype=torch.bfloat16)
    wr[3] = 1.0
    inp["router_w"] = wr
    layer, out, ids, w = run_layer(inp)
    assert np.all(ids == 3) and np.all(w == 1.0)
    ov = oracle.layer(*oracle_args(inp), ids_override=ids)
    compare_out(bf16_to_f64(out), ov["out"])


def test_empty_batch_launches_nothing():
    s = I.shape("verify_t8", T=0)
    inp = I.make_inputs(s, 0)
    layer = MoeLayer(inp, "cuda")
    before = abi.moe_kernel_launch_count()
    out = torch.full((0, s.d), 7.0, dtype=torch.bfloat16, device="cuda")
    layer.forward(torch.empty((0, s.d), dtype=torch.bfloat16, device="cuda"), out=out)
    assert abi.moe_kernel_launch_count() == before


# ----------------------------------------------------------------------------- stage tests


def _stage_tensors(s):
    S = s.T * s.k
    cap = S + s.E * (s.block - 1)
    dev = "cuda"
    return {"ids": torch.empty((s.T, s.k), dtype=torch.int32, device=dev),
            "w": torch.empty((s.T, s.k), dtype=torch.float32, device=dev),
            "sorted": torch.full((cap,), -1, dtype=torch.int32, device=dev),
            "blocks": torch.full((cap // s.block + 1,), -1, dtype=torch.int32, device=dev),
            "npp": torch.zeros((1,), dtype=torch.int32, device=dev),
            "offs": torch.zeros((s.E + 1,), dtype=torch.int32, device=dev)}


@pytest.mark.parametrize("name,over", [("tiny", {}), ("verify_t8", {}), ("verify_t64", {}),
                                       ("int4_t32", {}),
                                       # T >= 256, E % 64 == 0: router logits on the tensor cores
                                       ("prefill_t4096", {"T": 1000, "I": 16, "Is": 16})])
def test_stage_route(name, over):
    s = I.shape(name, **over)
    inp = inputs(name, 0, **over)
    dims = abi.dims_of(s)
    ws = abi.alloc_workspace(dims)
    t = _stage_tensors(s)
    abi.moe_route(dims, inp["x"].cuda(), inp["router_w"].cuda(), t["ids"], t["w"], ws)
    torch.cuda.synchronize()
    L = logits64(inp)
    ids_ref, w_ref, margin, _ = oracle.topk(L, s.k, s.renormalize)
    ids = t["ids"].cpu().numpy()
    far = margin > NEAR_TIE
    assert np.array_equal(ids[far], ids_ref[far])
    w_ov = oracle.weights_for_ids(L, ids, s.renormalize)
    np.testing.assert_allclose(t["w"].cpu().numpy(), w_ov, rtol=WEIGHT_RTOL, atol=1e-7)


@pytest.mark.parametrize("T,E,k,B,seed", [(4, 8, 2, 16, 0), (8, 256, 8, 16, 1), (64, 256, 8, 16, 2),
                                          (4096, 256, 8, 128, 3), (32, 512, 10, 16, 4),
                                          (37, 5, 3, 1, 5), (300, 17, 4, 64, 6), (1, 1024, 16, 16, 7),
                                          # several 1024-slot chunks, the last one ragged
                                          (1000, 64, 5, 32, 8), (600, 1024, 16, 16, 9)])
def test_stage_align_bit_exact(T, E, k, B, seed):
    s = I.LayerShape(T=T, d=64, E=E, k=k, I=16, block=B)
    rng = np.random.default_rng(seed)
    ids_np = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    dims = abi.dims_of(s)
    ws = abi.alloc_workspace(dims)
    t = _stage_tensors(s)
    ids = torch.from_numpy(ids_np).cuda()
    abi.moe_align_block_size(dims, ids, t["sorted"], t["blocks"], t["npp"], t["offs"], ws)
    torch.cuda.synchronize()
    ref = oracle.align(ids_np.reshape(-1), E, B)
    n = int(t["npp"].item())
    assert n == ref["num_post_pad"]
    assert np.array_equal(t["sorted"].cpu().numpy()[:n], ref["sorted_ids"])
    assert np.array_equal(t["blocks"].cpu().numpy()[: n // B], ref["block_expert_ids"])
    assert np.array_equal(t["offs"].cpu().numpy(), ref["expert_offsets"])
    assert abi.moe_read_device_status(ws) == abi.MOE_OK


def test_stage_align_multi_chunk_skewed():
    """Most slots on one expert, spread over several chunks: ranks must run on
    across chunk boundaries in arrival order."""
    T, E, k, B = 3000, 16, 2, 64
    s = I.LayerShape(T=T, d=64, E=E, k=k, I=16, block=B)
    rng = np.random.default_rng(11)
    ids_np = np.empty((T, k), dtype=np.int32)
    ids_np[:, 0] = np.where(rng.random(T) < 0.9, 3, rng.integers(0, E, T))
    ids_np[:, 1] = (ids_np[:, 0] + 1 + rng.integers(0, E - 1, T)) % E
    dims = abi.dims_of(s)
    ws = abi.alloc_workspace(dims)
    t = _stage_tensors(s)
    abi.moe_align_block_size(dims, torch.from_numpy(ids_np).cuda(), t["sorted"], t["blocks"],
                             t["npp"], t["offs"], ws)
    torch.cuda.synchronize()
    ref = oracle.align(ids_np.reshape(-1), E, B)
    n = int(t["npp"].item())
    assert n == ref["num_post_pad"]
    assert np.array_equal(t["sorted"].cpu().numpy()[:n], ref["sorted_ids"])
    assert np.array_equal(t["offs"].cpu().numpy(), ref["expert_offsets"])


def test_stage_align_rejects_out_of_range_ids_without_fault():
    s = I.LayerShape(T=4, d=64, E=8, k=2, I=16, block=4)
    dims = abi.dims_of(s)
    ws = abi.alloc_workspace(dims)
    t = _stage_tensors(s)
    ids = torch.tensor([[0, 1], [2, 13], [-1, 3], [4, 5]], dtype=torch.int32, device="cuda")
    abi.moe_align_block_size(dims, ids, t["sorted"], t["blocks"], t["npp"], t["offs"], ws)
    assert abi.moe_read_device_status(ws) == abi.MOE_ERR_DEVICE_CHECK
    assert abi.moe_read_device_status(ws) == abi.MOE_OK  # read clears it


@pytest.mark.parametrize("name", ["tiny", "verify_t8", "verify_t64", "int4_t32"])
def test_stage_expert_forward_from_oracle_routing(name):
    """moe_expert_forward fed the oracle's routing and align layout (the
    workspace plan; at verify_t64 and int4_t32 both GEMV stages have dynamic
    tails)."""
    s = I.shape(name)
    inp = I.make_inputs(s, 1)
    args = oracle_args(inp)
    ref = oracle.layer(*args)
    al = oracle.align(ref["ids"].reshape(-1), s.E, s.block)
    layer = MoeLayer(inp, "cuda")
    t = _stage_tensors(s)
    n = al["num_post_pad"]
    t["sorted"][:n] = torch.from_numpy(al["sorted_ids"]).cuda()
    t["blocks"][: n // s.block] = torch.from_numpy(al["block_expert_ids"]).cuda()
    t["npp"][0] = n
    t["offs"].copy_(torch.from_numpy(al["expert_offsets"]))
    w = torch.from_numpy(ref["w"].astype(np.float32)).cuda()
    out = layer.new_out()
    abi.moe_expert_forward(layer.dims, inp["x"].cuda(), w, t["sorted"], t["blocks"], t["npp"],
                           t["offs"], layer.experts, layer.shared, out, layer.ws)
    torch.cuda.synchronize()
    assert layer.device_status() == abi.MOE_OK
    compare_out(bf16_to_f64(out), ref["out"])


@pytest.mark.parametrize("name", ["verify_t64_skew", "int4_t32"])
def test_repeat_calls_are_bitwise_deterministic(name):
    """Which CTA takes a unit of a dynamic tail changes from call to call; the
    output may not."""
    inp = inputs(name, 0)
    layer = MoeLayer(inp, "cuda")
    x = inp["x"].cuda()
    a = layer.forward(x).clone()
    for _ in range(3):
        b = layer.forward(x)
        assert torch.equal(a, b)


def test_timed_entry_point_matches_and_records_events():
    inp = inputs("verify_t8", 0)
    layer = MoeLayer(inp, "cuda")
    x = inp["x"].cuda()
    a = layer.forward(x).clone()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(abi.MOE_EV_COUNT)]
    b = layer.forward_timed(x, layer.new_out(), ev)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(abi.MOE_EV_COUNT - 1)]
    assert all(t >= 0 for t in times)


# ----------------------------------------------------------------------------- tensor-core path
# Dims with T >= 256, 128-row align blocks, I % 128 == 0, d % 256 == 0 and a
# shared expert of the routed width run the expert stages as grouped tcgen05
# GEMMs.


@pytest.mark.parametrize("over,seed", [
    ({"T": 256, "d": 256, "E": 4, "k": 2, "I": 128, "Is": 128, "block": 128}, 0),
    ({"T": 300, "d": 512, "E": 16, "k": 4, "I": 256, "Is": 256, "block": 128}, 1),
    ({"T": 512, "d": 768, "E": 9, "k": 3, "I": 384, "Is": 0, "block": 128}, 2),
    ({"T": 257, "d": 256, "E": 64, "k": 8, "I": 128, "Is": 128, "block": 256}, 3),
    # S = 5600 routing slots: the multi-chunk align
    ({"T": 700, "d": 256, "E": 64, "k": 8, "I": 128, "Is": 128, "block": 128}, 4),
])
def test_tensor_core_path_parity(over, seed):
    r = layer_parity(I.make_inputs(I.shape("verify_t8", **over), seed))
    print(f"tc {over}: rel-L2 {r['rel']:.2e} max/rms {r['max']:.2e}")


def test_tensor_core_path_one_expert_holds_every_token():
    s = I.shape("verify_t8", T=384, d=256, E=8, k=1, I=128, Is=128, block=128)
    inp = I.make_inputs(s, 4)
    inp["x"] = inp["x"].abs()
    wr = torch.zeros((s.E, s.d), dtype=torch.bfloat16)
    wr[5] = 1.0
    inp["router_w"] = wr
    layer, out, ids, w = run_layer(inp)
    assert np.all(ids == 5)
    ov = oracle.layer(*oracle_args(inp), ids_override=ids)
    compare_out(bf16_to_f64(out), ov["out"])


@pytest.mark.parametrize("name", ["tiny", "verify_t8"])
def test_layer_forward_replays_from_a_cuda_graph(name):
    """One layer call captured into a CUDA graph and replayed gives the eager
    call's output bit for bit, for new tokens copied into the captured x too."""
    s = I.shape(name)
    layer = MoeLayer(inputs(name, 0), "cuda")
    x = I.make_x(s, 100).cuda()
    out_g = layer.new_out()
    layer.forward(x, out_g)  # warm-up: one-time kernel attributes stay out of the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, out_g)
    for seed in (101, 102):
        x.copy_(I.make_x(s, seed).cuda())
        g.replay()
        ref = layer.forward(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(out_g, ref)
    assert layer.device_status() == abi.MOE_OK


# ----------------------------------------------------------------------------- batch invariance
# "veloGB10", Kernel work: batch-invariant GEMMs, so that a verify pass gives
# exactly what plain decode steps give.  Each token of a batched call must equal,
# bit for bit, the same token run alone.


def _single_token_rows(inp, flags=0):
    s = inp["shape"]
    one = dict(inp, shape=dataclasses.replace(s, T=1))
    one["x"] = inp["x"][:1].clone()
    layer = MoeLayer(one, "cuda", flags)
    rows, ids = [], []
    for t in range(s.T):
        x = inp["x"][t:t + 1].cuda()
        i1 = torch.empty((1, s.k), dtype=torch.int32, device="cuda")
        rows.append(layer.forward(x, topk_ids=i1).clone())
        ids.append(i1.clone())
    torch.cuda.synchronize()
    assert layer.device_status() == abi.MOE_OK
    return torch.cat(rows), torch.cat(ids)


@pytest.mark.parametrize("name,over", [("verify_t8", {}), ("verify_t64", {}),
                                       ("verify_t64_skew", {}), ("int4_t32", {}),
                                       # above the single-launch routing (unfused router)
                                       ("verify_t8", {"T": 160, "d": 512, "E": 64, "I": 128,
                                                      "Is": 128})])
def test_batch_invariance_decode_path(name, over):
    inp = inputs(name, 0, **over)
    layer, out, ids, _ = run_layer(inp)
    rows, ids1 = _single_token_rows(inp)
    assert np.array_equal(ids1.cpu().numpy(), ids)
    assert torch.equal(out, rows), "batched rows differ from single-token calls"


def test_batch_invariance_flag_keeps_prefill_sizes_invariant():
    """T >= 256 with tensor-core dims: only with MOE_FLAG_BATCH_INVARIANT do
    the rows equal single-token calls; the flagged call still meets parity."""
    s = I.shape("verify_t8", T=300, d=512, E=64, k=4, I=128, Is=128, block=128)
    inp = I.make_inputs(s, 5)
    f = abi.MOE_FLAG_BATCH_INVARIANT
    r = layer_parity(inp, "T=300 tensor-core dims, batch-invariant flag", flags=f)
    rows, ids1 = _single_token_rows(inp, flags=f)
    assert np.array_equal(ids1.cpu().numpy(), r["ids"])
    assert torch.equal(r["out"], rows)


# ----------------------------------------------------------------------------- bounded waits


def test_bounded_wait_times_out_and_the_workspace_recovers():
    """The stall hook makes the gate_up kernel's producers issue nothing: its
    consumers' bounded waits run out (no fault, nothing read out of bounds),
    the call records MOE_ERR_TIMEOUT, and after moe_workspace_init the same
    workspace gives the correct output again."""
    inp = inputs("verify_t8", 0)
    layer = MoeLayer(inp, "cuda")
    x = inp["x"].cuda()
    ref = layer.forward(x).clone()
    torch.cuda.synchronize()
    abi.moe_workspace_inject_stall(layer.ws, layer.ws.numel(), 2000)  # 2 ms
    t0 = time.perf_counter()
    layer.forward(x)
    code = layer.device_status()  # synchronises
    took = time.perf_counter() - t0
    assert code == abi.MOE_ERR_TIMEOUT
    assert took < 10.0
    abi.moe_workspace_init(layer.ws, layer.ws.numel())
    again = layer.forward(x)
    torch.cuda.synchronize()
    assert layer.device_status() == abi.MOE_OK
    assert torch.equal(again, ref)


# ----------------------------------------------------------------------------- layer chains
# A decode step runs the MoE layer of every transformer block in turn; the
# pages' engines capture that step into CUDA graphs ("Qwen3.6-35B-A3B on NVIDIA
# GB10", CUDA graphs; "Qwen3.8 Flash-Next - GB10 UltraFast", How it works:
# piecewise graphs).  Here several layers, each reading the previous layer's
# output, run back to back on one stream -- every launch with programmatic
# dependent launch, so a layer's routing starts while the previous layer's
# combine finishes -- once eagerly and once as one captured graph.


@pytest.mark.parametrize("T", [1, 8])
def test_multi_layer_chain_in_a_cuda_graph(T):
    s = I.shape("verify_t8", T=T, d=512, E=32, k=4, I=128, Is=64)
    n_layers = 4
    layers = [MoeLayer(I.make_inputs(s, 20 + i), "cuda") for i in range(n_layers)]
    acts = [torch.empty((T, s.d), dtype=torch.bfloat16, device="cuda") for _ in range(n_layers + 1)]

    def chain():
        for i, L in enumerate(layers):
            L.forward(acts[i], acts[i + 1])

    acts[0].copy_(I.make_x(s, 5).cuda())
    chain()  # eager; also sets the kernels' one-time attributes before the capture
    torch.cuda.synchronize()
    eager = [a.clone() for a in acts]
    # each layer against the oracle fed that layer's actual (bf16) input
    for i in range(n_layers):
        inp = dict(I.make_inputs(s, 20 + i), x=eager[i].cpu())
        ids = layers[i].layout()["topk_ids"]
        ov = oracle.layer(*oracle_args(inp), ids_override=ids)
        compare_out(bf16_to_f64(eager[i + 1]), ov["out"], f"chain T={T} layer {i}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for seed in (6, 7):
        acts[0].copy_(I.make_x(s, seed).cuda())
        g.replay()
        torch.cuda.synchronize()
        replayed = [a.clone() for a in acts]
        chain()
        torch.cuda.synchronize()
        for a, b in zip(replayed[1:], acts[1:]):
            assert torch.equal(a, b)
    for L in layers:
        assert L.device_status() == abi.MOE_OK
