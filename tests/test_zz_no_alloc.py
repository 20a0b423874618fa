"""moe_layer_forward_static, the entry point for callers that may not allocate
device memory (no cudaMalloc allowed or available, so no workspace to pass): it
runs the layer with scratch in a fixed array inside the library.

It runs the very kernels moe_layer_forward runs, on the same inputs, so its
output must equal that entry point's bit for bit, on two calls in a row (the
second call reuses the array the first one left behind); it is also held to the
parity bar against the fp64 oracle.  This file is collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_gemv_gb300 import abi, build
from moe_expert_layer_gemv_gb300 import inputs as I
from moe_expert_layer_gemv_gb300.layer import MoeLayer

from _common import bf16_to_f64, compare_out, oracle_args

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    abi.load()


@pytest.mark.parametrize("name", ["verify_t8", "int4_t32"])
def test_static_scratch_matches_workspace_entry_point(name):
    s = I.shape(name)
    inp0 = I.make_inputs(s, 0)
    layer = MoeLayer(inp0, "cuda")
    lib = abi.load()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for seed in (11, 12):  # two calls in a row, different token batches
        x = I.make_x(s, seed).cuda()
        ids_ref = torch.empty((s.T, s.k), dtype=torch.int32, device="cuda")
        ref = layer.forward(x, topk_ids=ids_ref)
        out = torch.empty_like(ref)
        ids = torch.empty_like(ids_ref)
        sh = C.byref(layer.shared) if layer.shared is not None else None
        rc = lib.moe_layer_forward_static(C.byref(layer.dims), x.data_ptr(),
                                          layer.router_w.data_ptr(), C.byref(layer.experts), sh,
                                          out.data_ptr(), ids.data_ptr(), None, status.data_ptr(),
                                          C.c_void_p(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        assert rc == abi.MOE_OK, abi.moe_status_string(rc)
        assert int(status.item()) == abi.MOE_OK
        assert torch.equal(ids, ids_ref)
        assert torch.equal(out, ref)
        inp = dict(inp0, x=x.cpu())
        ov = oracle.layer(*oracle_args(inp), ids_override=ids.cpu().numpy())
        compare_out(bf16_to_f64(out), ov["out"], f"{name} static scratch, batch {seed}")


def test_static_scratch_checks_arguments_before_enqueueing_anything():
    """Argument errors come back before any GPU work (no launch counted)."""
    s = I.shape("verify_t8")
    dims = abi.dims_of(s)
    lib = abi.load()
    ex = abi.moe_expert_weights_t(1 << 40, None, 1 << 40, None)
    sh = abi.moe_shared_weights_t(1 << 40, 1 << 40, 1 << 40)
    before = abi.moe_kernel_launch_count()
    assert lib.moe_layer_forward_static(C.byref(dims), None, 1 << 40, C.byref(ex), C.byref(sh),
                                        1 << 40, None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_static(C.byref(dims), (1 << 40) + 2, 1 << 40, C.byref(ex),
                                        C.byref(sh), 1 << 40, None, None, None,
                                        None) == abi.MOE_ERR_INVALID_ARG
    assert abi.moe_kernel_launch_count() == before


def test_static_scratch_rejects_dims_beyond_its_size():
    s = I.shape("prefill_t4096")
    dims = abi.dims_of(s)
    assert abi.moe_workspace_bytes(dims) > abi.MOE_STATIC_SCRATCH_BYTES
    ex = abi.moe_expert_weights_t(1 << 40, None, 1 << 40, None)
    sh = abi.moe_shared_weights_t(1 << 40, 1 << 40, 1 << 40)
    rc = abi.load().moe_layer_forward_static(C.byref(dims), 1 << 40, 1 << 40, C.byref(ex),
                                             C.byref(sh), 1 << 40, None, None, None, None)
    assert rc == abi.MOE_ERR_WORKSPACE
