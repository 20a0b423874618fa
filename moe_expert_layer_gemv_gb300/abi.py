"""ctypes binding of the C ABI in include/moe.h -- argument marshalling only.

Every function here has the name of the C entry point it calls and takes torch
CUDA tensors (or raw device addresses as ints) where the C call takes device
pointers.  All arithmetic runs in libmoe_gb300.so; if that library is missing
the first call raises, there is no fallback.
"""
import ctypes as C
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_DEVICE_CHECK, MOE_ERR_TIMEOUT = 4, 5, 6
MOE_WEIGHTS_BF16, MOE_WEIGHTS_INT4_G32 = 0, 1
MOE_EV_BEGIN, MOE_EV_ROUTED, MOE_EV_GATE_UP, MOE_EV_DOWN, MOE_EV_END, MOE_EV_COUNT = range(6)

# Every extern "C" symbol include/moe.h declares.
EXPORTS = ("moe_status_string", "moe_workspace_bytes", "moe_workspace_init",
           "moe_workspace_views", "moe_workspace_inject_stall", "moe_route",
           "moe_align_block_size", "moe_expert_forward", "moe_layer_forward",
           "moe_layer_forward_timed", "moe_layer_forward_static", "moe_read_device_status",
           "moe_kernel_launch_count")
MOE_STATIC_SCRATCH_BYTES = 32 << 20
MOE_FLAG_BATCH_INVARIANT = 1


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where}: {text}")
        self.status = status


class moe_dims_t(C.Structure):
    _fields_ = [("T", C.c_int32), ("d", C.c_int32), ("E", C.c_int32), ("top_k", C.c_int32),
                ("I", C.c_int32), ("I_shared", C.c_int32), ("renormalize", C.c_int32),
                ("block_size", C.c_int32), ("weight_format", C.c_int32), ("group_size", C.c_int32),
                ("flags", C.c_int32)]


class moe_workspace_views_t(C.Structure):
    _fields_ = [("topk_ids", C.c_size_t), ("topk_weights", C.c_size_t), ("sorted_ids", C.c_size_t),
                ("block_expert_ids", C.c_size_t), ("num_post_pad", C.c_size_t),
                ("expert_offsets", C.c_size_t)]


class moe_expert_weights_t(C.Structure):
    _fields_ = [("gate_up", C.c_void_p), ("gate_up_scales", C.c_void_p), ("down", C.c_void_p),
                ("down_scales", C.c_void_p)]


class moe_shared_weights_t(C.Structure):
    _fields_ = [("gate_up", C.c_void_p), ("down", C.c_void_p), ("gate_w", C.c_void_p)]


_lib = None
_P = C.c_void_p
_D = C.POINTER(moe_dims_t)


def load():
    """Load libmoe_gb300.so (built in-tree by build.py).  Raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    L = C.CDLL(LIB_PATH)
    L.moe_status_string.argtypes = [C.c_int]
    L.moe_status_string.restype = C.c_char_p
    L.moe_workspace_bytes.argtypes = [_D, C.POINTER(C.c_size_t)]
    L.moe_workspace_init.argtypes = [_P, C.c_size_t, _P]
    L.moe_workspace_views.argtypes = [_D, C.POINTER(moe_workspace_views_t)]
    L.moe_workspace_inject_stall.argtypes = [_P, C.c_size_t, C.c_uint32, _P]
    L.moe_route.argtypes = [_D, _P, _P, _P, _P, _P, C.c_size_t, _P]
    L.moe_align_block_size.argtypes = [_D, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]
    L.moe_expert_forward.argtypes = [_D, _P, _P, _P, _P, _P, _P, C.POINTER(moe_expert_weights_t),
                                     C.POINTER(moe_shared_weights_t), _P, _P, C.c_size_t, _P]
    L.moe_layer_forward.argtypes = [_D, _P, _P, C.POINTER(moe_expert_weights_t),
                                    C.POINTER(moe_shared_weights_t), _P, _P, _P, _P, C.c_size_t, _P]
    L.moe_layer_forward_timed.argtypes = L.moe_layer_forward.argtypes + [C.POINTER(C.c_void_p)]
    L.moe_layer_forward_static.argtypes = [_D, _P, _P, C.POINTER(moe_expert_weights_t),
                                           C.POINTER(moe_shared_weights_t), _P, _P, _P, _P, _P]
    L.moe_read_device_status.argtypes = [_P, C.POINTER(C.c_int32), _P]
    L.moe_kernel_launch_count.argtypes = []
    L.moe_kernel_launch_count.restype = C.c_uint64
    for name in EXPORTS:
        if name not in ("moe_status_string", "moe_kernel_launch_count"):
            getattr(L, name).restype = C.c_int
    _lib = L
    return L


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where, load().moe_status_string(status).decode())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_dims(T, d, E, top_k, I, I_shared=0, renormalize=True, block_size=16,
              weight_format=MOE_WEIGHTS_BF16, group_size=32, flags=0) -> moe_dims_t:
    return moe_dims_t(int(T), int(d), int(E), int(top_k), int(I), int(I_shared),
                      int(bool(renormalize)), int(block_size), int(weight_format), int(group_size),
                      int(flags))


def dims_of(shape, flags=0) -> moe_dims_t:
    """moe_dims_t of an inputs.LayerShape."""
    fmt = MOE_WEIGHTS_INT4_G32 if shape.fmt == "int4" else MOE_WEIGHTS_BF16
    return make_dims(shape.T, shape.d, shape.E, shape.k, shape.I, shape.Is, shape.renormalize,
                     shape.block, fmt, shape.group, flags)


def expert_weights(gate_up, down, gate_up_scales=None, down_scales=None) -> moe_expert_weights_t:
    return moe_expert_weights_t(_ptr(gate_up), _ptr(gate_up_scales), _ptr(down), _ptr(down_scales))


def shared_weights(gate_up, down, gate_w) -> moe_shared_weights_t:
    return moe_shared_weights_t(_ptr(gate_up), _ptr(down), _ptr(gate_w))


def moe_status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def moe_workspace_bytes(dims: moe_dims_t) -> int:
    n = C.c_size_t(0)
    _check(load().moe_workspace_bytes(C.byref(dims), C.byref(n)), "moe_workspace_bytes")
    return int(n.value)


def moe_workspace_init(ws, nbytes: int, stream=None):
    _check(load().moe_workspace_init(_ptr(ws), int(nbytes), _stream(stream)), "moe_workspace_init")


def moe_workspace_views(dims: moe_dims_t) -> dict:
    """Byte offsets of the routing and align layout inside a workspace."""
    v = moe_workspace_views_t()
    _check(load().moe_workspace_views(C.byref(dims), C.byref(v)), "moe_workspace_views")
    return {name: int(getattr(v, name)) for name, _ in moe_workspace_views_t._fields_}


def moe_workspace_inject_stall(ws, nbytes: int, wait_limit_us: int, stream=None):
    _check(load().moe_workspace_inject_stall(_ptr(ws), int(nbytes), int(wait_limit_us),
                                             _stream(stream)), "moe_workspace_inject_stall")


def alloc_workspace(dims: moe_dims_t, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace tensor (torch's allocator aligns to 512 B)."""
    n = moe_workspace_bytes(dims)
    ws = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    moe_workspace_init(ws, ws.numel())
    return ws


def moe_route(dims, x, router_w, topk_ids, topk_weights, ws, stream=None):
    _check(load().moe_route(C.byref(dims), _ptr(x), _ptr(router_w), _ptr(topk_ids),
                            _ptr(topk_weights), _ptr(ws), ws.numel(), _stream(stream)), "moe_route")


def moe_align_block_size(dims, topk_ids, sorted_ids, block_expert_ids, num_post_pad,
                         expert_offsets, ws, stream=None):
    _check(load().moe_align_block_size(C.byref(dims), _ptr(topk_ids), _ptr(sorted_ids),
                                       _ptr(block_expert_ids), _ptr(num_post_pad),
                                       _ptr(expert_offsets), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_align_block_size")


def moe_expert_forward(dims, x, topk_weights, sorted_ids, block_expert_ids, num_post_pad,
                       expert_offsets, experts: moe_expert_weights_t, shared, out, ws, stream=None):
    sh = C.byref(shared) if shared is not None else None
    _check(load().moe_expert_forward(C.byref(dims), _ptr(x), _ptr(topk_weights), _ptr(sorted_ids),
                                     _ptr(block_expert_ids), _ptr(num_post_pad),
                                     _ptr(expert_offsets), C.byref(experts), sh, _ptr(out),
                                     _ptr(ws), ws.numel(), _stream(stream)), "moe_expert_forward")


def moe_layer_forward(dims, x, router_w, experts: moe_expert_weights_t, shared, out,
                      topk_ids_out=None, topk_weights_out=None, ws=None, stream=None):
    sh = C.byref(shared) if shared is not None else None
    _check(load().moe_layer_forward(C.byref(dims), _ptr(x), _ptr(router_w), C.byref(experts), sh,
                                    _ptr(out), _ptr(topk_ids_out), _ptr(topk_weights_out),
                                    _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_timed(dims, x, router_w, experts, shared, out, topk_ids_out, topk_weights_out,
                            ws, events, stream=None):
    """events: a list of MOE_EV_COUNT torch.cuda.Event(enable_timing=True) or None."""
    for e in events:
        if e is not None and not e.cuda_event:
            e.record()  # torch creates the underlying cudaEvent_t on first record
    arr = (C.c_void_p * MOE_EV_COUNT)(*[None if e is None else e.cuda_event for e in events])
    sh = C.byref(shared) if shared is not None else None
    _check(load().moe_layer_forward_timed(C.byref(dims), _ptr(x), _ptr(router_w), C.byref(experts),
                                          sh, _ptr(out), _ptr(topk_ids_out), _ptr(topk_weights_out),
                                          _ptr(ws), ws.numel(), _stream(stream), arr),
           "moe_layer_forward_timed")


def moe_layer_forward_static(dims, x, router_w, experts, shared, out, topk_ids_out=None,
                             topk_weights_out=None, device_status_out=None, stream=None):
    """The layer with the library's own static scratch: no workspace argument,
    nothing allocated (for callers that may not allocate device memory)."""
    sh = C.byref(shared) if shared is not None else None
    _check(load().moe_layer_forward_static(C.byref(dims), _ptr(x), _ptr(router_w), C.byref(experts),
                                           sh, _ptr(out), _ptr(topk_ids_out),
                                           _ptr(topk_weights_out), _ptr(device_status_out),
                                           _stream(stream)), "moe_layer_forward_static")


def moe_read_device_status(ws, stream=None) -> int:
    code = C.c_int32(0)
    _check(load().moe_read_device_status(_ptr(ws), C.byref(code), _stream(stream)),
           "moe_read_device_status")
    return int(code.value)


def moe_kernel_launch_count() -> int:
    return int(load().moe_kernel_launch_count())
