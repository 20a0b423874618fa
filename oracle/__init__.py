"""fp64 CPU oracle of the sparse-MoE expert layer -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It never imports, links or calls the CUDA library,
and the CUDA library never calls it.

Thin ctypes wrappers around ``libmoe_oracle.so`` (``moe_oracle.c``); numpy in,
numpy out.  bf16 tensors travel as their raw uint16 bit patterns and are decoded
exactly inside the C code.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


class Dims(C.Structure):
    _fields_ = [("T", C.c_int32), ("d", C.c_int32), ("E", C.c_int32), ("k", C.c_int32),
                ("I", C.c_int32), ("Is", C.c_int32), ("renormalize", C.c_int32)]


class Experts(C.Structure):
    _fields_ = [("format", C.c_int32), ("group", C.c_int32), ("gate_up", C.c_void_p),
                ("gate_up_scales", C.c_void_p), ("down", C.c_void_p), ("down_scales", C.c_void_p),
                ("gate_up_global", C.c_void_p), ("down_global", C.c_void_p)]


class Shared(C.Structure):
    _fields_ = [("gate_up", C.c_void_p), ("down", C.c_void_p), ("gate_w", C.c_void_p)]


BF16, INT4, F64, FP8, NVFP4 = 0, 1, 2, 3, 4

_P = C.c_void_p


def _declare(L):
    L.moe_oracle_bf16_to_f64.argtypes = [C.c_uint16]
    L.moe_oracle_bf16_to_f64.restype = C.c_double
    L.moe_oracle_decode_bf16.argtypes = [C.c_size_t, _P, _P]
    L.moe_oracle_decode_bf16.restype = None
    L.moe_oracle_dequant_int4.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P]
    L.moe_oracle_e4m3_to_f64.argtypes = [C.c_uint8]
    L.moe_oracle_e4m3_to_f64.restype = C.c_double
    L.moe_oracle_e2m1_to_f64.argtypes = [C.c_uint8]
    L.moe_oracle_e2m1_to_f64.restype = C.c_double
    L.moe_oracle_dequant_fp8.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P]
    L.moe_oracle_dequant_nvfp4.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, C.c_float, _P]
    L.moe_oracle_router_logits.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P]
    L.moe_oracle_router_logits.restype = None
    L.moe_oracle_topk.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P]
    L.moe_oracle_weights_for_ids.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int32, _P, _P, _P]
    L.moe_oracle_align.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P]
    L.moe_oracle_swiglu_expert.argtypes = [C.c_int32, C.c_int32, _P, _P, _P, _P]
    L.moe_oracle_swiglu_expert.restype = None
    L.moe_oracle_combine.argtypes = [C.c_int32, C.c_int32, C.c_int32, _P, _P, _P, _P, _P]
    L.moe_oracle_combine.restype = None
    L.moe_oracle_layer.argtypes = [C.POINTER(Dims), _P, _P, C.POINTER(Experts), C.POINTER(Shared),
                                   _P, _P, C.c_int32, _P, _P, _P, _P, _P, C.c_int32]
    L.moe_oracle_max_threads.argtypes = []


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return int(lib().moe_oracle_max_threads())


def decode_bf16(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    lib().moe_oracle_decode_bf16(bits.size, _ptr(bits), _ptr(out))
    return out


def dequant_int4(codes, scales, cols: int, group: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    rows = codes.size // (cols // 2)
    out = np.empty((rows, cols), np.float64)
    rc = lib().moe_oracle_dequant_int4(rows, cols, group, _ptr(codes), _ptr(scales), _ptr(out))
    if rc:
        raise ValueError(f"moe_oracle_dequant_int4 failed ({rc})")
    return out.reshape(codes.shape[:-1] + (cols,))


def e4m3_to_f64(b: int) -> float:
    return float(lib().moe_oracle_e4m3_to_f64(int(b)))


def e2m1_to_f64(code: int) -> float:
    return float(lib().moe_oracle_e2m1_to_f64(int(code)))


def dequant_fp8(codes, scales, cols: int, group: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    rows = codes.size // cols
    out = np.empty((rows, cols), np.float64)
    rc = lib().moe_oracle_dequant_fp8(rows, cols, group, _ptr(codes), _ptr(scales), _ptr(out))
    if rc:
        raise ValueError(f"moe_oracle_dequant_fp8 failed ({rc})")
    return out.reshape(codes.shape[:-1] + (cols,))


def dequant_nvfp4(codes, scales, global_scale: float, cols: int, group: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    rows = codes.size // (cols // 2)
    out = np.empty((rows, cols), np.float64)
    rc = lib().moe_oracle_dequant_nvfp4(rows, cols, group, _ptr(codes), _ptr(scales),
                                        float(global_scale), _ptr(out))
    if rc:
        raise ValueError(f"moe_oracle_dequant_nvfp4 failed ({rc})")
    return out.reshape(codes.shape[:-1] + (cols,))


def router_logits(x, wr) -> np.ndarray:
    x = _c(x, np.float64)
    wr = _c(wr, np.float64)
    T, d = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    lib().moe_oracle_router_logits(T, d, E, _ptr(x), _ptr(wr), _ptr(out))
    return out


def topk(logits, k: int, renormalize: bool = True):
    """Return ids int32[T,k], w f64[T,k], margin f64[T], probs f64[T,E]."""
    logits = _c(logits, np.float64)
    T, E = logits.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    margin = np.empty((T,), np.float64)
    probs = np.empty((T, E), np.float64)
    rc = lib().moe_oracle_topk(T, E, k, int(renormalize), _ptr(logits), _ptr(ids), _ptr(w),
                               _ptr(margin), _ptr(probs))
    if rc:
        raise ValueError(f"moe_oracle_topk failed ({rc})")
    return ids, w, margin, probs


def weights_for_ids(logits, ids, renormalize: bool = True) -> np.ndarray:
    logits = _c(logits, np.float64)
    ids = _c(ids, np.int32)
    T, E = logits.shape
    k = ids.shape[1]
    w = np.empty((T, k), np.float64)
    rc = lib().moe_oracle_weights_for_ids(T, E, k, int(renormalize), _ptr(logits), _ptr(ids), _ptr(w))
    if rc:
        raise ValueError(f"moe_oracle_weights_for_ids failed ({rc})")
    return w


def align_capacity(S: int, E: int, B: int) -> int:
    return S + E * (B - 1)


def align(ids_flat, E: int, B: int) -> dict:
    ids_flat = _c(ids_flat, np.int32).reshape(-1)
    S = ids_flat.size
    cap = align_capacity(S, E, B)
    sorted_ids = np.full((cap,), -1, np.int32)
    block_ids = np.full((cap // B + 1,), -1, np.int32)
    npp = np.zeros((1,), np.int32)
    offs = np.empty((E + 1,), np.int32)
    counts = np.empty((E,), np.int32)
    rc = lib().moe_oracle_align(S, E, B, _ptr(ids_flat), _ptr(sorted_ids), _ptr(block_ids),
                                _ptr(npp), _ptr(offs), _ptr(counts))
    if rc:
        raise ValueError(f"moe_oracle_align failed ({rc})")
    n = int(npp[0])
    return {"sorted_ids": sorted_ids[:n].copy(), "block_expert_ids": block_ids[: n // B].copy(),
            "num_post_pad": n, "expert_offsets": offs, "counts": counts}


def swiglu_expert(x, wgu, wd) -> np.ndarray:
    x = _c(x, np.float64)
    wgu = _c(wgu, np.float64)
    wd = _c(wd, np.float64)
    d = x.shape[0]
    I = wgu.shape[0] // 2
    y = np.empty((d,), np.float64)
    lib().moe_oracle_swiglu_expert(d, I, _ptr(x), _ptr(wgu), _ptr(wd), _ptr(y))
    return y


def combine(w, y, sg_logit=None, ys=None) -> np.ndarray:
    """w f64[T,k], y f64[T*k,d], sg_logit f64[T] | None, ys f64[T,d] | None."""
    w = _c(w, np.float64)
    T, k = w.shape
    y = _c(y, np.float64).reshape(T * k, -1)
    d = y.shape[1]
    if ys is not None:
        ys = _c(ys, np.float64)
        sg_logit = _c(sg_logit, np.float64)
    out = np.empty((T, d), np.float64)
    lib().moe_oracle_combine(T, k, d, _ptr(w), _ptr(y), _ptr(sg_logit), _ptr(ys), _ptr(out))
    return out


def layer(x_bits, router_bits, experts: dict, shared, dims: dict, ids_override=None,
          tokens=None, nthreads: int = 0) -> dict:
    """Full layer.

    x_bits uint16[T,d]; router_bits uint16[E,d].
    experts: {"format": BF16|INT4|F64|FP8|NVFP4, "group": g, "gate_up": arr, "down": arr,
              "gate_up_scales": arr|None, "down_scales": arr|None,
              "gate_up_global": f32[E]|None, "down_global": f32[E]|None (NVFP4)}
    shared:  None or {"gate_up": uint16[2Is,d], "down": uint16[d,Is], "gate_w": uint16[d]}
    dims:    {"T","d","E","k","I","Is","renormalize"}
    Returns {"out": f64[n,d], "ids", "w", "margin", "sg"} for the listed tokens.
    """
    fmt = experts.get("format", BF16)
    dt = {BF16: np.uint16, INT4: np.uint8, F64: np.float64, FP8: np.uint8, NVFP4: np.uint8}[fmt]
    st = np.uint8 if fmt == NVFP4 else np.uint16  # E4M3 block scales, else bf16
    gu = _c(experts["gate_up"], dt)
    dn = _c(experts["down"], dt)
    gus = None if experts.get("gate_up_scales") is None else _c(experts["gate_up_scales"], st)
    dns = None if experts.get("down_scales") is None else _c(experts["down_scales"], st)
    gug = None if experts.get("gate_up_global") is None else _c(experts["gate_up_global"],
                                                                np.float32)
    dng = None if experts.get("down_global") is None else _c(experts["down_global"], np.float32)
    ex = Experts(fmt, int(experts.get("group", 0)), _ptr(gu), _ptr(gus), _ptr(dn), _ptr(dns),
                 _ptr(gug), _ptr(dng))
    x_bits = _c(x_bits, np.uint16)
    router_bits = _c(router_bits, np.uint16)
    dm = Dims(dims["T"], dims["d"], dims["E"], dims["k"], dims["I"],
              dims.get("Is", 0) if shared is not None else 0, int(dims.get("renormalize", 1)))
    keep = [gu, dn, gus, dns, gug, dng]
    sh_ptr = None
    if shared is not None:
        sgu = _c(shared["gate_up"], np.uint16)
        sdn = _c(shared["down"], np.uint16)
        sgw = _c(shared["gate_w"], np.uint16)
        keep += [sgu, sdn, sgw]
        sh = Shared(_ptr(sgu), _ptr(sdn), _ptr(sgw))
        sh_ptr = C.pointer(sh)
    ov = None if ids_override is None else _c(ids_override, np.int32)
    tl = None if tokens is None else _c(tokens, np.int32)
    n = dims["T"] if tl is None else tl.size
    k = dims["k"]
    out = np.empty((n, dims["d"]), np.float64)
    ids = np.empty((n, k), np.int32)
    w = np.empty((n, k), np.float64)
    margin = np.empty((n,), np.float64)
    sg = np.empty((n,), np.float64)
    rc = lib().moe_oracle_layer(C.byref(dm), _ptr(x_bits), _ptr(router_bits), C.byref(ex), sh_ptr,
                                _ptr(ov), _ptr(tl), n, _ptr(out), _ptr(ids), _ptr(w), _ptr(margin),
                                _ptr(sg), int(nthreads))
    del keep
    if rc:
        raise ValueError(f"moe_oracle_layer failed ({rc})")
    return {"out": out, "ids": ids, "w": w, "margin": margin, "sg": sg}
