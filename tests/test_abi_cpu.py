"""CPU tier of the C ABI: the library builds for sm_103a, loads without a GPU,
exports every entry point include/moe.h declares, and rejects bad arguments on
the host before launching anything (no CUDA call is reached by these cases)."""
import ctypes as C
import os
import re

import pytest

from moe_expert_layer_gemv_gb300 import abi, build
from moe_expert_layer_gemv_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return abi.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(names) == set(abi.EXPORTS), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert C.cast(getattr(lib, name), C.c_void_p).value


def test_status_strings(lib):
    for code in range(7):
        assert abi.moe_status_string(code).startswith("MOE_")
    assert abi.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_workspace_bytes_and_dims_validation(lib):
    d8 = abi.dims_of(I.shape("verify_t8"))
    n8 = abi.moe_workspace_bytes(d8)
    n64 = abi.moe_workspace_bytes(abi.dims_of(I.shape("verify_t64")))
    assert 0 < n8 < n64
    assert n8 % 256 == 0
    bad = [abi.make_dims(8, 2047, 256, 8, 512),        # d % 8
           abi.make_dims(8, 2048, 2048, 8, 512),       # E > 1024
           abi.make_dims(8, 2048, 8, 9, 512),          # k > E
           abi.make_dims(8, 2048, 64, 17, 512),        # k > 16
           abi.make_dims(8, 2048, 64, 8, 100),         # I % 8
           abi.make_dims(8, 2048, 64, 8, 512, weight_format=1, group_size=64),  # int4 group
           abi.make_dims(8, 2048 + 8, 64, 8, 512, weight_format=1),  # int4 needs d % 256
           abi.make_dims(8, 2048, 64, 8, 512, block_size=2048)]
    for dm in bad:
        with pytest.raises(abi.MoeError) as e:
            abi.moe_workspace_bytes(dm)
        assert e.value.status == abi.MOE_ERR_UNSUPPORTED
    with pytest.raises(abi.MoeError) as e:
        abi.moe_workspace_bytes(abi.make_dims(-1, 2048, 64, 8, 512))
    assert e.value.status == abi.MOE_ERR_INVALID_ARG
    n = C.c_size_t(7)
    assert lib.moe_workspace_bytes(None, C.byref(n)) == abi.MOE_ERR_INVALID_ARG and n.value == 0


FAKE = 1 << 40  # an aligned, never-dereferenced address: these calls stop before any launch


def _layer(lib, dims, ws=FAKE, ws_bytes=1 << 40, x=FAKE, shared=True, out=FAKE, ex=None):
    ex = ex or abi.moe_expert_weights_t(FAKE, None, FAKE, None)
    sh = abi.moe_shared_weights_t(FAKE, FAKE, FAKE) if shared else None
    return lib.moe_layer_forward(C.byref(dims), x, FAKE, C.byref(ex),
                                 C.byref(sh) if sh is not None else None, out, None, None, ws,
                                 ws_bytes, None)


def test_layer_forward_host_side_rejections(lib):
    dims = abi.dims_of(I.shape("verify_t8"))
    need = abi.moe_workspace_bytes(dims)
    assert _layer(lib, dims, x=None) == abi.MOE_ERR_INVALID_ARG
    assert _layer(lib, dims, x=FAKE + 2) == abi.MOE_ERR_INVALID_ARG          # misaligned
    assert _layer(lib, dims, out=None) == abi.MOE_ERR_INVALID_ARG
    assert _layer(lib, dims, shared=False) == abi.MOE_ERR_INVALID_ARG         # I_shared > 0
    assert _layer(lib, dims, ws=None) == abi.MOE_ERR_WORKSPACE
    assert _layer(lib, dims, ws=FAKE + 16) == abi.MOE_ERR_WORKSPACE           # not 256-aligned
    assert _layer(lib, dims, ws_bytes=need - 1) == abi.MOE_ERR_WORKSPACE
    assert _layer(lib, dims, ex=abi.moe_expert_weights_t(FAKE, None, None, None)) == \
        abi.MOE_ERR_INVALID_ARG
    d4 = abi.dims_of(I.shape("int4_t32"))
    assert _layer(lib, d4, ex=abi.moe_expert_weights_t(FAKE, None, FAKE, None)) == \
        abi.MOE_ERR_INVALID_ARG                                                # scales missing
    assert lib.moe_layer_forward(None, FAKE, FAKE, None, None, FAKE, None, None, FAKE, 1, None) == \
        abi.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_timed(C.byref(dims), FAKE, FAKE, None, None, FAKE, None, None,
                                       FAKE, need, None, None) == abi.MOE_ERR_INVALID_ARG


def test_stage_calls_host_side_rejections(lib):
    dims = abi.dims_of(I.shape("verify_t8"))
    need = abi.moe_workspace_bytes(dims)
    assert lib.moe_route(C.byref(dims), FAKE, FAKE, None, FAKE, FAKE, need, None) == \
        abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(C.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, need - 256, None) == \
        abi.MOE_ERR_WORKSPACE
    assert lib.moe_align_block_size(C.byref(dims), FAKE, FAKE, FAKE, None, FAKE, FAKE, need,
                                    None) == abi.MOE_ERR_INVALID_ARG
    ex = abi.moe_expert_weights_t(FAKE, None, FAKE, None)
    sh = abi.moe_shared_weights_t(FAKE, FAKE, FAKE)
    assert lib.moe_expert_forward(C.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, C.byref(ex),
                                  C.byref(sh), FAKE, FAKE, 16, None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_workspace_init(None, 1024, None) == abi.MOE_ERR_WORKSPACE
    code = C.c_int32(0)
    assert lib.moe_read_device_status(None, C.byref(code), None) == abi.MOE_ERR_INVALID_ARG


def test_workspace_views_point_inside_the_workspace(lib):
    for name in ("tiny", "verify_t8", "verify_t64", "int4_t32", "prefill_t4096"):
        s = I.shape(name)
        dims = abi.dims_of(s)
        need = abi.moe_workspace_bytes(dims)
        v = abi.moe_workspace_views(dims)
        S = s.T * s.k
        cap = S + s.E * (s.block - 1)
        sizes = {"topk_ids": 4 * S, "topk_weights": 4 * S, "sorted_ids": 4 * cap,
                 "block_expert_ids": 4 * (cap // s.block + 1), "num_post_pad": 4,
                 "expert_offsets": 4 * (s.E + 1)}
        spans = sorted((v[k], v[k] + n) for k, n in sizes.items())
        for (a0, a1), (b0, _) in zip(spans, spans[1:]):
            assert a1 <= b0  # disjoint
        assert all(off % 256 == 0 for off in v.values())
        assert spans[0][0] >= 256 and spans[-1][1] <= need  # past the header, inside
    vv = abi.moe_workspace_views_t()
    assert lib.moe_workspace_views(None, C.byref(vv)) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_views(C.byref(abi.dims_of(I.shape("tiny"))), None) == \
        abi.MOE_ERR_INVALID_ARG


def test_flags_and_stall_hook_host_checks(lib):
    dims = abi.dims_of(I.shape("verify_t8"), flags=abi.MOE_FLAG_BATCH_INVARIANT)
    assert abi.moe_workspace_bytes(dims) > 0
    with pytest.raises(abi.MoeError) as e:
        abi.moe_workspace_bytes(abi.dims_of(I.shape("verify_t8"), flags=2))
    assert e.value.status == abi.MOE_ERR_UNSUPPORTED
    assert lib.moe_workspace_inject_stall(None, 1024, 100, None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_workspace_inject_stall(FAKE + 16, 1024, 100, None) == abi.MOE_ERR_WORKSPACE
    assert lib.moe_workspace_inject_stall(FAKE, 1024, 0, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_inject_stall(FAKE, 1024, 2000000, None) == abi.MOE_ERR_INVALID_ARG


def test_static_entry_point_host_checks_launch_nothing(lib):
    dims = abi.dims_of(I.shape("verify_t8"))
    ex = abi.moe_expert_weights_t(FAKE, None, FAKE, None)
    sh = abi.moe_shared_weights_t(FAKE, FAKE, FAKE)
    assert lib.moe_layer_forward_static(C.byref(dims), None, FAKE, C.byref(ex), C.byref(sh), FAKE,
                                        None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    assert lib.moe_layer_forward_static(C.byref(dims), FAKE, FAKE, C.byref(ex), None, FAKE,
                                        None, None, None, None) == abi.MOE_ERR_INVALID_ARG
    big = abi.dims_of(I.shape("prefill_t4096"))
    assert lib.moe_layer_forward_static(C.byref(big), FAKE, FAKE, C.byref(ex), C.byref(sh), FAKE,
                                        None, None, None, None) == abi.MOE_ERR_WORKSPACE
    zero = abi.dims_of(I.shape("verify_t8", T=0))
    assert lib.moe_layer_forward_static(C.byref(zero), None, None, None, None, None, None, None,
                                        None, None) == abi.MOE_OK
    assert abi.moe_kernel_launch_count() == 0


def test_launch_counter_starts_at_zero_without_launches(lib):
    assert abi.moe_kernel_launch_count() == 0


def test_header_is_plain_c_and_links_against_the_library(lib, tmp_path):
    """A C99 program that includes moe.h compiles with warnings as errors, links
    against libmoe_gb300.so, and gets host-side answers without a GPU."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_moe.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "moe.h"

int main(void) {
  moe_dims_t d;
  size_t n = 0;
  memset(&d, 0, sizeof d);
  d.T = 8; d.d = 2048; d.E = 256; d.top_k = 8; d.I = 512; d.I_shared = 512;
  d.renormalize = 1; d.block_size = 16; d.weight_format = MOE_WEIGHTS_BF16; d.group_size = 32;
  d.flags = MOE_FLAG_BATCH_INVARIANT;
  if (moe_workspace_bytes(&d, &n) != MOE_OK || n == 0) return 1;
  d.top_k = 0;
  if (moe_workspace_bytes(&d, &n) == MOE_OK) return 2;
  if (moe_layer_forward(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL) == MOE_OK)
    return 3;
  {
    moe_workspace_views_t v;
    d.top_k = 8;
    if (moe_workspace_views(&d, &v) != MOE_OK || v.sorted_ids == 0 || v.expert_offsets == 0)
      return 4;
  }
  printf("%s|%s\n", moe_status_string(MOE_OK), moe_status_string(MOE_ERR_INVALID_ARG));
  return 0;
}
''')
    exe = tmp_path / "use_moe"
    so = abi.LIB_PATH
    p = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        so, "-Wl,-rpath," + os.path.dirname(so)],
                       capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    ok, bad = r.stdout.strip().split("|")
    assert ok and bad and ok != bad
