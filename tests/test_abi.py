"""The C-ABI library builds, loads and exports every entry point include/tb.h declares (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "tb.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"TB_API\s+[\w\s\*]*?\b(tb_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib_path():
    from predicted_token_importance_tb_b300 import build
    return build.build()


def test_header_declares_entry_points():
    names = _declared()
    for n in ["tb_project_append", "tb_score", "tb_topk", "tb_sparse_decode_attn", "tb_decode_step"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], check=True, capture_output=True, text=True).stdout
    exported = set(re.findall(r"\sT\s(tb_\w+)$", out, re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(lib_path)
    for n in _declared():
        assert hasattr(lib, n)


def test_binding_loads_and_reports(lib_path):
    import predicted_token_importance_tb_b300 as tb
    lib = tb.load_library()
    assert lib.tb_version() == 1
    assert tb.status_string(tb.TB_ERR_WORKSPACE) == "workspace missing or too small"
    for n in tb.EXPORTED:
        assert n in _declared()


def test_host_validation_without_gpu(lib_path):
    # Argument checks run before any CUDA call, so they answer on a CPU-only host.
    import predicted_token_importance_tb_b300 as tb
    lib = tb.load_library()
    bad = tb.Shape(1, 6, 4, 128, 32, 100).c()       # Hq not a multiple of Hkv
    sz = ctypes.c_size_t(0)
    assert lib.tb_workspace_size(ctypes.byref(bad), 10, 4, 4, ctypes.byref(sz)) == tb.TB_ERR_INVALID_ARG
    odd = tb.Shape(1, 8, 8, 60, 16, 100).c()        # D not a multiple of 8
    assert lib.tb_workspace_size(ctypes.byref(odd), 10, 4, 4, ctypes.byref(sz)) == tb.TB_ERR_UNSUPPORTED
    ok = tb.Shape(1, 32, 8, 128, 32, 32768).c()
    assert lib.tb_workspace_size(ctypes.byref(ok), 32767, 3277, 3277, ctypes.byref(sz)) == tb.TB_OK
    assert sz.value > 0
    # k > n is rejected before launch; so is a missing workspace
    assert lib.tb_topk(ctypes.byref(ok), ctypes.c_void_p(16), 10, 11, ctypes.c_void_p(16), None, 0, None,
                       None) == tb.TB_ERR_INVALID_ARG
    assert lib.tb_topk(ctypes.byref(ok), ctypes.c_void_p(16), 10, 5, ctypes.c_void_p(16), None, 0, None,
                       None) == tb.TB_ERR_WORKSPACE


def test_host_validation_of_the_newer_calls(lib_path):
    # the buffered step and the predictor check their arguments before any CUDA call
    import predicted_token_importance_tb_b300 as tb
    lib = tb.load_library()
    fake = ctypes.c_void_p(1 << 20)              # aligned, never dereferenced: the checks fail first
    sp = tb.Shape(1, 8, 2, 64, 16, 1000).c()
    params = tb._StepParams(10, 1, 0, 0, 0.125, 0)
    i64 = ctypes.c_int64
    n_pred, proj_end = i64(0), i64(0)
    for sink, window, want in [(4, 0, tb.TB_ERR_INVALID_ARG), (-1, 8, tb.TB_ERR_INVALID_ARG)]:
        bufs = tb._BufferParams(sink, window)
        st = lib.tb_decode_step_buffered(ctypes.byref(sp), ctypes.byref(params), ctypes.byref(bufs), 0, 100,
                                         fake, fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(n_pred),
                                         ctypes.byref(proj_end), fake, 64, fake, fake, fake, 1 << 30, None, None)
        assert st == want
    proj_end.value = 500                         # more rows projected than tokens
    bufs = tb._BufferParams(4, 8)
    st = lib.tb_decode_step_buffered(ctypes.byref(sp), ctypes.byref(params), ctypes.byref(bufs), 0, 100,
                                     fake, fake, fake, fake, fake, fake, fake, fake, fake, ctypes.byref(n_pred),
                                     ctypes.byref(proj_end), fake, 64, fake, fake, fake, 1 << 30, None, None)
    assert st == tb.TB_ERR_INVALID_ARG
    bad_flags = tb._StepParams(10, 1, 0, 0, 0.125, 64)
    st = lib.tb_decode_step(ctypes.byref(sp), ctypes.byref(bad_flags), 0, 100, fake, fake, fake, fake, fake, fake,
                            fake, fake, fake, ctypes.byref(n_pred), fake, 64, fake, fake, fake, 1 << 30, None, None)
    assert st == tb.TB_ERR_INVALID_ARG
    # predictor: too many tokens, a width that is not a multiple of 8, a workspace too small
    assert lib.tb_predict_queries(fake, fake, fake, 17, 64, 32, 16, fake, fake, 1 << 20, None, None) == \
        tb.TB_ERR_UNSUPPORTED
    assert lib.tb_predict_queries(fake, fake, fake, 2, 60, 32, 16, fake, fake, 1 << 20, None, None) == \
        tb.TB_ERR_UNSUPPORTED
    assert lib.tb_predict_queries(fake, fake, fake, 2, 64, 32, 16, fake, fake, 16, None, None) == \
        tb.TB_ERR_WORKSPACE


def test_binding_refuses_tensors_shorter_than_the_call_touches(lib_path):
    # The Python binding compares every tensor's extent with what the call
    # reads or writes before marshalling any pointer, so a short tensor is a
    # ValueError on the host (CPU tensors suffice: the check comes first).
    import torch
    import predicted_token_importance_tb_b300 as tb
    B, Hq, Hkv, D, dp, cap = 1, 4, 2, 64, 16, 128
    shape = tb.Shape(B, Hq, Hkv, D, dp, cap)
    bf = torch.bfloat16

    def z(n, dtype=bf):
        return torch.zeros(n, dtype=dtype)

    K, V, Kp, Wk = z(B * Hkv * cap * D), z(B * Hkv * cap * D), z(B * Hkv * cap * dp), z(Hkv * D * dp)
    with pytest.raises(ValueError, match="K_src"):
        tb.tb_project_append(shape, z(B * Hkv * cap * D - 1), cap, Wk, Kp, 0, cap)
    with pytest.raises(ValueError, match="K_src"):   # rows from an offset past the end
        tb.tb_project_append(shape, K, cap, Wk, Kp, 5, cap, K_src_offset_rows=5)
    with pytest.raises(ValueError, match="Wk"):
        tb.tb_project_append(shape, K, cap, z(Hkv * D * dp - 8), Kp, 0, cap)
    with pytest.raises(ValueError, match="Kp"):
        tb.tb_project_append(shape, K, cap, Wk, z(B * Hkv * cap * dp - 1), 0, cap)
    with pytest.raises(ValueError, match="^s "):
        tb.tb_score(shape, z(B * Hq * dp), Kp, cap, z(B * Hkv * cap - 1, torch.float32))
    with pytest.raises(ValueError, match="Kp"):
        tb.tb_score(shape, z(B * Hq * dp), z(B * Hkv * cap * dp - 1), cap, z(B * Hkv * cap, torch.float32))
    with pytest.raises(ValueError, match="idx"):
        tb.tb_topk(shape, z(B * Hkv * cap, torch.float32), cap, 10, z(B * Hkv * 10 - 1, torch.int32), z(1, torch.uint8))
    with pytest.raises(ValueError, match="sel"):
        tb.tb_expand(shape, z(B * Hkv * 4, torch.int32), 4, 1, cap, cap, z(B * Hkv * 12 - 1, torch.int32), 12,
                     z(B * Hkv, torch.int32))
    with pytest.raises(ValueError, match="^V "):
        tb.tb_sparse_decode_attn(shape, z(B * Hq * D), K, z(B * Hkv * cap * D - 1), z(B * Hkv * 8, torch.int32),
                                 None, 8, 0.125, z(B * Hq * D), z(1, torch.uint8))
    with pytest.raises(ValueError, match="out"):
        tb.tb_decode_step(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, cap - 1, q=z(B * Hq * D), q_imp=z(B * Hq * dp),
                          K_new=z(B * Hkv * D), V_new=z(B * Hkv * D), Wk=Wk, K=K, V=V, Kp=Kp,
                          idx_state=z(B * Hkv * 8, torch.int32), n_pred=ctypes.c_int64(0),
                          sel=z(B * Hkv * 8, torch.int32), sel_stride=8, counts=z(B * Hkv, torch.int32),
                          out=z(B * Hq * D - 1), ws=z(1, torch.uint8))
    with pytest.raises(ValueError, match="idx_state"):
        tb.tb_decode_step(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, cap - 1, q=z(B * Hq * D), q_imp=z(B * Hq * dp),
                          K_new=z(B * Hkv * D), V_new=z(B * Hkv * D), Wk=Wk, K=K, V=V, Kp=Kp,
                          idx_state=z(B * Hkv * 8 - 1, torch.int32), n_pred=ctypes.c_int64(0),
                          sel=z(B * Hkv * 8, torch.int32), sel_stride=8, counts=z(B * Hkv, torch.int32),
                          out=z(B * Hq * D), ws=z(1, torch.uint8))
    # the full-size tensors pass the extent checks and fail only at pointer marshalling (CPU tensors)
    with pytest.raises(ValueError, match="CUDA device"):
        tb.tb_project_append(shape, K, cap, Wk, Kp, 0, cap)


C_CLIENT = r"""
#include <stdio.h>
#include "tb.h"

int main(void) {
    /* a plain C caller: the header compiles as C and the calls below need no GPU */
    if (tb_version() != 1) return 1;
    tb_shape ok = {1, 32, 8, 128, 32, 32768};
    size_t bytes = 0;
    if (tb_workspace_size(&ok, 32767, 3277, 3277, &bytes) != TB_OK || bytes == 0) return 2;
    tb_shape bad = {1, 6, 4, 128, 32, 100};            /* Hq not a multiple of Hkv */
    if (tb_workspace_size(&bad, 10, 4, 4, &bytes) != TB_ERR_INVALID_ARG) return 3;
    if (tb_topk(&ok, (const float *)16, 10, 11, (int32_t *)16, NULL, 0, NULL, 0) != TB_ERR_INVALID_ARG) return 4;
    printf("%s|%zu\n", tb_status_string(TB_ERR_WORKSPACE), bytes);
    return 0;
}
"""


def test_plain_c_client_compiles_links_and_runs(lib_path, tmp_path):
    # include/tb.h is a C header and libtb.so a C library: a C program uses both without torch
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib_path)
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe), f"-L{libdir}", "-l:libtb.so", f"-Wl,-rpath,{libdir}"], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0, (res.returncode, res.stderr)
    text, nbytes = res.stdout.strip().split("|")
    assert text == "workspace missing or too small" and int(nbytes) > 0


def test_binding_has_a_function_of_the_same_name_for_every_entry_point(lib_path):
    import predicted_token_importance_tb_b300 as tb
    missing = [n for n in _declared() if not callable(getattr(tb, n, None))]
    assert not missing, missing
    assert tb.tb_version() == 1 and tb.tb_status_string(tb.TB_OK) == "ok"


def test_ragged_binding_checks_its_arguments(lib_path):
    import torch
    import predicted_token_importance_tb_b300 as tb
    B, Hq, Hkv, D, dp, cap = 2, 4, 2, 64, 16, 128
    shape = tb.Shape(B, Hq, Hkv, D, dp, cap)
    bf = torch.bfloat16

    def z(n, dtype=bf):
        return torch.zeros(n, dtype=dtype)

    kw = dict(q=z(B * Hq * D), q_imp=z(B * Hq * dp), K_new=z(B * Hkv * D), V_new=z(B * Hkv * D),
              Wk=z(Hkv * D * dp), K=z(B * Hkv * cap * D), V=z(B * Hkv * cap * D), Kp=z(B * Hkv * cap * dp),
              idx_state=z(B * Hkv * 8, torch.int32), n_pred=(ctypes.c_int64 * B)(), sel=z(B * Hkv * 8, torch.int32),
              sel_stride=8, counts=z(B * Hkv, torch.int32), out=z(B * Hq * D), ws=z(1, torch.uint8))
    n_host = (ctypes.c_int64 * B)(40, 90)
    with pytest.raises(ValueError, match="entries"):
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, (ctypes.c_int64 * 1)(40),
                                 z(B, torch.int64), **kw)
    with pytest.raises(TypeError, match="int64"):
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, n_host, z(B, torch.int32), **kw)
    # host arrays of another element type or a plain list: refused before the C side reads 8 B per entry
    with pytest.raises(TypeError, match="n_host"):
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, (ctypes.c_int32 * B)(40, 90),
                                 z(B, torch.int64), **kw)
    with pytest.raises(TypeError, match="n_pred"):
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, n_host, z(B, torch.int64),
                                 **{**kw, "n_pred": [0, 0]})
    with pytest.raises(ValueError, match="^K "):
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, n_host, z(B, torch.int64),
                                 **{**kw, "K": z(B * Hkv * cap * D - 1)})
    with pytest.raises(ValueError, match="CUDA device"):   # full extents pass; CPU tensors stop at marshalling
        tb.tb_decode_step_ragged(shape, 8, 1, 0, tb.TB_AGG_MEAN, 0.125, 0, n_host, z(B, torch.int64), **kw)


def test_noalloc_row_limit_matches_the_header():
    """The binding's copy of TB_TOPK_NOALLOC_MAX_ROWS is the header's value."""
    import re
    import predicted_token_importance_tb_b300 as tb
    with open(os.path.join(ROOT, "include", "tb.h")) as f:
        m = re.search(r"#define\s+TB_TOPK_NOALLOC_MAX_ROWS\s+(\d+)", f.read())
    assert m and int(m.group(1)) == tb.TB_TOPK_NOALLOC_MAX_ROWS


def test_host_validation_of_the_layer_stack(lib_path):
    # tb_decode_layers refuses bad settings before any CUDA call
    import predicted_token_importance_tb_b300 as tb
    lib = tb.load_library()
    fake = 1 << 20
    sp = tb.Shape(1, 32, 8, 128, 32, 40000).c()
    arr = (tb._LayerBuffers * 2)()
    for i in range(2):
        arr[i] = tb._LayerBuffers(*([fake] * 12), fake + (i + 1) * 4096, 1 << 30)
    s1, s2 = ctypes.c_void_p(0x10), ctypes.c_void_p(0x20)
    cases = [
        (tb._StepParams(3277, 2, 0, 0, 0.088, 0), 32767, 2, 3277, s1, s2, tb.TB_ERR_INVALID_ARG),   # T != 1
        (tb._StepParams(3277, 1, 1, 0, 0.088, 0), 32767, 2, 3277, s1, s2, tb.TB_ERR_INVALID_ARG),   # r != 0
        (tb._StepParams(3277, 1, 0, 0, 0.088, 0), 32767, 0, 3277, s1, s2, tb.TB_ERR_INVALID_ARG),   # no layers
        (tb._StepParams(3277, 1, 0, 0, 0.088, 0), 32767, 2, 3000, s1, s2, tb.TB_ERR_INVALID_ARG),   # sel_stride < k
        (tb._StepParams(3277, 1, 0, 0, 0.088, 0), 32767, 2, 3277, s1, s1, tb.TB_ERR_INVALID_ARG),   # one stream
        (tb._StepParams(3277, 1, 0, 0, 0.088, 0), 500, 2, 3277, s1, s2, tb.TB_ERR_INVALID_ARG),     # k > n + 1
        (tb._StepParams(300, 1, 0, 0, 0.088, 0), 500, 2, 3277, s1, s2, tb.TB_ERR_UNSUPPORTED),      # n too small
        (tb._StepParams(3277, 1, 0, 0, 0.088, tb.TB_STEP_PIPELINE), 32767, 2, 3277, s1, s2,
         tb.TB_ERR_INVALID_ARG),                                                                    # flags
    ]
    for params, n, L, stride, a, b, want in cases:
        st = lib.tb_decode_layers(ctypes.byref(sp), ctypes.byref(params), n, L, arr, stride, None, a, b)
        assert st == want, (params.T, params.r, n, L, stride, st)
    # two layers sharing one workspace would overlap on the GPU
    arr[1].ws = arr[0].ws
    st = lib.tb_decode_layers(ctypes.byref(sp), ctypes.byref(tb._StepParams(3277, 1, 0, 0, 0.088, 0)), 32767, 2,
                              arr, 3277, None, s1, s2)
    assert st == tb.TB_ERR_INVALID_ARG
