"""tb_topk_noalloc against tb_topk, through the C ABI.

tb_topk_noalloc serves callers that cannot allocate device memory (a host
runtime that owns every allocation, a server whose memory is fixed at
start-up): its scratch is a static array inside libtb instead of a workspace.
Its indices must be bit-identical to tb_topk's on the same scores, and stay so
on back-to-back calls, since every call reuses the array the previous call
left behind. This file is collected last so that a failing run stopped at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


def _scores(B, Hkv, n, seed, levels=0):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn((B, Hkv, n), generator=g, dtype=torch.float32) * 5.0
    if levels:   # few distinct values: the budget boundary falls inside a tie
        s = torch.floor(s.clamp(-levels, levels - 1))
    return s


def _both(shape, s_host, k):
    n = s_host.shape[-1]
    s = s_host.cuda()
    rows = (shape.B, shape.Hkv)
    idx_ws = torch.full(rows + (k,), -1, dtype=torch.int32, device="cuda")
    idx_na = torch.full(rows + (k,), -1, dtype=torch.int32, device="cuda")
    ws = tb.workspace(shape, n, k, k)
    st_ws, st_na = tb.dev_status(), tb.dev_status()
    tb.tb_topk(shape, s, n, k, idx_ws, ws, dev_status=st_ws)
    tb.tb_topk_noalloc(shape, s, n, k, idx_na, dev_status=st_na)
    torch.cuda.synchronize()
    tb.check_dev_status(st_ws, "tb_topk")
    tb.check_dev_status(st_na, "tb_topk_noalloc")
    return idx_ws.cpu().numpy(), idx_na.cpu().numpy()


def test_noalloc_matches_workspace_topk_on_consecutive_calls():
    # first call: the bench layer's selection (8 KV heads, N = 32768, 10% budget)
    sh1 = tb.Shape(1, 32, 8, 128, 32, 32768)
    a, b = _both(sh1, _scores(1, 8, 32768, seed=11), 3277)
    assert np.array_equal(a, b)
    assert (np.diff(b, axis=-1) > 0).all()
    # second call right after it: more rows, a ragged n and heavy ties, on the
    # array the first call left behind
    sh2 = tb.Shape(4, 32, 8, 128, 32, 20001)
    a, b = _both(sh2, _scores(4, 8, 20001, seed=12, levels=6), 2048)
    assert np.array_equal(a, b)
    # and the first problem once more, after the second
    a, b = _both(sh1, _scores(1, 8, 32768, seed=13), 3277)
    assert np.array_equal(a, b)


def test_noalloc_rejects_more_rows_than_its_array_holds():
    rows = tb.TB_TOPK_NOALLOC_MAX_ROWS
    sh = tb.Shape(rows // 8 + 1, 8, 8, 64, 16, 128)     # B*Hkv = rows + 8
    s = torch.zeros((sh.B, sh.Hkv, 128), dtype=torch.float32, device="cuda")
    idx = torch.zeros((sh.B, sh.Hkv, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(tb.TBError) as e:
        tb.tb_topk_noalloc(sh, s, 128, 4, idx)
    assert e.value.status == tb.TB_ERR_UNSUPPORTED
