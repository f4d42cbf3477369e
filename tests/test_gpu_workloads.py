"""Full-size workloads through the C ABI: long context with planted heavy hitters, prefill + budget sweep."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OUT_ATOL, assert_kp_close, assert_scores_close, assert_topk_end_to_end, kp_l1, u16

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


def _prefill(w, L, shape):
    K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
    Kp = torch.empty((w.B, w.Hkv, w.N, w.dp), dtype=torch.bfloat16, device="cuda")
    st = tb.dev_status()
    tb.tb_project_append(shape, K, w.N, Wk, Kp, 0, w.N, dev_status=st)
    torch.cuda.synchronize()
    tb.check_dev_status(st)
    return K, V, Wk, Kp


def _select_attend(w, shape, L, K, V, Kp, k):
    ws = tb.workspace(shape, w.N, k, k)
    st = tb.dev_status()
    s = torch.empty((w.B, w.Hkv, w.N), dtype=torch.float32, device="cuda")
    idx = torch.empty((w.B, w.Hkv, k), dtype=torch.int32, device="cuda")
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    q_imp, q = L["q_imp"].cuda(), L["q"].cuda()
    tb.tb_score(shape, q_imp, Kp, w.N, s, dev_status=st)
    tb.tb_topk(shape, s, w.N, k, idx, ws, dev_status=st)
    tb.tb_sparse_decode_attn(shape, q, K, V, idx, None, k, w.scale, out, ws, dev_status=st)
    torch.cuda.synchronize()
    tb.check_dev_status(st)
    return s.cpu().numpy(), idx.cpu().numpy(), out.float().cpu().numpy()


def test_long_context_planted_heavy_hitters():
    w = synth.WORKLOADS[3]
    L = synth.make_layer(w)
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, w.N)
    K, V, Wk, Kp = _prefill(w, L, shape)
    gKp = u16(Kp)
    # projection: a sample of rows per head against the oracle
    rows = np.random.default_rng(0).choice(w.N, 1024, replace=False)
    Kin = np.ascontiguousarray(u16(L["K"])[:, :, rows])
    want, want64 = oracle.project(Kin, L["Wk"])
    assert_kp_close(gKp[:, :, rows], want64, kp_l1(Kin, u16(L["Wk"])))
    s, idx, out = _select_attend(w, shape, L, K, V, Kp, w.k)
    s_ref, l1 = oracle.score(L["q_imp"], gKp)
    assert_scores_close(s, s_ref, l1)
    assert np.array_equal(idx, oracle.topk(s, w.k))          # bit-exact on identical scores
    for b in range(w.B):
        for h in range(w.Hkv):
            assert set(L["planted_pos"][b, h].tolist()) <= set(idx[b, h].tolist())   # recall 64/64
    ref = oracle.attn(L["q"], L["K"], L["V"], idx, np.full((w.B, w.Hkv), w.k, np.int32), w.scale)
    assert np.abs(out - ref).max() <= OUT_ATOL


def test_prefill_then_budget_sweep():
    w = synth.WORKLOADS[4]
    L = synth.make_layer(w)
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, w.N)
    K, V, Wk, Kp = _prefill(w, L, shape)
    gKp = u16(Kp)
    want, want64 = oracle.project(L["K"], L["Wk"])
    rows = np.random.default_rng(1).choice(w.N, 2048, replace=False)
    assert_kp_close(gKp[:, :, rows], want64[:, :, rows], kp_l1(np.ascontiguousarray(u16(L["K"])[:, :, rows]),
                                                               u16(L["Wk"])))
    assert (gKp != want).mean() < 0.01
    s_ref_own, _ = oracle.score(L["q_imp"], want)        # scores on the oracle's own Kp
    dense = oracle.dense_attn(L["q"], L["K"], L["V"], w.N, w.scale)
    for p in w.budgets:
        k = synth.budget(p, w.N)
        s, idx, out = _select_attend(w, shape, L, K, V, Kp, k)
        assert np.array_equal(idx, oracle.topk(s, k))
        assert_topk_end_to_end(idx, s_ref_own, k)
        ref = oracle.attn(L["q"], L["K"], L["V"], idx, np.full((w.B, w.Hkv), k, np.int32), w.scale)
        assert np.abs(out - ref).max() <= OUT_ATOL, p
        if k == w.N:
            assert np.array_equal(idx, np.broadcast_to(np.arange(w.N, dtype=np.int32), idx.shape))
            assert np.abs(out - dense).max() <= OUT_ATOL
