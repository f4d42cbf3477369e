"""GPU parity of the decode step for a batch of sequences of different lengths against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OUT_ATOL, assert_kp_close, assert_topk_end_to_end, kp_l1, u16

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


@pytest.mark.parametrize("T,r,ns,agg,bn", [(1, 0, [1500, 2201, 3000], 0, False), (2, 1, [2999, 1024, 1777], 0, False),
                                          (3, 2, [700, 701, 1600], 0, False), (2, 1, [900, 2500], 1, True),
                                          (1, 0, [8192, 32767], 0, False)])
def test_ragged_batch_matches_oracle(T, r, ns, agg, bn):
    steps = 5
    B = len(ns)
    w = synth.small(B=B, Hq=8, Hkv=2, D=128, dp=32, N=max(ns), k=100, seed=61 + T, outliers=2)
    cap = max(ns) + steps
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=max(ns))
    K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
    Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K, cap, Wk, Kp, 0, max(ns))
    dec = tb.RaggedDecodeLayer(shape, w.k, T=T, r=r, agg=agg, scale=w.scale, n_max=cap - 1, budget_neighbours=bn)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    oK, oV, oKp = u16(L["K"]).copy(), u16(L["V"]).copy(), u16(Kp).copy()
    sts = [oracle.DecodeState() for _ in range(B)]
    Wb = u16(L["Wk"])
    for t in range(steps):
        cur = [n + t for n in ns]
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        dec.step(t, cur, q=d["q"].cuda(), q_imp=d["q_imp"].cuda(), K_new=d["K_new"].cuda(), V_new=d["V_new"].cuda(),
                 Wk=Wk, K=K, V=V, Kp=Kp, out=out)
        torch.cuda.synchronize()
        tb.check_dev_status(dec.status, f"step {t}")
        oracle.decode_step_ragged(sts, t, cur, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"],
                                  Wk=L["Wk"], K=oK, V=oV, Kp=oKp, k=w.k, T=T, r=r, agg=agg, scale=w.scale,
                                  budget_neighbours=bn)
        gidx = dec.idx_state.cpu().numpy()
        gsel, gcnt = dec.sel.cpu().numpy(), dec.counts.cpu().numpy()
        for b, n in enumerate(cur):
            # the appended row of this sequence, at its own position
            assert np.array_equal(u16(K[b, :, n]), oK[b, :, n])
            kn = np.ascontiguousarray(oK[b:b + 1, :, n:n + 1])
            _, kp64 = oracle.project(kn, Wb)
            g = u16(Kp[b:b + 1, :, n])[:, :, None]
            assert_kp_close(g, kp64, kp_l1(kn, Wb))
            oKp[b, :, n] = g[0, :, 0]            # both score the GPU's row from here on
            assert dec.n_pred[b] == sts[b].n_pred
            if t % T == 0:
                s_ref, _ = oracle.score(d["q_imp"][b:b + 1], np.ascontiguousarray(oKp[b:b + 1, :, : n + 1]), agg)
                assert_topk_end_to_end(gidx[b:b + 1], s_ref, dec.kc)
            want, wcnt = oracle.expand(gidx[b:b + 1], r, sts[b].n_pred, n + 1, sel_stride=dec.sel_stride)
            assert np.array_equal(gcnt[b], wcnt[0])
            for h in range(w.Hkv):
                assert np.array_equal(gsel[b, h, : gcnt[b, h]], want[0, h, : wcnt[0, h]])
        ref = oracle.attn(d["q"], oK, oV, gsel, gcnt, w.scale)
        assert np.abs(out.float().cpu().numpy() - ref).max() <= OUT_ATOL
