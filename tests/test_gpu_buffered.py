"""GPU parity of the decode step with sink and local-window buffers and batched key projection
(gist.science summary, Inference Strategy; Optimizations, Batching) against the oracle."""
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


def run_buffered_parity(w, n0, steps, S, W, T, r, k, P0, kv_host=False, budget_neighbours=False, agg=0,
                        layer_hook=None):
    """Drive the buffered step on the GPU; check, every step, the batches of Kp (1 ulp of the oracle's
    projection, then adopted by the oracle so both score identical inputs), the centres (top-k under the
    tie band), the selection exactly (the oracle's construction from the GPU's centres), and the output
    against the oracle's attention over the GPU's selection."""
    cap = n0 + steps
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    if layer_hook is not None:
        layer_hook(L)
    K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
    Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K, cap, Wk, Kp, 0, P0)
    if kv_host:
        K, V = K.cpu().pin_memory(), V.cpu().pin_memory()
    dec = tb.BufferedDecodeLayer(shape, k, sink=S, window=W, proj_end=P0, T=T, r=r, agg=agg, scale=w.scale,
                                 n_max=cap - 1, budget_neighbours=budget_neighbours)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    oK, oV = u16(L["K"]).copy(), u16(L["V"]).copy()
    oKp = u16(Kp).copy()
    Wb = u16(L["Wk"])
    st = oracle.BufferedState(P0)
    want_rows = None
    rows = w.B * w.Hkv
    for t in range(steps):
        n = n0 + t
        n_t = n + 1
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        dec.step(t, n, q=d["q"].cuda(), q_imp=d["q_imp"].cuda(), K_new=d["K_new"].cuda(), V_new=d["V_new"].cuda(),
                 Wk=Wk, K=K, V=V, Kp=Kp, out=out)
        torch.cuda.synchronize()
        tb.check_dev_status(dec.status, f"step {t}")
        pe = st.proj_end
        ref_out, _, _ = oracle.decode_step_buffered(
            st, t, n, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=L["Wk"], K=oK, V=oV,
            Kp=oKp, k=k, T=T, r=r, agg=agg, scale=w.scale, sink=S, window=W, budget_neighbours=budget_neighbours)
        P = st.proj_end
        assert dec.proj_end.value == P
        assert np.array_equal(u16(K[:, :, n]), oK[:, :, n])
        if P > pe:   # a batch of projected rows
            g = u16(Kp[:, :, pe:P])
            kn = np.ascontiguousarray(oK[:, :, pe:P])
            _, kp64 = oracle.project(kn, Wb)
            assert_kp_close(g, kp64, kp_l1(kn, Wb))
            oKp[:, :, pe:P] = g
        if t % T == 0:
            kc = min(dec.kc, max(0, P - S))
            gidx = dec.idx_state.flatten()[: rows * kc].reshape(w.B, w.Hkv, kc).cpu().numpy()
            if kc > 0:
                s_ref, _ = oracle.score(d["q_imp"], np.ascontiguousarray(oKp[:, :, S:P]), agg)
                assert_topk_end_to_end(gidx, s_ref, kc)
            want_rows = oracle.buffered_select(gidx, r, S, P, n_t)
            same = np.array_equal(gidx, st.idx)
        else:
            want_rows = [x + [n] for x in want_rows]
        gcnt = dec.counts.cpu().numpy()
        gsel = dec.sel.cpu().numpy()
        for x in range(rows):
            b, h = divmod(x, w.Hkv)
            assert gsel[b, h, : gcnt[b, h]].tolist() == want_rows[x], (t, b, h)
        got = out.float().cpu().numpy()
        ref_g = oracle.attn(d["q"], oK, oV, gsel, gcnt, w.scale)
        assert np.abs(got - ref_g).max() <= OUT_ATOL, t
        if same:
            assert np.abs(got - ref_out).max() <= OUT_ATOL, t
    return dec


def test_buffered_small_interval_neighbours():
    # batches of 16 rows on the CUDA cores, prediction every 3 steps, +-1 neighbours
    w = synth.small(B=2, Hq=8, Hkv=2, D=128, dp=32, N=600, k=40, seed=51, outliers=2)
    run_buffered_parity(w, n0=w.N, steps=12, S=4, W=16, T=3, r=1, k=40, P0=560)


def test_buffered_tensor_core_batches_per_step():
    # batches of 128 rows (the tcgen05 projection), prediction at every step
    w = synth.small(B=1, Hq=8, Hkv=2, D=128, dp=32, N=3000, k=200, seed=52, outliers=2)
    run_buffered_parity(w, n0=w.N, steps=4, S=8, W=128, T=1, r=0, k=200, P0=2600)


def test_buffered_prefill_far_behind_and_budget_neighbours():
    # nothing projected at prefill beyond the sink: the first prediction projects many batches at once
    w = synth.small(B=1, Hq=4, Hkv=4, D=64, dp=16, N=900, k=30, seed=53)
    run_buffered_parity(w, n0=w.N, steps=5, S=2, W=32, T=2, r=2, k=30, P0=0, budget_neighbours=True)


def test_buffered_host_kv():
    w = synth.small(B=1, Hq=8, Hkv=2, D=128, dp=32, N=800, k=50, seed=54, outliers=2)
    run_buffered_parity(w, n0=w.N, steps=4, S=4, W=32, T=2, r=1, k=50, P0=700, kv_host=True)


def test_buffered_window_wider_than_the_batches_so_far():
    # W above the unprojected span: no batch is projected, the candidates are the prefill rows
    w = synth.small(B=1, Hq=8, Hkv=2, D=64, dp=16, N=500, k=20, seed=55)
    run_buffered_parity(w, n0=w.N, steps=3, S=0, W=300, T=1, r=0, k=20, P0=400, agg=1)


def test_buffered_sink_covers_every_projected_row():
    # S >= proj_end: no candidates at all; the selection is the sink and the window
    w = synth.small(B=2, Hq=4, Hkv=2, D=128, dp=32, N=300, k=10, seed=56)
    run_buffered_parity(w, n0=w.N, steps=3, S=280, W=64, T=2, r=1, k=10, P0=200)


def test_buffered_single_launch_general_select():
    # blocky scores send the single-launch step to its general select; the centres then come from the
    # row's merging CTA
    from test_gpu_decode import general_select_steps
    w = synth.small(B=1, Hq=32, Hkv=8, D=128, dp=32, N=32767, k=3277, seed=57, outliers=4)

    def hot_blocks(L):
        g = torch.Generator().manual_seed(77)
        nblk = L["K"].shape[2] // 32
        hot = torch.randperm(nblk, generator=g)[: nblk // 10]
        rows = (hot[:, None] * 32 + torch.arange(32)[None, :]).reshape(-1)
        rows = rows[rows < L["K"].shape[2]]
        L["K"][:, :, rows] = L["K"][:, :, rows] * 8

    dec = run_buffered_parity(w, n0=w.N, steps=2, S=64, W=256, T=1, r=0, k=3277, P0=32256, layer_hook=hot_blocks)
    assert sum(general_select_steps(dec)) > 0


def test_buffered_single_launch_everything_forced():
    # S >= proj_end with a prediction at every step: the single-launch step keeps every token
    w = synth.small(B=2, Hq=4, Hkv=2, D=128, dp=32, N=300, k=10, seed=58)
    run_buffered_parity(w, n0=w.N, steps=2, S=280, W=64, T=1, r=0, k=10, P0=200)


def test_buffered_single_launch_host_kv():
    w = synth.small(B=1, Hq=8, Hkv=2, D=128, dp=32, N=4000, k=300, seed=59, outliers=2)
    run_buffered_parity(w, n0=w.N, steps=3, S=16, W=128, T=1, r=0, k=300, P0=3700, kv_host=True)
