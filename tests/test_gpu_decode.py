"""GPU parity of the whole decode step (append, predict every T steps, widen, attend) against the oracle."""
import ctypes

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


def run_decode_parity(w: synth.Workload, n0: int, steps: int, layers=(0,), k=None, fused=True, agg=0,
                      layer_hook=None, kv_host=False, budget_neighbours=False, pipeline=False):
    """Drive `steps` decode steps per layer on the GPU and check every step against the oracle.

    The oracle starts from the GPU-projected prefix of Kp (identical inputs),
    projects each appended row itself, and makes its own selections; top-k
    sets are compared under the tie band, the selection rows exactly against
    the oracle's expansion of the GPU's prediction, and the output against the
    oracle's attention over the GPU's selection. kv_host: K and V live in
    pinned host memory (the offloaded cache). budget_neighbours: k // (2r+1)
    centres per prediction. pipeline: a step with T = 1, r = 0 runs as the
    three-kernel form rather than the single cooperative kernel.
    """
    k = w.k if k is None else k
    cap = n0 + steps
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    dec = None
    for layer in layers:
        L = synth.make_layer(w, layer=layer, cap=cap, n=n0)
        if layer_hook is not None:
            layer_hook(L)
        K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
        Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
        tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n0)
        if kv_host:
            K, V = K.cpu().pin_memory(), V.cpu().pin_memory()
        dec = tb.DecodeLayer(shape, k, T=w.T, r=w.r, agg=agg, scale=w.scale, n_max=cap - 1, fused=fused,
                             budget_neighbours=budget_neighbours, pipeline=pipeline)
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        oK, oV = u16(L["K"]).copy(), u16(L["V"]).copy()
        oKp = u16(Kp).copy()
        st = oracle.DecodeState()
        for t in range(steps):
            n = n0 + t
            d = synth.make_step(w, layer, t, L["outlier_ch"])
            dec.step(t, n, q=d["q"].cuda(), q_imp=d["q_imp"].cuda(), K_new=d["K_new"].cuda(),
                     V_new=d["V_new"].cuda(), Wk=Wk, K=K, V=V, Kp=Kp, out=out)
            torch.cuda.synchronize()
            tb.check_dev_status(dec.status, f"layer {layer} step {t}")
            ref_out, ref_sel, ref_cnt = oracle.decode_step(
                st, t, n, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=L["Wk"], K=oK, V=oV,
                Kp=oKp, k=k, T=w.T, r=w.r, agg=agg, scale=w.scale, budget_neighbours=budget_neighbours)
            # appended rows
            gKp = u16(Kp[:, :, n])[:, :, None]
            kn = np.ascontiguousarray(oK[:, :, n:n + 1])
            _, kp64 = oracle.project(kn, u16(L["Wk"]))
            assert_kp_close(gKp, kp64, kp_l1(kn, u16(L["Wk"])))
            assert np.array_equal(u16(K[:, :, n]), oK[:, :, n])
            n_t = n + 1
            assert dec.n_pred.value == st.n_pred
            gidx = dec.idx_state.cpu().numpy()
            if t % w.T == 0:
                s_ref, _ = oracle.score(d["q_imp"], np.ascontiguousarray(oKp[:, :, :n_t]), agg)
                assert_topk_end_to_end(gidx, s_ref, dec.kc)
            # selection = the oracle's expansion of the GPU's prediction, plus the tail
            want_sel, want_cnt = oracle.expand(gidx, w.r, st.n_pred, n_t, sel_stride=dec.sel_stride)
            gcnt = dec.counts.cpu().numpy()
            gsel = dec.sel.cpu().numpy()
            assert np.array_equal(gcnt, want_cnt)
            for b in range(w.B):
                for h in range(w.Hkv):
                    assert np.array_equal(gsel[b, h, :gcnt[b, h]], want_sel[b, h, :gcnt[b, h]])
            # output over the GPU's selection
            ref_g = oracle.attn(d["q"], oK, oV, gsel, gcnt, w.scale)
            got = out.float().cpu().numpy()
            assert np.abs(got - ref_g).max() <= OUT_ATOL, (layer, t)
            # and the end-to-end output where the predictions agree
            if np.array_equal(gidx, st.idx):
                assert np.abs(got - ref_out).max() <= OUT_ATOL
    return dec


def general_select_steps(dec) -> list:
    """Per (batch, KV head) row: decode steps whose single-exchange selection fell back to the general one.

    The count sits in the row's control block at the start of the workspace
    (fourth 32-bit word of each block)."""
    rows = dec.shape.B * dec.shape.Hkv
    ws = dec.ws.cpu().numpy()
    stride = ROWCTL_BYTES
    return [int(ws[r * stride + 12:r * stride + 16].view(np.uint32)[0]) for r in range(rows)]


# bytes of one row control block: 4 words, 3 x 2048 histogram words, 2 x 512 chunk words, 4096 (key, token) pairs
ROWCTL_BYTES = 4 * 4 + 3 * 2048 * 4 + 2 * 512 * 4 + 4096 * 8


@pytest.mark.parametrize("fused", [True, False])
def test_decode_small_per_step(fused):
    w = synth.WORKLOADS[0]
    run_decode_parity(w, n0=w.N - 1, steps=3, fused=fused)


@pytest.mark.parametrize("pipeline", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,D,dp,N,k,agg", [(2, 8, 2, 128, 32, 5000, 500, 0), (1, 4, 4, 64, 16, 777, 1, 0),
                                                   (1, 8, 2, 128, 32, 3001, 3001, 0), (3, 6, 3, 64, 24, 2500, 99, 1),
                                                   (1, 16, 1, 32, 8, 20000, 6000, 1), (4, 8, 8, 128, 16, 40, 7, 0),
                                                   (1, 16, 1, 128, 32, 20000, 2000, 0), (2, 32, 4, 64, 16, 9000, 900, 1)])
def test_decode_fused_matches_oracle_shapes(B, Hq, Hkv, D, dp, N, k, agg, pipeline):
    # (shapes the three-kernel form does not take run the cooperative kernel either way)
    w = synth.small(B=B, Hq=Hq, Hkv=Hkv, D=D, dp=dp, N=N, k=k, seed=N + k, outliers=2)
    run_decode_parity(w, n0=w.N - 1, steps=2, agg=agg, pipeline=pipeline)


def test_decode_fused_equals_unfused_bitwise_selection():
    # identical scores on the cooperative kernel and the separate kernels, so identical selections; outputs
    # agree to rounding
    w = synth.WORKLOADS[1]
    cap = w.N
    n0 = w.N - 1
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    res = []
    for fused in (True, False):
        K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
        Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
        tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n0)
        dec = tb.DecodeLayer(shape, w.k, scale=w.scale, n_max=n0, fused=fused)
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        d = synth.make_step(w, 0, 0, L["outlier_ch"])
        for rep in range(3):   # repeated calls reuse the workspace
            dec.step(0, n0, q=d["q"].cuda(), q_imp=d["q_imp"].cuda(), K_new=d["K_new"].cuda(),
                     V_new=d["V_new"].cuda(), Wk=Wk, K=K, V=V, Kp=Kp, out=out)
        torch.cuda.synchronize()
        tb.check_dev_status(dec.status)
        res.append((dec.idx_state.cpu().numpy(), dec.sel.cpu().numpy(), dec.counts.cpu().numpy(),
                    out.float().cpu().numpy(), u16(Kp)))
    assert np.array_equal(res[0][0], res[1][0])
    assert np.array_equal(res[0][2], res[1][2])
    assert np.array_equal(res[0][1][..., :w.k], res[1][1][..., :w.k])
    assert np.array_equal(res[0][4], res[1][4])
    assert np.abs(res[0][3] - res[1][3]).max() <= 2e-3


def test_decode_fast_step_takes_the_single_exchange_on_smooth_scores():
    w = synth.WORKLOADS[1]
    dec = run_decode_parity(w, n0=w.N - 1, steps=2)
    assert sum(general_select_steps(dec)) == 0


def test_decode_blocky_scores_fall_back_to_the_general_select():
    # 10% of the 32-token blocks hold keys scaled by 8: the CTAs of a row own
    # very different shares of them, so their local threshold estimates miss
    # and the step must take the general distributed select, with the same
    # exact result.
    w = synth.WORKLOADS[1]

    def hot_blocks(L):
        g = torch.Generator().manual_seed(77)
        nblk = L["K"].shape[2] // 32
        hot = torch.randperm(nblk, generator=g)[: nblk // 10]
        rows = (hot[:, None] * 32 + torch.arange(32)[None, :]).reshape(-1)
        rows = rows[rows < L["K"].shape[2]]
        L["K"][:, :, rows] = L["K"][:, :, rows] * 8

    dec = run_decode_parity(w, n0=w.N - 1, steps=2, layer_hook=hot_blocks)
    assert sum(general_select_steps(dec)) > 0


def test_decode_blocky_scores_three_kernel_form():
    # the same hot blocks through the three-kernel form (its selection has no local estimate to miss)
    w = synth.WORKLOADS[1]

    def hot_blocks(L):
        g = torch.Generator().manual_seed(77)
        nblk = L["K"].shape[2] // 32
        hot = torch.randperm(nblk, generator=g)[: nblk // 10]
        rows = (hot[:, None] * 32 + torch.arange(32)[None, :]).reshape(-1)
        rows = rows[rows < L["K"].shape[2]]
        L["K"][:, :, rows] = L["K"][:, :, rows] * 8

    run_decode_parity(w, n0=w.N - 1, steps=2, layer_hook=hot_blocks, pipeline=True)


def test_decode_small_interval_with_neighbours():
    w = synth.small(B=2, Hq=8, Hkv=2, D=128, dp=32, N=3000, k=100, T=4, r=1, seed=31, outliers=4)
    run_decode_parity(w, n0=w.N, steps=10)


def test_decode_interval_r2_group_of_one():
    w = synth.small(B=1, Hq=4, Hkv=4, D=64, dp=16, N=1500, k=40, T=3, r=2, seed=32)
    run_decode_parity(w, n0=w.N, steps=7)


@pytest.mark.parametrize("fused,pipeline", [(True, False), (True, True), (False, False)])
def test_decode_llama_layer_step(fused, pipeline):
    # the 32K-token Llama-3-8B-shaped layer: one step at N = 32768 after the append
    w = synth.WORKLOADS[1]
    run_decode_parity(w, n0=w.N - 1, steps=2, fused=fused, pipeline=pipeline)


def test_decode_32layer_stack_interval_sampled_layers():
    # the 32-layer B=8 stack at full per-layer shape, two of its 32 layers sampled (0 and 31; every layer runs
    # the same code on its own seeded data), all 64 steps
    w = synth.WORKLOADS[2]
    run_decode_parity(w, n0=w.N, steps=w.steps, layers=(0, 31))


def test_decode_budget_preserving_neighbours():
    # k // (2r + 1) centres widened by +-r: the selection stays within the budget
    w = synth.small(B=2, Hq=8, Hkv=2, D=128, dp=32, N=4000, k=300, T=3, r=2, seed=33, outliers=2)
    dec = run_decode_parity(w, n0=w.N, steps=5, budget_neighbours=True)
    assert dec.kc == 60
    assert int(dec.counts.max().item()) <= w.k + w.T - 1
