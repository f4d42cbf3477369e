"""GPU parity of the three-kernel decode step (selection over the cached tokens, the exact cut, then the
attention kernel that appends the new token and lets it displace the k-th) and of the multi-layer step built on
it.

Exact cases use integer-valued inputs and a projection that copies the first dp key dimensions: every
projected key, every fp32 score and the oracle's fp64 scores are then the same numbers, so the selection must
match the oracle's bit for bit, ties included (they are frequent with small integers).
"""
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


def _bf(x):
    return x.to(torch.bfloat16)


def exact_layer(B, Hq, Hkv, D, dp, n, seed, krange=4, qrange=2, equal_rows=False):
    """Integer K (|K| <= krange), V ~ N(0,1), integer q_imp (|q| <= qrange), Wk copying dims [0, dp)."""
    g = torch.Generator().manual_seed(seed)
    cap = n + 1
    K = torch.randint(-krange, krange + 1, (B, Hkv, cap, D), generator=g).float()
    if equal_rows:
        K[:] = K[:, :, :1, :]
    V = torch.randn((B, Hkv, cap, D), generator=g)
    Wk = torch.zeros((Hkv, D, dp))
    for i in range(dp):
        Wk[:, i, i] = 1.0
    q = torch.randn((B, Hq, D), generator=g)
    q_imp = torch.randint(-qrange, qrange + 1, (B, Hq, dp), generator=g).float()
    K_new = torch.randint(-krange, krange + 1, (B, Hkv, D), generator=g).float()
    V_new = torch.randn((B, Hkv, D), generator=g)
    return {k: _bf(v) for k, v in dict(K=K, V=V, Wk=Wk, q=q, q_imp=q_imp, K_new=K_new, V_new=V_new).items()}


def _ctl_report(dec, n, k, L, agg):
    """The three-kernel step's per-row result block (cut, offsets) next to the true cut (debugging aid)."""
    sh = dec.shape
    rows = sh.B * sh.Hkv
    rowctl = 16 + 3 * 2048 * 4 + 2 * 512 * 4 + 4096 * 8
    off = -(-(rows * rowctl) // 256) * 256
    off = -(-(off + rows * 4) // 256) * 256
    ws = dec.ws.cpu().numpy()
    prow = 32 + 64 * 4 + 68 * 4 + 4096 * 4
    s, _ = oracle.score(u16(L["q_imp"]), u16(L["K"])[:, :, :n, :sh.dp].copy(), agg)
    out = []
    for r in range(rows):
        w = ws[off + r * prow: off + (r + 1) * prow].view(np.uint32)
        b1, ck, ci, k1 = int(w[4]), int(w[5]), int(w[6]), int(w[7])
        offs = w[8 + 64: 8 + 64 + 8].view(np.int32).tolist()
        sr = s.reshape(rows, -1)[r]
        order = sorted(range(n), key=lambda t: (-sr[t], t))
        kk = min(k, n)
        true_e = order[kk - 1]
        out.append(f"ctl row {r}: b1 {b1} cut_idx {ci} k1 {k1} offs[:8] {offs}; true k-th {true_e} "
                   f"(score {sr[true_e]}), cut_idx score {sr[ci] if 0 <= ci < n else None}, "
                   f"next ranked {order[kk] if kk < n else None}")
    return "\n".join(out)


def run_exact(B, Hq, Hkv, D, dp, n, k, agg=0, seed=0, K_new_hook=None, equal_rows=False):
    """One step through the three-kernel form on exact inputs; the selection must equal the oracle's exactly."""
    L = exact_layer(B, Hq, Hkv, D, dp, n, seed, equal_rows=equal_rows)
    if K_new_hook is not None:
        K_new_hook(L)
    cap = n + 1
    shape = tb.Shape(B, Hq, Hkv, D, dp, cap)
    K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
    Kp = torch.zeros((B, Hkv, cap, dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n)
    dec = tb.DecodeLayer(shape, k, agg=agg, scale=D ** -0.5, n_max=n, pipeline=True)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    for rep in range(2):   # the second call finds the workspace the first one left
        dec.step(0, n, q=L["q"].cuda(), q_imp=L["q_imp"].cuda(), K_new=L["K_new"].cuda(), V_new=L["V_new"].cuda(),
                 Wk=Wk, K=K, V=V, Kp=Kp, out=out)
    torch.cuda.synchronize()
    tb.check_dev_status(dec.status)
    oK, oV = u16(L["K"]).copy(), u16(L["V"]).copy()
    oKp = u16(Kp).copy()
    oKp[:, :, n:] = 0
    st = oracle.DecodeState()
    ref_out, ref_sel, ref_cnt = oracle.decode_step(
        st, 0, n, q=L["q"], q_imp=L["q_imp"], K_new=L["K_new"], V_new=L["V_new"], Wk=L["Wk"], K=oK, V=oV, Kp=oKp,
        k=k, T=1, r=0, agg=agg, scale=D ** -0.5)
    gidx = dec.idx_state.cpu().numpy()
    if not np.array_equal(gidx, st.idx):
        msg = []
        for b in range(B):
            for h in range(Hkv):
                g, o = set(gidx[b, h].tolist()), set(st.idx[b, h].tolist())
                if g != o or not np.array_equal(gidx[b, h], st.idx[b, h]):
                    bad = np.nonzero(gidx[b, h] != st.idx[b, h])[0]
                    msg.append(f"row ({b},{h}): gpu-only {sorted(g - o)[:6]} oracle-only {sorted(o - g)[:6]} "
                               f"first differing positions {bad[:6].tolist()} gpu {gidx[b, h][bad[:6]].tolist()} "
                               f"oracle {st.idx[b, h][bad[:6]].tolist()}")
        if n <= 6000:
            msg.append(_ctl_report(dec, n, k, L, agg))
        raise AssertionError("selection differs from the oracle's on exact scores:\n" + "\n".join(msg))
    assert np.array_equal(dec.sel.cpu().numpy()[..., :k], st.idx)
    assert np.array_equal(dec.counts.cpu().numpy(), np.full((B, Hkv), k, dtype=np.int32))
    assert np.array_equal(u16(Kp[:, :, n]), oKp[:, :, n])          # the appended projected key, exact here
    assert np.array_equal(u16(K[:, :, n]), oK[:, :, n])
    assert np.array_equal(u16(V[:, :, n]), oV[:, :, n])
    got = out.float().cpu().numpy()
    assert np.abs(got - ref_out).max() <= OUT_ATOL
    return gidx, st, L


@pytest.mark.parametrize("B,Hq,Hkv,D,dp,n,k,agg", [
    (2, 8, 2, 64, 16, 5000, 500, 0),       # several chunks per row, ties everywhere
    (1, 8, 2, 128, 32, 3000, 3001, 0),     # k = n + 1: every token kept, the new one appended
    (1, 8, 2, 128, 32, 3000, 3000, 0),     # k = n: the new token displaces the lowest ranked if above it
    (2, 8, 2, 64, 16, 2048, 1, 1),         # a single token, max over the group
    (1, 32, 8, 128, 32, 20000, 7000, 0),   # kept tokens span several compaction segments per chunk
    (1, 16, 1, 128, 64, 9000, 900, 1),     # dp = 64, G = 16
])
def test_pipeline_selection_bit_exact_on_exact_scores(B, Hq, Hkv, D, dp, n, k, agg):
    run_exact(B, Hq, Hkv, D, dp, n, k, agg=agg, seed=n + k + agg)


def test_pipeline_new_token_displaces_the_kth():
    # the new key scores above every cached token: it must be kept and the k-th ranked cached token dropped
    def planted(L):
        qbar = L["q_imp"].float().reshape(1, 2, 4, 16).mean(2)            # [B, Hkv, dp]
        kn = torch.zeros_like(L["K_new"].float())
        kn[..., :16] = 4.0 * torch.sign(qbar)
        L["K_new"] = _bf(kn)

    gidx, st, L = run_exact(1, 8, 2, 64, 16, 4000, 300, seed=5, K_new_hook=planted)
    assert (gidx[..., -1] == 4000).all()


def test_pipeline_new_token_loses_a_tie_with_the_kth():
    # the new key equals the k-th ranked cached token's key: equal scores rank the lower index first, so the
    # new token stays out
    B, Hq, Hkv, D, dp, n, k = 1, 8, 2, 64, 16, 4000, 300
    L0 = exact_layer(B, Hq, Hkv, D, dp, n, seed=6)
    s, _ = oracle.score(u16(L0["q_imp"]), u16(L0["K"])[:, :, :n, :dp].copy())
    kth = [oracle.topk(s, k)[0, h] for h in range(Hkv)]
    # the k-th ranked token of each head: the lowest score among the kept, the highest index among equals
    e = []
    for h in range(Hkv):
        sel = kth[h]
        sv = s[0, h, sel]
        low = sel[sv == sv.min()].max()
        e.append(int(low))

    def tie(L):
        kn = L["K_new"].clone()
        for h in range(Hkv):
            kn[0, h] = L["K"][0, h, e[h]]
        L["K_new"] = kn

    gidx, st, _ = run_exact(B, Hq, Hkv, D, dp, n, k, seed=6, K_new_hook=tie)
    assert not (gidx == n).any()


def test_pipeline_all_equal_scores():
    # every cached key equal: one 12-bit bin holds the whole row (more entries than the resolver collects in
    # shared memory), the cut falls inside one tie and goes to the lowest indices
    run_exact(1, 8, 2, 64, 16, 20000, 3000, seed=7, equal_rows=True)


def _stack_parity(w, L_layers, n0, steps, agg=0):
    """tb_decode_layers over L layers and `steps` steps: each layer against oracle.decode_step on its own."""
    cap = n0 + steps
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    stack = tb.DecodeStack(shape, L_layers, w.k, agg=agg, scale=w.scale, n_max=cap - 1)
    lay = []
    for l in range(L_layers):
        Ld = synth.make_layer(w, layer=l, cap=cap, n=n0)
        K, V, Wk = Ld["K"].cuda(), Ld["V"].cuda(), Ld["Wk"].cuda()
        Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
        tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n0)
        lay.append(dict(L=Ld, K=K, V=V, Wk=Wk, Kp=Kp, oK=u16(Ld["K"]).copy(), oV=u16(Ld["V"]).copy(),
                        oKp=u16(Kp).copy(), st=oracle.DecodeState(),
                        out=torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")))
    for t in range(steps):
        n = n0 + t
        ds = [synth.make_step(w, l, t, lay[l]["L"]["outlier_ch"]) for l in range(L_layers)]
        dev = [{k: v.cuda() for k, v in d.items()} for d in ds]
        stack.step(n, q=[d["q"] for d in dev], q_imp=[d["q_imp"] for d in dev], K_new=[d["K_new"] for d in dev],
                   V_new=[d["V_new"] for d in dev], Wk=[y["Wk"] for y in lay], K=[y["K"] for y in lay],
                   V=[y["V"] for y in lay], Kp=[y["Kp"] for y in lay], out=[y["out"] for y in lay])
        torch.cuda.synchronize()
        tb.check_dev_status(stack.status, f"step {t}")
        for l, y in enumerate(lay):
            d = ds[l]
            ref_out, _, _ = oracle.decode_step(
                y["st"], t, n, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=y["L"]["Wk"],
                K=y["oK"], V=y["oV"], Kp=y["oKp"], k=w.k, T=1, r=0, agg=agg, scale=w.scale)
            n_t = n + 1
            kn = np.ascontiguousarray(y["oK"][:, :, n:n + 1])
            _, kp64 = oracle.project(kn, u16(y["L"]["Wk"]))
            assert_kp_close(u16(y["Kp"][:, :, n])[:, :, None], kp64, kp_l1(kn, u16(y["L"]["Wk"])))
            gidx = stack.idx_state[l].cpu().numpy()
            s_ref, _ = oracle.score(d["q_imp"], np.ascontiguousarray(y["oKp"][:, :, :n_t]), agg)
            assert_topk_end_to_end(gidx, s_ref, w.k)
            assert np.array_equal(stack.sel[l].cpu().numpy(), gidx)
            assert (stack.counts[l].cpu().numpy() == w.k).all()
            cnt = np.full((w.B, w.Hkv), w.k, dtype=np.int32)
            ref_g = oracle.attn(d["q"], y["oK"], y["oV"], gidx, cnt, w.scale)
            got = y["out"].float().cpu().numpy()
            assert np.abs(got - ref_g).max() <= OUT_ATOL, (l, t)
            if np.array_equal(gidx, y["st"].idx):
                assert np.abs(got - ref_out).max() <= OUT_ATOL


def test_decode_layers_small_stack():
    w = synth.small(B=2, Hq=16, Hkv=4, D=128, dp=32, N=6000, k=600, seed=71, outliers=4)
    _stack_parity(w, L_layers=4, n0=w.N - 1, steps=3)


def test_decode_layers_max_aggregation_d64():
    w = synth.small(B=1, Hq=8, Hkv=2, D=64, dp=16, N=4096, k=409, seed=72, outliers=2)
    _stack_parity(w, L_layers=3, n0=w.N - 1, steps=2, agg=1)


def test_decode_layers_llama_shape_eight_layers():
    # eight layers of the 32K-token Llama-3-8B-shaped layer, one step
    w = synth.WORKLOADS[1]
    _stack_parity(w, L_layers=8, n0=w.N - 1, steps=1)
