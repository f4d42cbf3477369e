"""Pins for the CPU oracle: each check ties it to something other than itself.

Kinds of pin used: hand-derived worked examples (tests/golden), closed forms,
brute force on tiny inputs, library routines (numpy matmul / einsum, torch's
bf16 conversion and scaled_dot_product_attention in fp64) and invariants the
method's definition fixes (budget k = n gives dense attention, weights sum to
one, neighbour fetching yields a superset).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth


def _f64(bits):
    return oracle.bf16_bits_to_f64(bits)


def _rand_bf16(shape, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(torch.bfloat16)


# ------------------------------------------------------------------ bf16

def test_bf16_golden(golden_dir):
    with open(os.path.join(golden_dir, "bf16_rounding.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        x = math.ldexp(c["m"], c["e"])
        got = int(oracle.bf16_round([x])[0])
        assert got == int(c["bits"], 16), (c["x"], hex(got))


def test_bf16_matches_torch_on_binary32_values():
    # Values exactly representable in binary32 round once either way, so the
    # oracle must agree with torch's RNE conversion bit for bit.
    g = torch.Generator().manual_seed(7)
    x32 = torch.cat([torch.randn(20000, generator=g) * 10.0 ** torch.randint(-30, 30, (20000,), generator=g),
                     torch.tensor([0.0, -0.0, 1.0, -1.0, 65504.0, 3.0e38, -3.0e38, 1e-40, -1e-42])])
    ref = x32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x32.double().numpy())
    assert np.array_equal(got, ref)


def test_bf16_widening_is_exact():
    bits = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    for b, v in zip(bits[:400], t[:400]):
        w = oracle.bf16_to_double(int(b))
        assert (w == v) or (math.isnan(w) and math.isnan(v))


# ------------------------------------------------------------------ projection

def test_project_integer_brute_force():
    # Integer-valued inputs small enough that every sum is an exact bf16.
    B, Hkv, n, D, dp = 2, 3, 5, 8, 4
    K = synth.integer_valued((B, Hkv, n, D), -3, 3, seed=1)
    W = synth.integer_valued((Hkv, D, dp), -3, 3, seed=2)
    Kp, Kp64 = oracle.project(K, W)
    Ki = K.float().int().tolist()
    Wi = W.float().int().tolist()
    for b, h, t, j in itertools.product(range(B), range(Hkv), range(n), range(dp)):
        acc = 0
        for d in range(D):
            acc += Ki[b][h][t][d] * Wi[h][d][j]
        assert Kp64[b, h, t, j] == acc
        assert _f64(Kp[b, h, t, j]) == acc


def test_project_matches_numpy_matmul():
    B, Hkv, n, D, dp = 1, 2, 300, 64, 16
    K = _rand_bf16((B, Hkv, n, D), 3)
    W = _rand_bf16((Hkv, D, dp), 4, std=1 / 8)
    Kp, Kp64 = oracle.project(K, W)
    ref = np.matmul(K.double().numpy(), W.double().numpy()[None])
    assert np.allclose(Kp64, ref, rtol=1e-13, atol=1e-13)
    # torch rounds fp64 -> bf16 through binary32 (two steps); they may differ
    # only where the value sits within 2^-24 relative of a rounding tie.
    tref = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    diff = Kp != tref
    assert diff.mean() < 1e-3
    assert np.all(np.abs(_f64(Kp) - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


# ------------------------------------------------------------------ scores

@pytest.mark.parametrize("agg", [oracle.AGG_MEAN, oracle.AGG_MAX])
def test_score_integer_brute_force(agg):
    B, Hq, Hkv, n, dp = 2, 6, 2, 7, 8
    G = Hq // Hkv
    qi = synth.integer_valued((B, Hq, dp), -4, 4, seed=5)
    Kp = synth.integer_valued((B, Hkv, n, dp), -4, 4, seed=6)
    s, l1 = oracle.score(qi, Kp, agg)
    Q = qi.float().int().tolist()
    P = Kp.float().int().tolist()
    for b, h, t in itertools.product(range(B), range(Hkv), range(n)):
        dots = [sum(Q[b][h * G + g][i] * P[b][h][t][i] for i in range(dp)) for g in range(G)]
        mags = [sum(abs(Q[b][h * G + g][i] * P[b][h][t][i]) for i in range(dp)) for g in range(G)]
        if agg == oracle.AGG_MEAN:
            assert s[b, h, t] == sum(dots) / G
            assert l1[b, h, t] == sum(mags) / G
        else:
            assert s[b, h, t] == max(dots)
            assert l1[b, h, t] == max(mags)


def test_score_mean_is_group_mean_query_and_einsum():
    B, Hq, Hkv, n, dp = 2, 8, 2, 500, 32
    qi = _rand_bf16((B, Hq, dp), 8)
    Kp = _rand_bf16((B, Hkv, n, dp), 9)
    s_mean, _ = oracle.score(qi, Kp, oracle.AGG_MEAN)
    s_max, _ = oracle.score(qi, Kp, oracle.AGG_MAX)
    q = qi.double().numpy().reshape(B, Hkv, Hq // Hkv, dp)
    P = Kp.double().numpy()
    per_g = np.einsum("bhgi,bhti->bhgt", q, P)
    assert np.allclose(s_mean, per_g.mean(2), rtol=1e-12, atol=1e-12)
    assert np.allclose(s_max, per_g.max(2), rtol=0, atol=0)
    qbar = q.mean(2)
    assert np.allclose(s_mean, np.einsum("bhi,bhti->bht", qbar, P), rtol=1e-12, atol=1e-12)
    assert np.all(s_max >= s_mean - 1e-12)


def test_score_group_of_one_mean_equals_max():
    qi = _rand_bf16((1, 4, 16), 10)
    Kp = _rand_bf16((1, 4, 100, 16), 11)
    a, _ = oracle.score(qi, Kp, oracle.AGG_MEAN)
    b, _ = oracle.score(qi, Kp, oracle.AGG_MAX)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ top-k

def _brute_topk(s_row, k):
    # i is selected iff fewer than k elements beat it under (score desc, index asc).
    # O(n^2) rank count: a different algorithm from the oracle's sort.
    n = len(s_row)
    sel = []
    for i in range(n):
        better = 0
        for j in range(n):
            if s_row[j] > s_row[i] or (s_row[j] == s_row[i] and j < i):
                better += 1
        if better < k:
            sel.append(i)
    return sel


def test_topk_golden(golden_dir):
    with open(os.path.join(golden_dir, "topk_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        s = np.array([float(v) for v in c["scores"]], dtype=np.float64)
        got = oracle.topk(s[None], c["k"])[0].tolist()
        assert got == c["idx"], c["why"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_topk_brute_force(seed):
    rng = np.random.default_rng(seed)
    rows, n = 4, 257
    s = rng.standard_normal((rows, n))
    for k in [1, 2, 17, 128, 256, 257]:
        got = oracle.topk(s, k)
        for r in range(rows):
            assert got[r].tolist() == _brute_topk(s[r].tolist(), k)


def test_topk_tie_stress():
    rng = np.random.default_rng(5)
    n = 300
    s = rng.integers(0, 4, size=(3, n)).astype(np.float64)
    for k in [1, 50, 75, 76, 150, 299]:
        got = oracle.topk(s, k)
        for r in range(3):
            assert got[r].tolist() == _brute_topk(s[r].tolist(), k)


def test_topk_shift_invariance_and_full_budget():
    rng = np.random.default_rng(6)
    s = rng.standard_normal((2, 400))
    a = oracle.topk(s, 40)
    b = oracle.topk(s + 1024.0, 40)   # exact shift: 1024 + N(0,1) loses no ordering info at this size
    assert np.array_equal(a, b)
    full = oracle.topk(s, 400)
    assert np.array_equal(full, np.tile(np.arange(400, dtype=np.int32), (2, 1)))
    assert oracle.topk(s, 0).shape == (2, 0)


def test_topk_rejects_nan():
    s = np.array([[1.0, float("nan"), 0.0]])
    with pytest.raises(ValueError):
        oracle.topk(s, 1)


# ------------------------------------------------------------------ expand

def test_expand_golden(golden_dir):
    with open(os.path.join(golden_dir, "expand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        sel, cnt = oracle.expand(np.array([c["idx"]], dtype=np.int32), c["r"], c["n_pred"], c["n_t"])
        assert sel[0, : cnt[0]].tolist() == c["sel"], c["why"]


@pytest.mark.parametrize("r", [0, 1, 2, 5])
def test_expand_brute_force_and_invariants(r):
    rng = np.random.default_rng(10 + r)
    n_pred, k = 200, 30
    for trial in range(5):
        idx = np.sort(rng.choice(n_pred, size=(k,), replace=False)).astype(np.int32)[None]
        n_t = n_pred + trial
        sel, cnt = oracle.expand(idx, r, n_pred, n_t)
        got = sel[0, : cnt[0]].tolist()
        want = set()
        for i in idx[0].tolist():
            want.update(t for t in range(i - r, i + r + 1) if 0 <= t < n_pred)
        want = sorted(want) + list(range(n_pred, n_t))
        assert got == want
        body = got[: len(got) - (n_t - n_pred)]
        assert set(idx[0].tolist()) <= set(body)                       # superset
        assert k <= len(body) <= min(n_pred, k * (2 * r + 1))          # bounds
        assert all(a < b for a, b in zip(got, got[1:]))                # sorted, unique
        if r == 0:
            assert body == idx[0].tolist()


# ------------------------------------------------------------------ attention

def test_attn_golden(golden_dir):
    with open(os.path.join(golden_dir, "attn_closed_form.json")) as f:
        cases = json.load(f)["cases"]
    e = math.e
    for c in cases:
        D = c["D"]
        q = torch.tensor([[c["q"]]], dtype=torch.bfloat16)
        K = torch.tensor([[c["K"]]], dtype=torch.bfloat16)
        V = torch.tensor([[c["V"]]], dtype=torch.bfloat16)
        sel = np.array([[c["sel"]]], dtype=np.int32)
        cnt = np.array([[len(c["sel"])]], dtype=np.int32)
        out = oracle.attn(q, K, V, sel, cnt, c["scale"])
        want = [eval(expr.replace("^", "**"), {"e": e}) for expr in c["out"]]
        assert np.allclose(out[0, 0, :D], want, rtol=1e-14, atol=1e-14)


def _sdpa_ref(q, K, V, sel, scale):
    """torch scaled_dot_product_attention in fp64 on the gathered rows, one (b, h) row."""
    Kg = K[sel].double()[None, None]
    Vg = V[sel].double()[None, None]
    return torch.nn.functional.scaled_dot_product_attention(
        q.double()[None, :, None, :].transpose(0, 1).reshape(1, -1, 1, q.shape[-1]),
        Kg.expand(1, q.shape[0], -1, -1), Vg.expand(1, q.shape[0], -1, -1), scale=scale)[0, :, 0, :]


def test_attn_matches_sdpa_fp64():
    w = synth.small(B=2, Hq=8, Hkv=2, D=32, dp=8, N=300, k=40, seed=3)
    L = synth.make_layer(w)
    rng = np.random.default_rng(3)
    sel = np.stack([np.stack([np.sort(rng.choice(w.N, 40, replace=False)) for _ in range(w.Hkv)])
                    for _ in range(w.B)]).astype(np.int32)
    cnt = np.full((w.B, w.Hkv), 40, dtype=np.int32)
    out, wsum = oracle.attn(L["q"], L["K"], L["V"], sel, cnt, w.scale, with_wsum=True)
    for b in range(w.B):
        for h in range(w.Hkv):
            qh = L["q"][b, h * w.G:(h + 1) * w.G]
            ref = _sdpa_ref(qh, L["K"][b, h], L["V"][b, h], torch.from_numpy(sel[b, h]).long(), w.scale)
            assert np.allclose(out[b, h * w.G:(h + 1) * w.G], ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(np.abs(wsum - 1.0) <= 1e-12)


def test_attn_special_cases():
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=50, seed=4)
    L = synth.make_layer(w)
    Vf = L["V"].double().numpy()
    # one selected row: the output is that V row exactly
    sel = np.array([[[7], [33]]], dtype=np.int32)
    cnt = np.ones((1, 2), dtype=np.int32)
    out = oracle.attn(L["q"], L["K"], L["V"], sel, cnt, w.scale)
    assert np.array_equal(out[0, 0], Vf[0, 0, 7]) and np.array_equal(out[0, 3], Vf[0, 1, 33])
    # zero query: uniform weights, the output is the mean of the selected V rows
    sel = np.array([[[1, 4, 9, 20], [0, 2, 3, 49]]], dtype=np.int32)
    cnt = np.full((1, 2), 4, dtype=np.int32)
    q0 = torch.zeros_like(L["q"])
    out = oracle.attn(q0, L["K"], L["V"], sel, cnt, w.scale)
    assert np.allclose(out[0, 1], Vf[0, 0, [1, 4, 9, 20]].mean(0), rtol=1e-14, atol=1e-14)
    # permuting the selection changes nothing (up to fp64 summation order)
    perm = sel[:, :, ::-1].copy()
    a = oracle.attn(L["q"], L["K"], L["V"], sel, cnt, w.scale)
    b = oracle.attn(L["q"], L["K"], L["V"], perm, cnt, w.scale)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)


def test_full_budget_reproduces_dense():
    w = synth.small(B=1, Hq=8, Hkv=2, D=32, dp=8, N=200, seed=5)
    L = synth.make_layer(w)
    Kp, _ = oracle.project(L["K"], L["Wk"])
    s, _ = oracle.score(L["q_imp"], Kp)
    idx = oracle.topk(s, w.N)
    sel, cnt = oracle.expand(idx, 0, w.N, w.N)
    sparse = oracle.attn(L["q"], L["K"], L["V"], sel, cnt, w.scale)
    dense = oracle.dense_attn(L["q"], L["K"], L["V"], w.N, w.scale)
    assert np.array_equal(sparse, dense)
    for b, h in itertools.product(range(w.B), range(w.Hkv)):
        ref = _sdpa_ref(L["q"][b, h * w.G:(h + 1) * w.G], L["K"][b, h], L["V"][b, h],
                        torch.arange(w.N), w.scale)
        assert np.allclose(dense[b, h * w.G:(h + 1) * w.G], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_planted_heavy_hitters_are_selected():
    # The long-context recipe plants tokens whose keys align with the group's
    # importance query; every one of them must make the budget.
    w = synth.Workload("planted-small", B=1, Hq=8, Hkv=2, D=64, dp=16, N=4096, k=64,
                       outliers=4, planted=16, seed=9)
    L = synth.make_layer(w)
    Kp, _ = oracle.project(L["K"], L["Wk"])
    s, _ = oracle.score(L["q_imp"], Kp)
    idx = oracle.topk(s, w.k)
    for h in range(w.Hkv):
        assert set(L["planted_pos"][0, h].tolist()) <= set(idx[0, h].tolist())


# ------------------------------------------------------------------ decode steps

def _run_steps(w, T, r, steps, k, budget_neighbours=False):
    L = synth.make_layer(w, cap=w.N + steps, n=w.N)
    K = oracle.as_u16(L["K"]).copy()
    V = oracle.as_u16(L["V"]).copy()
    Kp = np.zeros((w.B, w.Hkv, w.N + steps, w.dp), dtype=np.uint16)
    Kp[:, :, : w.N], _ = oracle.project(np.ascontiguousarray(K[:, :, : w.N]), L["Wk"])
    st = oracle.DecodeState()
    outs = []
    for t in range(steps):
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        out, sel, cnt = oracle.decode_step(st, t, w.N + t, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"],
                                           V_new=d["V_new"], Wk=L["Wk"], K=K, V=V, Kp=Kp, k=k, T=T, r=r,
                                           agg=oracle.AGG_MEAN, scale=w.scale, budget_neighbours=budget_neighbours)
        outs.append((out, sel, cnt, st.idx.copy(), st.n_pred))
    return outs, (K, V, Kp, L)


def test_decode_interval_one_is_per_step_selection():
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=120, seed=11)
    outs, (K, V, Kp, L) = _run_steps(w, T=1, r=0, steps=4, k=10)
    for t, (out, sel, cnt, idx, n_pred) in enumerate(outs):
        n_t = w.N + t + 1
        assert n_pred == n_t
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        s, _ = oracle.score(d["q_imp"], np.ascontiguousarray(Kp[:, :, :n_t]))
        want = oracle.topk(s, 10)
        assert np.array_equal(sel[:, :, :10], want) and np.all(cnt == 10)


def test_prediction_sees_the_token_appended_at_its_own_step():
    # Reading of the prediction interval: a prediction step scores the cache
    # after its own append. The appended key is built to out-score every
    # cached token by far (K_new_d = 8 sign((Wk qbar)_d), qbar the group's mean
    # importance query), so the new token must be among the k kept.
    w = synth.small(B=2, Hq=4, Hkv=2, D=16, dp=8, N=100, seed=15)
    G = w.Hq // w.Hkv
    L = synth.make_layer(w, cap=w.N + 1, n=w.N)
    K = oracle.as_u16(L["K"]).copy()
    V = oracle.as_u16(L["V"]).copy()
    Kp = np.zeros((w.B, w.Hkv, w.N + 1, w.dp), dtype=np.uint16)
    Kp[:, :, : w.N], _ = oracle.project(np.ascontiguousarray(K[:, :, : w.N]), L["Wk"])
    d = synth.make_step(w, 0, 0, L["outlier_ch"])
    Wk = _f64(oracle.as_u16(L["Wk"]))                                   # [Hkv, D, dp]
    qbar = _f64(oracle.as_u16(d["q_imp"])).reshape(w.B, w.Hkv, G, w.dp).mean(axis=2)
    direction = np.einsum("hdj,bhj->bhd", Wk, qbar)
    K_new = torch.from_numpy(np.where(direction >= 0, 8.0, -8.0)).to(torch.bfloat16)
    st = oracle.DecodeState()
    out, sel, cnt = oracle.decode_step(st, 0, w.N, q=d["q"], q_imp=d["q_imp"], K_new=K_new, V_new=d["V_new"],
                                       Wk=L["Wk"], K=K, V=V, Kp=Kp, k=5, T=4, r=0, agg=oracle.AGG_MEAN,
                                       scale=w.scale)
    assert st.n_pred == w.N + 1
    for b, h in itertools.product(range(w.B), range(w.Hkv)):
        assert w.N in st.idx[b, h].tolist()
        assert w.N in sel[b, h, : cnt[b, h]].tolist()


def test_decode_interval_reuse_superset_and_tail():
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=150, seed=12)
    T, r, k = 4, 1, 12
    outs, _ = _run_steps(w, T=T, r=r, steps=9, k=k)
    for t, (out, sel, cnt, idx, n_pred) in enumerate(outs):
        t0 = (t // T) * T
        assert n_pred == w.N + t0 + 1
        n_t = w.N + t + 1
        for b, h in itertools.product(range(w.B), range(w.Hkv)):
            s = sel[b, h, : cnt[b, h]].tolist()
            assert set(idx[b, h].tolist()) <= set(s)
            assert s[len(s) - (n_t - n_pred):] == list(range(n_pred, n_t))
            body = len(s) - (n_t - n_pred)
            assert k <= body <= min(n_pred, k * (2 * r + 1))


def test_budget_preserving_neighbours_centres_and_bound():
    # k // (2r + 1) centres (at least one); r = 0 keeps k
    assert [oracle.centres(9, 1, True), oracle.centres(9, 0, True), oracle.centres(2, 2, True),
            oracle.centres(9, 1, False)] == [3, 9, 1, 9]
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=160, seed=13)
    T, r, k = 3, 2, 25
    kc = k // (2 * r + 1)
    outs, (K, V, Kp, L) = _run_steps(w, T=T, r=r, steps=6, k=k, budget_neighbours=True)
    for t, (out, sel, cnt, idx, n_pred) in enumerate(outs):
        n_t = w.N + t + 1
        assert idx.shape[-1] == kc
        if t % T == 0:
            # the centres are the top kc by a brute-force rank count on the step's own scores
            d = synth.make_step(w, 0, t, L["outlier_ch"])
            s_, _ = oracle.score(d["q_imp"], np.ascontiguousarray(Kp[:, :, :n_t]))
            for b, h in itertools.product(range(w.B), range(w.Hkv)):
                v = s_[b, h]
                rank = [sum(1 for j in range(n_t) if (v[j], -j) > (v[i], -i)) for i in range(n_t)]
                assert idx[b, h].tolist() == [i for i in range(n_t) if rank[i] < kc]
        for b, h in itertools.product(range(w.B), range(w.Hkv)):
            s = sel[b, h, : cnt[b, h]].tolist()
            body = s[: len(s) - (n_t - n_pred)]
            want = sorted({j for i in idx[b, h].tolist() for j in range(i - r, i + r + 1) if 0 <= j < n_pred})
            assert body == want
            assert kc <= len(body) <= k                                  # within the budget


def test_buffered_step_sink_window_batches_and_centres():
    # sink and local-window buffers with batched projection: the structure of every selection
    w = synth.small(B=1, Hq=4, Hkv=2, D=16, dp=8, N=90, seed=14)
    S, W, T, r, k = 5, 8, 3, 1, 12
    steps = 14
    L = synth.make_layer(w, cap=w.N + steps, n=w.N)
    K = oracle.as_u16(L["K"]).copy()
    V = oracle.as_u16(L["V"]).copy()
    Kp = np.zeros((w.B, w.Hkv, w.N + steps, w.dp), dtype=np.uint16)
    P0 = 64                                            # rows projected at prefill
    Kp[:, :, :P0], _ = oracle.project(np.ascontiguousarray(K[:, :, :P0]), L["Wk"])
    st = oracle.BufferedState(P0)
    for t in range(steps):
        n = w.N + t
        n_t = n + 1
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        pe_before = st.proj_end
        out, sel, cnt = oracle.decode_step_buffered(st, t, n, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"],
                                                    V_new=d["V_new"], Wk=L["Wk"], K=K, V=V, Kp=Kp, k=k, T=T, r=r,
                                                    agg=oracle.AGG_MEAN, scale=w.scale, sink=S, window=W)
        P = st.proj_end
        assert (P - pe_before) % W == 0 and P <= n_t
        if t % T == 0:
            assert W <= n_t - P < 2 * W                      # the window after the batches
            want_kp, _ = oracle.project(np.ascontiguousarray(K[:, :, :P]), L["Wk"])
            assert np.array_equal(Kp[:, :, :P], want_kp)      # batches equal one projection of all rows
            s_, _ = oracle.score(d["q_imp"], np.ascontiguousarray(Kp[:, :, S:P]))
            for b, h in itertools.product(range(w.B), range(w.Hkv)):
                v = s_[b, h]
                m = P - S
                rank = [sum(1 for j in range(m) if (v[j], -j) > (v[i], -i)) for i in range(m)]
                assert st.idx[b, h].tolist() == [i for i in range(m) if rank[i] < min(k, m)]
        for b, h in itertools.product(range(w.B), range(w.Hkv)):
            row = sel[b, h, : cnt[b, h]].tolist()
            assert all(a < c for a, c in zip(row, row[1:]))   # ascending, unique
            assert set(range(min(S, n_t))) <= set(row)        # sink
            assert set(range(max(P, S), n_t)) <= set(row)     # window (and the interval's new tokens)
            body = [j for j in row if S <= j < P]
            assert len(body) <= min(k, P - S) * (2 * r + 1)
            assert set(S + i for i in st.idx[b, h].tolist()) <= set(body)


# ------------------------------------------------------------------ predictor

def test_predictor_matches_torch_fp64_and_silu_identities():
    g = torch.Generator().manual_seed(21)
    B, E, F, O = 3, 64, 32, 24
    x = torch.randn(B, E, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(F, E, generator=g) / 8).to(torch.bfloat16)
    W2 = (torch.randn(O, F, generator=g) / 6).to(torch.bfloat16)
    bits, y, h = oracle.predict_queries(x, W1, W2)
    # the library routines: torch's SiLU and matmul in fp64 on the same bf16 values
    ht = torch.nn.functional.silu(x.double() @ W1.double().T)
    yt = ht @ W2.double().T
    assert np.allclose(h, ht.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(y, yt.numpy(), rtol=1e-12, atol=1e-14)
    assert np.array_equal(bits, oracle.bf16_round(yt.numpy()))
    # SiLU: odd part is the identity, zero at zero, -> v for large v, -> 0 for very negative v
    v = np.linspace(-20, 20, 81)
    assert np.allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=0, atol=1e-12)
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12 and abs(oracle.silu(-40.0)) < 1e-12


def test_ragged_step_with_equal_lengths_is_the_batched_step():
    # the ragged oracle applies the step per sequence: with equal lengths it must equal the batched step
    w = synth.small(B=3, Hq=4, Hkv=2, D=16, dp=8, N=100, seed=15)
    steps, T, r, k = 5, 2, 1, 9
    L = synth.make_layer(w, cap=w.N + steps, n=w.N)
    arrs = []
    for _ in range(2):
        K = oracle.as_u16(L["K"]).copy()
        V = oracle.as_u16(L["V"]).copy()
        Kp = np.zeros((w.B, w.Hkv, w.N + steps, w.dp), dtype=np.uint16)
        Kp[:, :, : w.N], _ = oracle.project(np.ascontiguousarray(K[:, :, : w.N]), L["Wk"])
        arrs.append((K, V, Kp))
    st = oracle.DecodeState()
    sts = [oracle.DecodeState() for _ in range(w.B)]
    for t in range(steps):
        d = synth.make_step(w, 0, t, L["outlier_ch"])
        kw = dict(q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=L["Wk"], k=k, T=T, r=r,
                  agg=oracle.AGG_MEAN, scale=w.scale)
        K, V, Kp = arrs[0]
        o1, s1, c1 = oracle.decode_step(st, t, w.N + t, K=K, V=V, Kp=Kp, **kw)
        K, V, Kp = arrs[1]
        o2, s2, c2 = oracle.decode_step_ragged(sts, t, [w.N + t] * w.B, K=K, V=V, Kp=Kp, **kw)
        assert np.array_equal(c1, c2) and np.array_equal(o1, o2)
        for b, h in itertools.product(range(w.B), range(w.Hkv)):
            assert np.array_equal(s1[b, h, : c1[b, h]], s2[b, h, : c2[b, h]])
    assert np.array_equal(arrs[0][2], arrs[1][2])


def test_ragged_step_with_unequal_lengths():
    # Sequences of different lengths in one batch: each sees only its own
    # n_b + 1 rows. The shortest one keeps all of its tokens (k = n_0 + 1), so
    # its output is dense attention over exactly those rows (torch SDPA in
    # fp64); the others keep the brute-force top k of their own scores; and
    # changing one sequence's data leaves the others' outputs unchanged.
    w = synth.small(B=3, Hq=4, Hkv=2, D=16, dp=8, N=74, seed=16)
    G = w.Hq // w.Hkv
    ns = [40, 73, 55]
    k = ns[0] + 1
    L = synth.make_layer(w, cap=w.N + 1, n=w.N)
    d = synth.make_step(w, 0, 0, L["outlier_ch"])

    def run(K_in, q_in):
        K = oracle.as_u16(K_in).copy()
        V = oracle.as_u16(L["V"]).copy()
        Kp = np.zeros((w.B, w.Hkv, w.N + 1, w.dp), dtype=np.uint16)
        Kp[:, :, : w.N], _ = oracle.project(np.ascontiguousarray(K[:, :, : w.N]), L["Wk"])
        sts = [oracle.DecodeState() for _ in range(w.B)]
        out, sel, cnt = oracle.decode_step_ragged(sts, 0, ns, q=q_in, q_imp=d["q_imp"], K_new=d["K_new"],
                                                  V_new=d["V_new"], Wk=L["Wk"], K=K, V=V, Kp=Kp, k=k, T=1, r=0,
                                                  agg=oracle.AGG_MEAN, scale=w.scale)
        return out, sel, cnt, K, V, Kp

    out, sel, cnt, K, V, Kp = run(L["K"], d["q"])
    for b, nb in enumerate(ns):
        assert np.array_equal(K[b, :, nb], oracle.as_u16(d["K_new"])[b])
        for h in range(w.Hkv):
            row = sel[b, h, : cnt[b, h]].tolist()
            assert cnt[b, h] == k and row == sorted(row) and max(row) <= nb
            s, _ = oracle.score(oracle.as_u16(d["q_imp"])[b:b + 1], np.ascontiguousarray(Kp[b:b + 1, :, : nb + 1]))
            v = s[0, h]
            rank = [sum(1 for j in range(nb + 1) if (v[j], -j) > (v[i], -i)) for i in range(nb + 1)]
            assert row == [i for i in range(nb + 1) if rank[i] < k]
    n0 = ns[0] + 1
    qf = torch.from_numpy(_f64(oracle.as_u16(d["q"]))[0]).reshape(1, w.Hq, 1, w.D)
    Kf = torch.from_numpy(_f64(K[0, :, :n0])).repeat_interleave(G, dim=0)[None]
    Vf = torch.from_numpy(_f64(V[0, :, :n0])).repeat_interleave(G, dim=0)[None]
    dense = torch.nn.functional.scaled_dot_product_attention(qf, Kf, Vf, scale=w.scale)[0, :, 0].numpy()
    assert np.allclose(out[0], dense, rtol=0, atol=1e-12)
    # sequence 2's keys and queries changed: sequences 0 and 1 are unaffected
    K2 = L["K"].clone()
    K2[2] = -K2[2]
    q2 = d["q"].clone()
    q2[2] = -q2[2]
    out_b, _, _, _, _, _ = run(K2, q2)
    assert np.array_equal(out_b[:2], out[:2]) and not np.array_equal(out_b[2], out[2])
