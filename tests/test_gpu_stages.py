"""Stage-wise GPU parity: each C-ABI call against the CPU oracle on identical inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OUT_ATOL, assert_kp_close, assert_scores_close, bf16_ulp_diff, kp_l1, u16

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


def _status():
    return tb.dev_status()


# ------------------------------------------------------------------ projection

@pytest.mark.parametrize("B,Hkv,n_new,D,dp,pos0", [(1, 8, 2048, 64, 16, 0), (2, 3, 1000, 128, 32, 17),
                                                   (1, 2, 77, 32, 8, 5), (1, 4, 300, 128, 64, 0),
                                                   # several tiles per CTA, ranges crossing heads and batches
                                                   (2, 3, 128 * 150 + 37, 128, 32, 0),
                                                   # a CTA's range spans every KV head
                                                   (160, 2, 128, 64, 16, 0)])
def test_project_within_one_ulp(B, Hkv, n_new, D, dp, pos0):
    g = torch.Generator().manual_seed(n_new)
    cap = pos0 + n_new + 3
    K = torch.randn((B, Hkv, cap, D), generator=g).to(torch.bfloat16)
    Wk = (torch.randn((Hkv, D, dp), generator=g) / math.sqrt(D)).to(torch.bfloat16)
    shape = tb.Shape(B, Hkv, Hkv, D, dp, cap)
    Kd, Wd = K.cuda(), Wk.cuda()
    Kp = torch.zeros((B, Hkv, cap, dp), dtype=torch.bfloat16, device="cuda")
    st = _status()
    tb.tb_project_append(shape, Kd, cap, Wd, Kp, pos0, n_new, dev_status=st, K_src_offset_rows=pos0)
    torch.cuda.synchronize()
    tb.check_dev_status(st)
    got = u16(Kp)[:, :, pos0:pos0 + n_new]
    Kin = np.ascontiguousarray(u16(K)[:, :, pos0:pos0 + n_new])
    want, want64 = oracle.project(Kin, Wk)
    assert_kp_close(got, want64, kp_l1(Kin, u16(Wk)))
    assert (got != want).mean() < 0.01
    # rows outside [pos0, pos0 + n_new) untouched
    assert not u16(Kp)[:, :, :pos0].any() and not u16(Kp)[:, :, pos0 + n_new:].any()


def test_project_integer_exact():
    B, Hkv, n, D, dp = 1, 2, 260, 64, 16
    K = synth.integer_valued((B, Hkv, n, D), -2, 2, seed=3)
    Wk = synth.integer_valued((Hkv, D, dp), -1, 1, seed=4)
    shape = tb.Shape(B, Hkv, Hkv, D, dp, n)
    Kp = torch.zeros((B, Hkv, n, dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K.cuda(), n, Wk.cuda(), Kp, 0, n)
    torch.cuda.synchronize()
    want, _ = oracle.project(K, Wk)
    assert np.array_equal(u16(Kp), want)


# ------------------------------------------------------------------ scores

@pytest.mark.parametrize("B,Hq,Hkv,n,dp,agg", [(1, 8, 8, 2048, 16, 0), (1, 32, 8, 32768, 32, 0),
                                               (1, 32, 8, 32768, 32, 1), (2, 6, 2, 1001, 24, 0),
                                               (2, 6, 2, 1001, 24, 1), (1, 4, 1, 5000, 64, 0),
                                               (3, 12, 4, 257, 8, 1)])
def test_score_parity(B, Hq, Hkv, n, dp, agg):
    g = torch.Generator().manual_seed(n + dp)
    cap = n + 5
    qi = torch.randn((B, Hq, dp), generator=g).to(torch.bfloat16)
    Kp = (torch.randn((B, Hkv, cap, dp), generator=g) * 2).to(torch.bfloat16)
    shape = tb.Shape(B, Hq, Hkv, 64, dp, cap)
    s = torch.empty((B, Hkv, n), dtype=torch.float32, device="cuda")
    tb.tb_score(shape, qi.cuda(), Kp.cuda(), n, s, agg=agg)
    torch.cuda.synchronize()
    ref, l1 = oracle.score(qi, np.ascontiguousarray(u16(Kp)[:, :, :n]), agg)
    assert_scores_close(s.cpu().numpy(), ref, l1)


@pytest.mark.parametrize("agg", [0, 1])
def test_score_integer_bit_exact(agg):
    B, Hq, Hkv, n, dp = 1, 16, 4, 3000, 32
    qi = synth.integer_valued((B, Hq, dp), -4, 4, seed=8)
    Kp = synth.integer_valued((B, Hkv, n, dp), -4, 4, seed=9)
    shape = tb.Shape(B, Hq, Hkv, 64, dp, n)
    s = torch.empty((B, Hkv, n), dtype=torch.float32, device="cuda")
    tb.tb_score(shape, qi.cuda(), Kp.cuda(), n, s, agg=agg)
    torch.cuda.synchronize()
    ref, _ = oracle.score(qi, Kp, agg)
    assert np.array_equal(s.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------------ top-k

def _topk_gpu(s_cpu: torch.Tensor, k: int, expect_status=0):
    B, Hkv, n = s_cpu.shape
    shape = tb.Shape(B, Hkv, Hkv, 64, 16, max(n, 1))
    ws = tb.workspace(shape, n, k, k)
    idx = torch.full((B, Hkv, k), -7, dtype=torch.int32, device="cuda")
    st = _status()
    sd = s_cpu.cuda()
    tb.tb_topk(shape, sd, n, k, idx, ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    first = idx.cpu().numpy()
    # a second call on the same workspace (its control words were reset) agrees
    idx2 = torch.full_like(idx, -7)
    tb.tb_topk(shape, sd, n, k, idx2, ws, dev_status=st)
    torch.cuda.synchronize()
    assert np.array_equal(idx2.cpu().numpy(), first)
    return first


@pytest.mark.parametrize("B,Hkv,n,k", [(1, 8, 2048, 128), (1, 8, 32768, 3277), (1, 1, 1, 1), (2, 3, 1000, 1),
                                       (2, 3, 1000, 1000), (1, 2, 4097, 999), (1, 4, 70001, 7000),
                                       (2, 8, 16385, 1024), (1, 2, 65536, 65535)])
def test_topk_bit_exact_random(B, Hkv, n, k):
    g = torch.Generator().manual_seed(n * 31 + k)
    s = torch.randn((B, Hkv, n), generator=g) * 5.0
    got = _topk_gpu(s, k)
    want = oracle.topk(s.numpy(), k)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("n,k,levels", [(2048, 700, 4), (20000, 9000, 4), (20000, 5001, 3), (50000, 123, 2),
                                        (9000, 4500, 1)])
def test_topk_tie_stress(n, k, levels):
    # a few distinct values: the k-th element sits inside a large tie, which
    # must go to the lowest indices (bins far beyond the candidate list)
    g = torch.Generator().manual_seed(n + k)
    s = torch.randint(0, levels, (1, 3, n), generator=g).float() * 0.5 - 0.25
    got = _topk_gpu(s, k)
    assert np.array_equal(got, oracle.topk(s.numpy(), k))


def test_topk_near_ties_and_specials():
    g = torch.Generator().manual_seed(5)
    n = 30000
    s = torch.round(torch.randn((2, 2, n), generator=g) * 1000.0) / 1000.0   # many exact repeats
    s[0, 0, :100] = 0.0
    s[0, 0, 100:200] = -0.0
    s[0, 1, 5] = float("inf")
    s[0, 1, 7] = float("-inf")
    s[1, 0] = s[1, 0].abs().neg()        # all non-positive
    for k in [1, 50, 2999, 15000, 29999]:
        got = _topk_gpu(s, k)
        assert np.array_equal(got, oracle.topk(s.numpy(), k)), k


def test_topk_shift_invariance():
    g = torch.Generator().manual_seed(6)
    s = torch.randn((1, 4, 12345), generator=g)
    a = _topk_gpu(s, 1234)
    b = _topk_gpu(s * 0.5 + 1024.0, 1234)   # order-preserving in fp32 at this scale? check vs oracle instead
    assert np.array_equal(b, oracle.topk((s * 0.5 + 1024.0).numpy(), 1234))
    assert np.array_equal(a, oracle.topk(s.numpy(), 1234))


def test_topk_nan_is_flagged():
    s = torch.randn((1, 2, 500))
    s[0, 1, 17] = float("nan")
    got = _topk_gpu(s, 10, expect_status=tb.TB_ERR_NONFINITE)
    assert 17 not in got[0, 1].tolist()
    assert np.array_equal(got[0, 0], oracle.topk(s[0, 0].numpy()[None], 10)[0])


# ------------------------------------------------------------------ expand

@pytest.mark.parametrize("r,k,n_pred,tail", [(0, 50, 1000, 0), (1, 1024, 16385, 15), (3, 100, 500, 2),
                                             (1, 300, 301, 4), (5, 1, 7, 0)])
def test_expand_exact(r, k, n_pred, tail):
    rng = np.random.default_rng(r * 100 + k)
    B, Hkv = 2, 3
    idx = np.stack([np.stack([np.sort(rng.choice(n_pred, k, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)]).astype(np.int32)
    n_t = n_pred + tail
    stride = min(n_pred, k * (2 * r + 1)) + tail + 3
    shape = tb.Shape(B, Hkv, Hkv, 64, 16, n_t + 1)
    sel = torch.full((B, Hkv, stride), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    st = _status()
    tb.tb_expand(shape, torch.from_numpy(idx).cuda(), k, r, n_pred, n_t, sel, stride, cnt, dev_status=st)
    torch.cuda.synchronize()
    tb.check_dev_status(st)
    want_sel, want_cnt = oracle.expand(idx, r, n_pred, n_t, sel_stride=stride)
    got_cnt = cnt.cpu().numpy()
    assert np.array_equal(got_cnt, want_cnt)
    gs = sel.cpu().numpy()
    for b in range(B):
        for h in range(Hkv):
            c = want_cnt[b, h]
            assert np.array_equal(gs[b, h, :c], want_sel[b, h, :c])


def test_expand_overflow_flagged():
    idx = torch.tensor([[[0, 10, 20]]], dtype=torch.int32, device="cuda")
    shape = tb.Shape(1, 1, 1, 64, 16, 64)
    sel = torch.zeros((1, 1, 5), dtype=torch.int32, device="cuda")
    cnt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    st = _status()
    tb.tb_expand(shape, idx, 3, 1, 30, 30, sel, 5, cnt, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_ERR_INVALID_ARG and int(cnt.item()) == 5


# ------------------------------------------------------------------ attention

def _attn_case(w: synth.Workload, sel: np.ndarray, counts: np.ndarray, L=None):
    L = L or synth.make_layer(w)
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, w.N)
    stride = sel.shape[-1]
    ws = tb.workspace(shape, w.N, stride, stride)
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    st = _status()
    tb.tb_sparse_decode_attn(shape, L["q"].cuda(), L["K"].cuda(), L["V"].cuda(), torch.from_numpy(sel).cuda(),
                             torch.from_numpy(counts).cuda(), stride, w.scale, out, ws, dev_status=st)
    torch.cuda.synchronize()
    tb.check_dev_status(st)
    ref = oracle.attn(L["q"], L["K"], L["V"], sel, counts, w.scale)
    return out.float().cpu().numpy(), ref, L, ws


@pytest.mark.parametrize("wi,k", [(0, 128), (1, 3277)])
def test_attn_parity_workloads(wi, k):
    w = synth.WORKLOADS[wi]
    rng = np.random.default_rng(wi)
    sel = np.stack([np.stack([np.sort(rng.choice(w.N, k, replace=False)) for _ in range(w.Hkv)])
                    for _ in range(w.B)]).astype(np.int32)
    counts = np.full((w.B, w.Hkv), k, dtype=np.int32)
    got, ref, _, _ = _attn_case(w, sel, counts)
    assert np.abs(got - ref).max() <= OUT_ATOL


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 2, 128), (10, 2, 64), (32, 2, 64), (24, 2, 128), (3, 3, 128)])
def test_attn_group_sizes(Hq, Hkv, D):
    """Group sizes on both sides of the eight heads one tensor-core tile column holds, odd sizes included."""
    w = synth.small(B=2, Hq=Hq, Hkv=Hkv, D=D, dp=16, N=3000, seed=Hq * 7 + D)
    rng = np.random.default_rng(Hq)
    stride = 1100
    sel = np.stack([np.stack([np.sort(rng.choice(w.N, stride, replace=False)) for _ in range(w.Hkv)])
                    for _ in range(w.B)]).astype(np.int32)
    counts = rng.integers(1, stride + 1, size=(w.B, w.Hkv)).astype(np.int32)
    got, ref, _, _ = _attn_case(w, sel, counts)
    assert np.abs(got - ref).max() <= OUT_ATOL


def test_attn_ragged_counts_and_single_row():
    w = synth.small(B=2, Hq=8, Hkv=2, D=128, dp=32, N=5000, seed=21)
    rng = np.random.default_rng(1)
    stride = 700
    sel = rng.integers(0, w.N, size=(w.B, w.Hkv, stride)).astype(np.int32)
    counts = np.array([[1, 699], [64, 65]], dtype=np.int32)
    got, ref, L, _ = _attn_case(w, sel, counts)
    assert np.abs(got - ref).max() <= OUT_ATOL
    # a single selected row returns that V row (exact after bf16 rounding)
    V = L["V"].float().numpy()
    for hq in range(4):
        assert np.array_equal(got[0, hq], V[0, 0, sel[0, 0, 0]])


def test_attn_full_selection_is_dense():
    w = synth.WORKLOADS[0]
    sel = np.broadcast_to(np.arange(w.N, dtype=np.int32), (w.B, w.Hkv, w.N)).copy()
    counts = np.full((w.B, w.Hkv), w.N, dtype=np.int32)
    got, ref, L, _ = _attn_case(w, sel, counts)
    dense = oracle.dense_attn(L["q"], L["K"], L["V"], w.N, w.scale)
    assert np.array_equal(ref, dense)
    assert np.abs(got - dense).max() <= OUT_ATOL


def test_attn_bad_index_flagged():
    w = synth.small(B=1, Hq=4, Hkv=1, D=64, dp=16, N=100, seed=2)
    L = synth.make_layer(w)
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, w.N)
    sel = torch.tensor([[[3, 5, 100, -1]]], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([[4]], dtype=torch.int32, device="cuda")
    ws = tb.workspace(shape, w.N, 4, 4)
    out = torch.empty((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    st = _status()
    tb.tb_sparse_decode_attn(shape, L["q"].cuda(), L["K"].cuda(), L["V"].cuda(), sel, cnt, 4, w.scale, out, ws,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == tb.TB_ERR_INVALID_ARG
    ref = oracle.attn(L["q"], L["K"], L["V"], np.array([[[3, 5]]], dtype=np.int32),
                      np.array([[2]], dtype=np.int32), w.scale)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= OUT_ATOL
