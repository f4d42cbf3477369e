"""K/V in pinned host memory (the offloaded cache of the TokenButler abstract and the gist.science summary,
"Significance"): the same calls and results, only the selected rows cross the host link. (Device-resident K/V
take the attention kernel that gathers with bulk copies; host-resident K/V the one that gathers with 16-byte
copies, so the two agree to the fp32 summation order, not bit for bit, where D allows the former.)"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OUT_ATOL, u16
from test_gpu_decode import run_decode_parity

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


@pytest.mark.parametrize("D", [128, 32])
def test_attention_over_host_kv_equals_device_kv(D):
    # D = 128: the streaming kernel (device K/V) and the tensor-core kernel with 16-byte copies (host K/V);
    # D = 32: the CUDA-core kernel for both, so the same bits
    w = synth.small(B=2, Hq=8, Hkv=2, D=D, dp=16, N=3000, k=300, seed=41)
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, w.N)
    L = synth.make_layer(w, cap=w.N, n=w.N)
    d = synth.make_step(w, 0, 0, L["outlier_ch"])
    g = torch.Generator().manual_seed(5)
    sel = torch.stack([torch.sort(torch.randperm(w.N, generator=g)[: w.k]).values for _ in range(w.B * w.Hkv)])
    sel = sel.reshape(w.B, w.Hkv, w.k).to(torch.int32).cuda()
    ws = tb.workspace(shape, w.N, w.k, w.k)
    st = tb.dev_status()
    q = d["q"].cuda()
    outs = []
    for host in (False, True):
        K, V = (L["K"].pin_memory(), L["V"].pin_memory()) if host else (L["K"].cuda(), L["V"].cuda())
        out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        tb.tb_sparse_decode_attn(shape, q, K, V, sel, None, w.k, w.scale, out, ws, dev_status=st)
        torch.cuda.synchronize()
        tb.check_dev_status(st)
        outs.append(u16(out))
    if D == 32:
        assert np.array_equal(outs[0], outs[1])
    else:
        assert np.abs(oracle.bf16_bits_to_f64(outs[0]) - oracle.bf16_bits_to_f64(outs[1])).max() <= 2e-3
    ref = oracle.attn(d["q"], u16(L["K"]), u16(L["V"]), sel.cpu().numpy(),
                      np.full((w.B, w.Hkv), w.k, dtype=np.int32), w.scale)
    assert np.abs(oracle.bf16_bits_to_f64(outs[1]) - ref).max() <= OUT_ATOL


@pytest.mark.parametrize("fused", [True, False])
def test_decode_step_with_host_kv_matches_oracle(fused):
    # the fused single-exchange step and the modular path, K/V appended to and gathered from host memory
    w = synth.small(B=2, Hq=8, Hkv=2, D=128, dp=32, N=5000, k=500, seed=43, outliers=2)
    run_decode_parity(w, n0=w.N - 1, steps=2, fused=fused, kv_host=True)


def test_decode_interval_with_host_kv_matches_oracle():
    w = synth.small(B=1, Hq=8, Hkv=2, D=128, dp=32, N=3000, k=100, T=4, r=1, seed=44, outliers=4)
    run_decode_parity(w, n0=w.N, steps=6, kv_host=True)


def test_llama_layer_step_with_host_kv():
    # the 32K-token Llama-3-8B-shaped layer with its K/V in pinned host memory, through the single-launch step
    w = synth.WORKLOADS[1]
    run_decode_parity(w, n0=w.N - 1, steps=1, kv_host=True)
