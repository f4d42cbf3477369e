"""A bounded device-side wait that runs out ends the call with TB_ERR_TIMEOUT instead of hanging, the context
stays usable, and a zero-filled workspace gives the normal result again.

The single-launch decode step's CTAs meet at a per-row exchange (a counter every CTA of the row adds to, which
each then waits on, for at most a fixed time). The workspace's test block (zero in normal use) lets one CTA of
row 0 leave out its arrival, so nothing ever completes that row's exchange: a barrier that nothing sets, no
fault. The block also shortens the limit to one millisecond so the test is quick.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OUT_ATOL, u16
from test_gpu_decode import ROWCTL_BYTES

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


def _arm(ws: torch.Tensor, rows: int, limit_ns: int, skip_cta: int):
    """Write the test block: it follows the rows' control blocks, at the next 256-byte boundary."""
    off = -(-(rows * ROWCTL_BYTES) // 256) * 256
    blk = np.zeros(16, dtype=np.uint8)
    blk[:8] = np.frombuffer(np.uint64(limit_ns).tobytes(), dtype=np.uint8)
    blk[8:12] = np.frombuffer(np.int32(skip_cta).tobytes(), dtype=np.uint8)
    ws[off:off + 16].copy_(torch.from_numpy(blk))


def test_exchange_wait_runs_out_and_the_workspace_recovers():
    w = synth.small(B=1, Hq=32, Hkv=8, D=128, dp=32, N=8192, k=820, seed=91, outliers=4)
    n0, cap = w.N - 1, w.N
    shape = tb.Shape(w.B, w.Hq, w.Hkv, w.D, w.dp, cap)
    L = synth.make_layer(w, cap=cap, n=n0)
    K, V, Wk = L["K"].cuda(), L["V"].cuda(), L["Wk"].cuda()
    Kp = torch.zeros((w.B, w.Hkv, cap, w.dp), dtype=torch.bfloat16, device="cuda")
    tb.tb_project_append(shape, K, cap, Wk, Kp, 0, n0)
    dec = tb.DecodeLayer(shape, w.k, scale=w.scale, n_max=n0)
    d = {k: v.cuda() for k, v in synth.make_step(w, 0, 0, L["outlier_ch"]).items()}
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")

    def step():
        dec.step(0, n0, q=d["q"], q_imp=d["q_imp"], K_new=d["K_new"], V_new=d["V_new"], Wk=Wk, K=K, V=V, Kp=Kp,
                 out=out)
        torch.cuda.synchronize()

    step()
    tb.check_dev_status(dec.status, "reference step")
    ref_out, ref_idx = out.clone(), dec.idx_state.clone()

    rows = w.B * w.Hkv
    _arm(dec.ws, rows, limit_ns=1_000_000, skip_cta=1)
    t0 = time.perf_counter()
    step()
    elapsed = time.perf_counter() - t0
    assert int(dec.status.item()) == tb.TB_ERR_TIMEOUT
    assert elapsed < 1.0, elapsed                     # the 1 ms limit, not the 2 s default, ended the waits

    # the context is usable; the workspace must be zero-filled again after a timeout
    tb.tb_workspace_init(dec.ws)
    dec.status.zero_()
    step()
    tb.check_dev_status(dec.status, "step after recovery")
    # the selection is exact, so the same as before the timeout; the output is the oracle's attention over it
    # within the contract's tolerance (its last bits follow the order in which the warps gathered the rows)
    assert torch.equal(dec.idx_state, ref_idx)
    got = out.float().cpu().numpy()
    ref = oracle.attn(d["q"].cpu(), u16(K), u16(V), dec.sel.cpu().numpy(), dec.counts.cpu().numpy(), w.scale)
    assert np.abs(got - ref).max() <= OUT_ATOL
