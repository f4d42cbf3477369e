"""GPU parity of the importance-query predictor (gist.science summary, Core Architecture, Query Prediction)
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle

tb = pytest.importorskip("predicted_token_importance_tb_b300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tb.load_library()


@pytest.mark.parametrize("B,E,F,O", [(1, 4096, 1024, 1024), (5, 512, 256, 136), (16, 2048, 512, 512),
                                     (2, 4104, 72, 32)])
def test_predictor_matches_oracle(B, E, F, O):
    g = torch.Generator().manual_seed(B * 1000 + E)
    x = torch.randn(B, E, generator=g).to(torch.bfloat16)
    W1 = (torch.randn(F, E, generator=g) * E ** -0.5).to(torch.bfloat16)
    W2 = (torch.randn(O, F, generator=g) * F ** -0.5).to(torch.bfloat16)
    q = torch.empty(B, O, dtype=torch.bfloat16, device="cuda")
    tb.tb_predict_queries(x.cuda(), W1.cuda(), W2.cuda(), q)
    torch.cuda.synchronize()
    got = oracle.bf16_bits_to_f64(oracle.as_u16(q.cpu()))
    _, y, h = oracle.predict_queries(x, W1, W2)
    # fp32 sums on the GPU: layer-1 error <= 2e-5 sum|x w1| (E/256 partials per lane, then 5 shuffle
    # levels), SiLU' <= 1.1 carries it into layer 2, whose own sum adds 2e-5 sum|h w2|; plus the final
    # bf16 rounding (half an ulp, 2^-9 relative)
    xf = oracle.bf16_bits_to_f64(oracle.as_u16(x))
    w1 = np.abs(oracle.bf16_bits_to_f64(oracle.as_u16(W1)))
    w2 = np.abs(oracle.bf16_bits_to_f64(oracle.as_u16(W2)))
    dh = 1.1 * 2e-5 * (np.abs(xf) @ w1.T)
    bound = dh @ w2.T + 2e-5 * (np.abs(h) @ w2.T) + np.abs(y) * 2.0 ** -8 + 1e-30
    assert np.all(np.abs(got - y) <= bound)


def test_predictor_rejects_unsupported_sizes():
    x = torch.zeros(17, 64, dtype=torch.bfloat16, device="cuda")
    W1 = torch.zeros(32, 64, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros(16, 32, dtype=torch.bfloat16, device="cuda")
    q = torch.empty(17, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tb.TBError):
        tb.tb_predict_queries(x, W1, W2, q)      # B > 16
