"""GPU parity of the projection kernel (df_linear) against the float64 oracle
on the same rounded inputs: ragged row counts (a tail shorter than a 128-row
tile, a single row), one to three outputs, with and without bias, bf16 and
fp16, and the fused-QKV and PK/PQ wrappers."""

import numpy as np
import pytest
import torch

from oracle import linear

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: (2e-2, 1e-2), torch.float16: (4e-3, 2e-3)}  # (atol, rtol) on unit-scale outputs


def _case(M, K, N, n_out, bias, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g).to(dtype)
    ws = [(torch.randn(N, K, generator=g) / K ** 0.5).to(dtype) for _ in range(n_out)]
    bs = [(torch.randn(N, generator=g) * 0.1).to(dtype) for _ in range(n_out)] if bias else None
    return x, ws, bs


def _check(got, want, dtype, what):
    atol, rtol = TOL[dtype]
    g = got.double().cpu().numpy()
    err = np.abs(g - want)
    assert np.isfinite(g).all(), what
    assert (err <= atol + rtol * np.abs(want)).all(), (what, float(err.max()))


@pytest.mark.parametrize("M,K,N,n_out,bias,dtype", [
    (1, 64, 256, 1, False, torch.bfloat16),
    (129, 768, 768, 3, True, torch.bfloat16),
    (1000, 128, 512, 2, True, torch.float16),
    (4725, 768, 768, 3, True, torch.bfloat16),
    (300, 1536, 1536, 1, False, torch.float16),
])
def test_linear_matches_oracle(lib, M, K, N, n_out, bias, dtype):
    x, ws, bs = _case(M, K, N, n_out, bias, dtype, M + K + N)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = lib.df_linear(x.cuda(), [w.cuda() for w in ws], None if bs is None else [b.cuda() for b in bs],
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = linear(x.double().numpy(), [w.double().numpy() for w in ws],
                  None if bs is None else [b.double().numpy() for b in bs])
    for i, (o, w) in enumerate(zip(outs, want)):
        _check(o, w, dtype, f"output {i}")


def test_qkv_and_relative_projections(lib):
    T, hidden, H = 777, 768, 12
    g = torch.Generator().manual_seed(7)
    h = torch.randn(T, hidden, generator=g).to(torch.bfloat16)
    w_qkv = (torch.randn(3 * hidden, hidden, generator=g) / hidden ** 0.5).to(torch.bfloat16)
    b_qkv = (torch.randn(3 * hidden, generator=g) * 0.1).to(torch.bfloat16)
    q, k, v = lib.qkv_projection(h.cuda(), w_qkv.cuda(), b_qkv.cuda(), H)
    assert q.shape == (T, H, hidden // H)
    want = linear(h.double().numpy(), [w_qkv[i * hidden:(i + 1) * hidden].double().numpy() for i in range(3)],
                  [b_qkv[i * hidden:(i + 1) * hidden].double().numpy() for i in range(3)])
    for got, w in zip((q, k, v), want):
        _check(got.reshape(T, hidden), w, torch.bfloat16, "qkv")
    rel = torch.randn(512, hidden, generator=g).to(torch.bfloat16)
    wk, wq = ((torch.randn(hidden, hidden, generator=g) / hidden ** 0.5).to(torch.bfloat16) for _ in range(2))
    pk, pq = lib.rel_projection(rel.cuda(), wk.cuda(), None, wq.cuda(), None, H)
    want = linear(rel.double().numpy(), [wk.double().numpy(), wq.double().numpy()])
    _check(pk.reshape(512, hidden), want[0], torch.bfloat16, "pk")
    _check(pq.reshape(512, hidden), want[1], torch.bfloat16, "pq")
