"""bq_gemm_noalloc: the prefill GEMM for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run (a plugin hook that must not
allocate, a process whose device memory is fixed after start-up) and have no
workspace to lend. bq_gemm_noalloc serves them from a fixed static device
array instead of a caller workspace. This test calls it through the C ABI
twice in a row, with different shapes (the second call reuses the scratch
the first one filled), and checks both outputs against bq_gemm's within the
tolerance of the other GEMM tests: 1e-5 of sum_b |scale_w scale_x sumi_b| per
element. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 1e-5
Q8 = 8


@pytest.fixture(scope="module")
def env():
    import __graft_entry__
    __graft_entry__.build()
    import block_quantized_weight_row_gb300 as bq
    from block_quantized_weight_row_gb300 import binding
    L = binding.lib()
    L.bq_gemm_noalloc.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]
    L.bq_gemm_noalloc.restype = ctypes.c_int
    return bq, L


def _call(L, wq, X, Y, M, N, K):
    s = torch.cuda.current_stream()
    assert L.bq_set_stream(ctypes.c_void_p(s.cuda_stream)) == 0
    return L.bq_gemm_noalloc(Q8, ctypes.c_void_p(wq.data_ptr()), ctypes.c_void_p(X.data_ptr()),
                             ctypes.c_void_p(Y.data_ptr()), M, N, K)


def test_noalloc_gemm_matches_gemm_on_two_calls_in_a_row(env, orc):
    bq, L = env
    from block_quantized_weight_row_gb300 import inputs
    dev = torch.device("cuda:0")
    cases = []
    for i, (M, N, K) in enumerate([(384, 96, 4096), (257, 150, 2304)]):
        W = inputs.weight(M, K, seed=900 + i)
        X = inputs.activation(K, seed=910 + i, rows=N)
        wq = orc.quantize_rows(Q8, W.numpy())
        cases.append((wq, X, M, N, K))
    outs = []
    for wq, X, M, N, K in cases:  # two calls in a row on one stream
        Y = torch.full((N, M), float("nan"), device=dev)
        rc = _call(L, torch.from_numpy(wq).to(dev), X.to(dev), Y, M, N, K)
        assert rc == 0, L.bq_last_error().decode()
        outs.append(Y)
    torch.cuda.synchronize()
    for (wq, X, M, N, K), Y in zip(cases, outs):
        Y_ref = bq.gemm(bq.Q8_0, torch.from_numpy(wq).to(dev), X.to(dev), M, N, K)
        _y, mag = orc.gemm(Q8, wq, X.numpy(), M, N, K, with_mag=True)
        err = np.abs(Y.cpu().numpy().astype(np.float64) - Y_ref.cpu().numpy().astype(np.float64))
        assert np.all(err <= TOL * mag)


def test_noalloc_gemm_rejects_sizes_beyond_its_scratch(env):
    _bq, L = env
    dev = torch.device("cuda:0")
    M, N, K = 64, 2048, 4096  # 2048 x 128 x 34 bytes > 8 MiB
    wq = torch.zeros(M * (K // 32) * 34, dtype=torch.uint8, device=dev)
    X = torch.zeros((N, K), device=dev)
    Y = torch.zeros((N, M), device=dev)
    assert _call(L, wq, X, Y, M, N, K) == -7
    assert "static scratch" in L.bq_last_error().decode()
