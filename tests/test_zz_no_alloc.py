"""bq_gemm_noalloc: the prefill GEMM for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run (a plugin hook that must not
allocate, a process whose device memory is fixed after start-up) and have no
workspace to lend. bq_gemm_noalloc serves them from a fixed static device
array instead of a caller workspace. These tests call it through the C ABI
several times in a row (each call reuses the scratch the previous one filled)
and check every output against the CPU oracle within the tolerance of the
other GEMM tests, 1e-5 of sum_b |scale_w scale_x sumi_b| per element, and
against bq_gemm's output on the same inputs. The cases cover both kernels the
entry point can reach inside its 8 MiB array: the tcgen05 kernel (binary16
activation codes fit the array), and the mma.sync kernel over Q8_0 codes,
taken when the binary16 codes would not fit (512 tokens at K = 11008) and for
any K that is not a multiple of 256. The file name makes pytest collect it
last.
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


SCRATCH = 8 << 20


def _cases(orc, shapes, seed):
    from block_quantized_weight_row_gb300 import inputs
    cases = []
    for i, (M, N, K) in enumerate(shapes):
        W = inputs.weight(M, K, seed=seed + i)
        X = inputs.activation(K, seed=seed + 10 + i, rows=N)
        cases.append((orc.quantize_rows(Q8, W.numpy()), X, M, N, K))
    return cases


def _run_in_a_row(env, orc, cases):
    """All cases on one stream, back to back, then each output against the
    oracle and against bq_gemm."""
    bq, L = env
    dev = torch.device("cuda:0")
    outs = []
    for wq, X, M, N, K in cases:
        Y = torch.full((N, M), float("nan"), device=dev)
        rc = _call(L, torch.from_numpy(wq).to(dev), X.to(dev), Y, M, N, K)
        assert rc == 0, L.bq_last_error().decode()
        outs.append(Y)
    torch.cuda.synchronize()
    for (wq, X, M, N, K), Y in zip(cases, outs):
        y = Y.cpu().numpy().astype(np.float64)
        Y_ref, mag = orc.gemm(Q8, wq, X.numpy(), M, N, K, with_mag=True)
        err = np.abs(y - Y_ref)
        assert np.all(err <= TOL * mag), f"{M}x{N}x{K}: worst normwise {float((err / mag).max()):.3g} vs the oracle"
        Y_gemm = bq.gemm(bq.Q8_0, torch.from_numpy(wq).to(dev), X.to(dev), M, N, K).cpu().numpy()
        assert np.all(np.abs(y - Y_gemm) <= TOL * mag), f"{M}x{N}x{K}: differs from bq_gemm"


def test_noalloc_gemm_tensor_core_path_two_calls_in_a_row(env, orc):
    """Binary16 activation codes that fit the array: the tcgen05 kernel."""
    _bq, L = env
    shapes = [(384, 96, 4096), (257, 150, 2304)]
    for M, N, K in shapes:
        assert L.bq_workspace_size(Q8, M, N, K) <= SCRATCH
    _run_in_a_row(env, orc, _cases(orc, shapes, 900))


def test_noalloc_gemm_mma_sync_paths_two_calls_in_a_row(env, orc):
    """512 tokens at K = 11008: bq_gemm would take the tcgen05 kernel with a
    workspace above the array (11.98 MB of binary16 codes), so the entry point
    runs the mma.sync kernel over 5.99 MB of Q8_0 codes in the array; then a
    K that is not a multiple of 256 (the generic mma.sync kernel), then the
    first shape again."""
    _bq, L = env
    shapes = [(64, 512, 11008), (72, 40, 2080), (64, 512, 11008)]
    assert L.bq_workspace_size(Q8, 64, 512, 11008) > SCRATCH
    assert 512 * (11008 // 32) * 34 <= SCRATCH
    _run_in_a_row(env, orc, _cases(orc, shapes, 930))


def test_noalloc_gemm_rejects_sizes_beyond_its_scratch(env):
    _bq, L = env
    dev = torch.device("cuda:0")
    M, N, K = 64, 2048, 4096  # 2048 x 128 x 34 bytes > 8 MiB
    wq = torch.zeros(M * (K // 32) * 34, dtype=torch.uint8, device=dev)
    X = torch.zeros((N, K), device=dev)
    Y = torch.zeros((N, M), device=dev)
    assert _call(L, wq, X, Y, M, N, K) == -7
    assert "static scratch" in L.bq_last_error().decode()
