"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Bars: quantized bytes and integer block dots bit-exact; float outputs within
1e-5 of sum_b |scale_w scale_x sumi_b| per element (normwise: a plain relative
bound is ill-posed where the sum cancels to ~0). Every input is seeded and
synthetic (block_quantized_weight_row_gb300.inputs); the oracle never sees a
value produced by the CUDA path.
"""
import math

import numpy as np
import pytest
import torch

from block_quantized_weight_row_gb300.inputs import LLAMA_7B_LAYER, QWEN3_0_6B_LAYER

pytestmark = pytest.mark.gpu

Q4, Q8 = 2, 8
TOL = 1e-5


@pytest.fixture(scope="module")
def bq():
    import __graft_entry__
    __graft_entry__.build()
    import block_quantized_weight_row_gb300 as m
    return m


@pytest.fixture(scope="module")
def dev():
    return torch.device("cuda:0")


def _np(t):
    return t.detach().cpu().numpy()


def _check_float(y, y_ref, mag, what=""):
    y = np.asarray(y, np.float64).reshape(-1)
    y_ref = np.asarray(y_ref, np.float64).reshape(-1)
    mag = np.asarray(mag, np.float64).reshape(-1)
    err = np.abs(y - y_ref)
    bad = err > TOL * mag
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs off; worst normwise "
                           f"{float((err / np.maximum(mag, 1e-300)).max()):.3g}")
    big = np.abs(y_ref) > 1e-3 * mag
    if big.any():  # element-wise relative error where it is meaningful
        assert float((err[big] / np.abs(y_ref[big])).max()) < 1e-3, what


# ------------------------------------------------------------ quantize ----

@pytest.mark.parametrize("t", [Q4, Q8])
@pytest.mark.parametrize("shape,std", [((1, 32), 1.0), ((3, 96), 0.02), ((257, 64), 1.0),
                                       ((64, 4096), 0.02), ((7, 11008), 1.0), ((1000, 1024), 0.02),
                                       ((1, 8192 + 32), 3.0)])
def test_quantize_rows_bit_exact(bq, orc, dev, t, shape, std):
    from block_quantized_weight_row_gb300 import inputs
    x = inputs.normal(shape, std, seed=shape[0] * 7 + shape[1])
    got = _np(bq.quantize_rows(t, x.to(dev)))
    ref = orc.quantize_rows(t, x.numpy())
    assert got.shape == ref.shape
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


@pytest.mark.parametrize("t", [Q4, Q8])
def test_quantize_adversarial_blocks(bq, orc, dev, t):
    from block_quantized_weight_row_gb300 import inputs
    x = inputs.adversarial_blocks()
    x = torch.cat([x, -x, x * 1e-4, x * 3e3]).contiguous()
    got = _np(bq.quantize_rows(t, x.to(dev)))
    assert np.array_equal(got, orc.quantize_rows(t, x.numpy()))


@pytest.mark.parametrize("t", [Q4, Q8])
def test_quantize_near_ties_bit_exact(bq, orc, dev, t):
    """Values placed on and within a few ulp of k + 0.5 times the block scale,
    under many scales: the kernel's fast rounding must hand every such value
    to its exact path and agree with the oracle's IEEE division bit for bit."""
    rng = np.random.default_rng(42)
    qmax = 7 if t == Q4 else 127
    rows = []
    for _ in range(3000):
        amax = np.float32(10.0 ** rng.uniform(-4, 3))
        d16 = np.float32(np.float16(amax / np.float32(qmax)))
        k = rng.integers(-qmax, qmax, 31).astype(np.float32)
        x = (k + np.float32(0.5)) * d16
        bump = rng.integers(-3, 4, 31)  # move by -3..3 ulp
        for i in range(31):
            for _s in range(abs(int(bump[i]))):
                x[i] = np.nextafter(x[i], np.float32(np.inf) if bump[i] > 0 else np.float32(-np.inf))
        rows.append(np.concatenate([[amax], x]).astype(np.float32))
    X = np.stack(rows)
    got = _np(bq.quantize_rows(t, torch.from_numpy(X).to(dev)))
    ref = orc.quantize_rows(t, X)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


@pytest.mark.parametrize("t", [Q4, Q8])
def test_dequantize_bit_exact(bq, orc, dev, t):
    from block_quantized_weight_row_gb300 import inputs
    x = inputs.normal((37, 160), 0.5, seed=11)
    q = orc.quantize_rows(t, x.numpy())
    got = _np(bq.dequantize_rows(t, torch.from_numpy(q).to(dev), 160))
    ref = orc.dequantize_rows(t, q, 160)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------- block dots -----

@pytest.mark.parametrize("t", [Q4, Q8])
@pytest.mark.parametrize("M,K", [(1, 32), (5, 96), (64, 4096), (3, 11008)])
def test_block_dots_bit_exact(bq, orc, dev, t, M, K):
    from block_quantized_weight_row_gb300 import inputs
    W = inputs.weight(M, K, seed=M + K)
    x = inputs.activation(K, seed=M + K + 1)
    wq = orc.quantize_rows(t, W.numpy())
    xq = orc.quantize_rows(Q8, x.numpy())
    got = _np(bq.block_dots(t, torch.from_numpy(wq).to(dev), torch.from_numpy(xq).to(dev), M, K))
    assert np.array_equal(got, orc.block_dots(t, wq, xq, M, K))


# ---------------------------------------------------------------- GEMV ----

def _gemv_case(bq, orc, dev, t, M, K, seed, std=0.02):
    from block_quantized_weight_row_gb300 import inputs
    W = inputs.normal((M, K), std, seed)
    x = inputs.activation(K, seed + 1)
    wq = orc.quantize_rows(t, W.numpy())
    y = _np(bq.gemv(t, torch.from_numpy(wq).to(dev), x.to(dev), M, K))
    y_ref, mag = orc.gemv(t, wq, x.numpy(), M, K, with_mag=True)
    _check_float(y, y_ref, mag, f"gemv t={t} M={M} K={K}")


@pytest.mark.parametrize("t", [Q4, Q8])
@pytest.mark.parametrize("M,K", [(1, 32), (3, 64), (17, 96), (64, 160), (333, 288),     # ragged K
                                 (1, 256), (3, 512), (17, 768), (64, 1280), (100, 2304),  # 1..9 groups
                                 (1, 4096), (3, 4096), (129, 4096), (257, 11008), (5, 16384)])
def test_gemv_shapes(bq, orc, dev, t, M, K):
    _gemv_case(bq, orc, dev, t, M, K, seed=M * 131 + K)


@pytest.mark.parametrize("t", [Q4, Q8])
def test_gemv_tiny_config(bq, orc, dev, t):
    """1024 x 1024 ~ N(0, 0.02), x ~ N(0, 1), seed 0, both weight types."""
    from block_quantized_weight_row_gb300 import inputs
    W, x = inputs.tiny()
    wq_dev = bq.quantize_rows(t, W.to(dev))
    wq = orc.quantize_rows(t, W.numpy())
    assert np.array_equal(_np(wq_dev), wq)
    y = _np(bq.gemv(t, wq_dev, x.to(dev), 1024, 1024))
    y_ref, mag = orc.gemv(t, wq, x.numpy(), 1024, 1024, with_mag=True)
    _check_float(y, y_ref, mag, "tiny")


@pytest.mark.parametrize("M,K", sorted({(m, k) for _n, m, k in QWEN3_0_6B_LAYER + LLAMA_7B_LAYER}))
def test_gemv_model_shapes_full(bq, orc, dev, M, K):
    """Every distinct matrix shape of the 0.6B and 7B decode steps, whole
    matrix, Q4_0; also checks the GPU row quantizer on the full matrix."""
    from block_quantized_weight_row_gb300 import inputs
    W = inputs.weight(M, K, seed=M + 3 * K)
    x = inputs.activation(K, seed=M + 3 * K + 1)
    wq_dev = bq.quantize_rows(Q4, W.to(dev))
    wq = orc.quantize_rows(Q4, W.numpy())
    assert np.array_equal(_np(wq_dev), wq)
    y = _np(bq.gemv(Q4, wq_dev, x.to(dev), M, K))
    y_ref, mag = orc.gemv(Q4, wq, x.numpy(), M, K, with_mag=True)
    _check_float(y, y_ref, mag, f"model shape {M}x{K}")


def test_gemv_on_side_stream(bq, orc, dev):
    """Quantize then GEMV enqueued on a non-default stream, no sync in between."""
    from block_quantized_weight_row_gb300 import inputs
    W = inputs.weight(512, 4096, seed=5)
    x = inputs.activation(4096, seed=6)
    s = torch.cuda.Stream(dev)
    Wd, xd = W.to(dev), x.to(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        wq = bq.quantize_rows(Q4, Wd)
        y = bq.gemv(Q4, wq, xd, 512, 4096)
    s.synchronize()
    wq_ref = orc.quantize_rows(Q4, W.numpy())
    y_ref, mag = orc.gemv(Q4, wq_ref, x.numpy(), 512, 4096, with_mag=True)
    _check_float(_np(y), y_ref, mag, "side stream")


def test_gemv_k_zero_gives_zeros(bq, dev):
    y = torch.full((7,), 5.0, device=dev)
    bq.gemv(Q4, torch.empty(16, dtype=torch.uint8, device=dev), torch.empty(4, device=dev), 0, 0)
    bq.gemv(Q4, torch.empty(16, dtype=torch.uint8, device=dev), torch.empty(4, device=dev), 7, 0, out=y)
    assert torch.all(y == 0)


def test_gemv_timeout_path_returns_error(bq, orc, dev):
    """With a poll budget of 0 every bounded wait gives up at once: the kernel
    drains its own copies, returns, and the status reports the timeout; the
    next call with the default budget is correct again."""
    from block_quantized_weight_row_gb300 import binding, inputs
    L = binding.lib()
    W = inputs.weight(256, 4096, seed=9)
    x = inputs.activation(4096, seed=10)
    wq = bq.quantize_rows(Q4, W.to(dev))
    assert binding.device_status() == 0
    try:
        assert L.bq_set_spin_limit(0) == 0
        bq.gemv(Q4, wq, x.to(dev), 256, 4096)
        assert binding.device_status() == -6
    finally:
        L.bq_set_spin_limit(-1)
    y = bq.gemv(Q4, wq, x.to(dev), 256, 4096)
    assert binding.device_status() == 0
    y_ref, mag = orc.gemv(Q4, orc.quantize_rows(Q4, W.numpy()), x.numpy(), 256, 4096, with_mag=True)
    _check_float(_np(y), y_ref, mag, "after timeout")


# ---------------------------------------------------------------- GEMM ----

# K a multiple of 256 runs the tcgen05 kernel (128 x 128 tiles, partial sums
# folded every 16 blocks), other K the mma.sync kernel. The shapes cover M and
# N tails inside and beyond one tile, a single token, block counts that end
# on and between fold boundaries (8, 24, 40, 72, 256, 344 blocks) and K not a
# multiple of 256.
@pytest.mark.parametrize("M,N,K", [(64, 16, 256), (130, 70, 512), (33, 5, 96), (256, 128, 4096),
                                   (200, 65, 2304), (1, 1, 32), (128, 64, 11008), (129, 1, 256),
                                   (300, 129, 768), (1000, 300, 1280), (384, 256, 8192), (257, 131, 4352),
                                   (64, 16, 4128)])
def test_gemm_shapes(bq, orc, dev, M, N, K):
    from block_quantized_weight_row_gb300 import inputs
    W = inputs.weight(M, K, seed=M * 7 + K)
    X = inputs.activation(K, seed=N * 3 + K, rows=N)
    wq = orc.quantize_rows(Q8, W.numpy())
    Y = _np(bq.gemm(Q8, torch.from_numpy(wq).to(dev), X.to(dev), M, N, K))
    Y_ref, mag = orc.gemm(Q8, wq, X.numpy(), M, N, K, with_mag=True)
    _check_float(Y, Y_ref, mag, f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,K", [(4096, 4096), (11008, 4096), (4096, 11008)])
def test_gemm_prefill_config_sampled(bq, orc, dev, M, K):
    """512 tokens at full size; 48 sampled tokens x 96 sampled weight rows
    are recomputed by the oracle (each output depends on one row of each)."""
    from block_quantized_weight_row_gb300 import inputs
    N = 512
    W = inputs.weight(M, K, seed=inputs.seed_of("prefill-q8_0", 0, M // 1000 + K // 1000), device=dev)
    X = inputs.activation(K, seed=inputs.seed_of("prefill-q8_0", 1, K // 1000), device=dev, rows=N)
    wq = bq.quantize_rows(Q8, W)
    Y = _np(bq.gemm(Q8, wq, X, M, N, K))
    rng = np.random.default_rng(M + K)
    ns = np.sort(rng.choice(N, 48, replace=False))
    ms = np.sort(rng.choice(M, 96, replace=False))
    W_s = _np(W[torch.from_numpy(ms).to(dev)])
    X_s = _np(X[torch.from_numpy(ns).to(dev)])
    wq_s = orc.quantize_rows(Q8, W_s)
    assert np.array_equal(_np(wq[torch.from_numpy(ms).to(dev)]), wq_s)
    Y_ref, mag = orc.gemm(Q8, wq_s, X_s, len(ms), len(ns), K, with_mag=True)
    _check_float(Y[np.ix_(ns, ms)], Y_ref, mag, f"prefill {M}x{K}")


def test_gemm_full_code_range(bq, orc, dev):
    """Weight blocks the quantizer never writes but the format allows: every
    int8 code including -128 and arbitrary binary16 scales; activations with
    the adversarial blocks (zeros, spikes, ties, tiny and huge scales)."""
    from block_quantized_weight_row_gb300 import inputs
    M, N, K = 260, 136, 512
    rng = np.random.default_rng(77)
    nb = K // 32
    blocks = np.empty((M, nb, 34), np.uint8)
    scales = rng.uniform(1e-4, 1e-1, size=(M, nb)).astype(np.float16)
    blocks[:, :, 0:2] = scales.view(np.uint8).reshape(M, nb, 2)
    blocks[:, :, 2:] = rng.integers(0, 256, size=(M, nb, 32), dtype=np.uint8)
    blocks[0, 0, 2:] = 0x80  # a block of -128 codes
    wq = blocks.reshape(-1)
    adv = inputs.adversarial_blocks().numpy()
    X = np.resize(adv, (N * nb, 32)).reshape(N, K).astype(np.float32)
    X[N // 2:] = inputs.activation(K, seed=5, rows=N - N // 2).numpy()
    Y = _np(bq.gemm(Q8, torch.from_numpy(wq).to(dev), torch.from_numpy(X).to(dev), M, N, K))
    Y_ref, mag = orc.gemm(Q8, wq, X, M, N, K, with_mag=True)
    _check_float(Y, Y_ref, mag, "gemm full code range")


def test_gemm_timeout_path_returns_error(bq, orc, dev):
    """The tcgen05 GEMM with a poll budget of 0: every role gives up at its
    first wait, the MMAs and copies already issued are waited for, the tensor
    memory is freed, and the status reports the timeout; the next call with
    the default budget is correct (it could not allocate tensor memory if the
    failed one had kept it)."""
    from block_quantized_weight_row_gb300 import binding, inputs
    L = binding.lib()
    M, N, K = 256, 130, 1024
    W = inputs.weight(M, K, seed=19)
    X = inputs.activation(K, seed=20, rows=N)
    wq = torch.from_numpy(orc.quantize_rows(Q8, W.numpy())).to(dev)
    assert binding.device_status() == 0
    try:
        assert L.bq_set_spin_limit(0) == 0
        bq.gemm(Q8, wq, X.to(dev), M, N, K)
        assert binding.device_status() == -6
    finally:
        L.bq_set_spin_limit(-1)
    Y = _np(bq.gemm(Q8, wq, X.to(dev), M, N, K))
    assert binding.device_status() == 0
    Y_ref, mag = orc.gemm(Q8, _np(wq), X.numpy(), M, N, K, with_mag=True)
    _check_float(Y, Y_ref, mag, "gemm after timeout")


def test_gemm_errors(bq, dev):
    from block_quantized_weight_row_gb300 import binding
    wq = torch.zeros(64 * 34, dtype=torch.uint8, device=dev)
    with pytest.raises(binding.BQError) as e:
        bq.gemm(Q4, wq, torch.zeros(2, 64, device=dev), 2, 2, 64)
    assert e.value.status == -3


# ----------------------------------------------------------- KV write -----

@pytest.mark.parametrize("tokens", [1, 37, 1024])
def test_kv_write_bit_exact(bq, orc, dev, tokens):
    from block_quantized_weight_row_gb300 import inputs
    L = inputs.kv_layer(2, tokens=tokens, kv_heads=8, head_dim=128, calib_tokens=64)
    bias = L.K_calib.double().mean(dim=0).float()
    kq = _np(bq.kv_quantize(Q4, L.K.to(dev), bias.to(dev)))
    assert np.array_equal(kq, orc.kv_quantize(Q4, L.K.numpy(), bias.numpy(), tokens, 8, 128))
    vq = _np(bq.kv_quantize(Q8, L.V.to(dev), None))
    assert np.array_equal(vq, orc.kv_quantize(Q8, L.V.numpy(), None, tokens, 8, 128))
    k_plain = _np(bq.kv_quantize(Q4, L.K.to(dev), None))
    assert np.array_equal(k_plain, orc.kv_quantize(Q4, L.K.numpy(), None, tokens, 8, 128))


def test_kv_write_full_layer(bq, orc, dev):
    """One layer of the KV-write workload at full size: 32768 tokens x 8 kv
    heads x 128, K with the calibrated bias to Q4_0 and V to Q8_0."""
    from block_quantized_weight_row_gb300 import inputs
    cfg = inputs.WORKLOADS["kv-write"]
    L = inputs.kv_layer(0, cfg["tokens"], cfg["kv_heads"], cfg["head_dim"], cfg["calib_tokens"], device=dev)
    bias = L.K_calib.double().mean(dim=0).float()
    kq = _np(bq.kv_quantize(Q4, L.K, bias))
    vq = _np(bq.kv_quantize(Q8, L.V, None))
    T, H, D = L.K.shape
    assert np.array_equal(kq, orc.kv_quantize(Q4, _np(L.K), _np(bias), T, H, D))
    assert np.array_equal(vq, orc.kv_quantize(Q8, _np(L.V), None, T, H, D))


@pytest.mark.parametrize("T,NKV,D,kt,vt,basis,with_bias", [
    (1, 1, 32, Q4, Q8, 0, True), (37, 8, 128, Q4, Q8, 0, True), (1000, 8, 128, Q4, Q8, 1, True),
    (33, 3, 64, Q4, Q4, 1, False), (130, 3, 96, Q8, Q8, 0, False), (7, 2, 256, Q8, Q4, 1, False),
    (4099, 5, 64, Q4, Q8, 0, True),
    # a bias of 160 blocks: read from global memory, in both bases
    (9, 5, 1024, Q4, Q8, 0, True), (9, 5, 1024, Q4, Q8, 1, True)])
def test_kv_write_layer_matches_oracle(bq, orc, dev, T, NKV, D, kt, vt, basis, with_bias):
    """bq_kv_write (K and V of a layer in one call, V's launch not waiting for
    K's): K and V bytes equal to the oracle's and to one bq_kv_quantize call
    per tensor, for block counts
    that leave a ragged last tile (1 block; 21 x 3 x 2; 4099 x 5 x 2), both
    bases, with and without the bias, every type pair."""
    rng = np.random.default_rng(T + 3 * NKV + D + basis)
    K = _outlier_rows(rng, T, NKV, D)
    V = rng.normal(size=(T, NKV, D)).astype(np.float32)
    bias = orc.kv_bias(_outlier_rows(rng, 64, NKV, D), basis, 64, NKV, D) if with_bias else None
    Kd, Vd = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    bd = torch.from_numpy(bias).to(dev) if with_bias else None
    kq, vq = bq.kv_write(kt, Kd, bd, vt, Vd, basis=basis)
    assert np.array_equal(_np(kq), orc.kv_quantize(kt, K, bias, T, NKV, D, basis=basis))
    assert np.array_equal(_np(vq), orc.kv_quantize(vt, V, None, T, NKV, D))
    assert torch.equal(kq, bq.kv_quantize(kt, Kd, bd, basis=basis))
    assert torch.equal(vq, bq.kv_quantize(vt, Vd, None))


def test_kv_write_layer_full_size(bq, orc, dev):
    """One full layer of the KV-write workload through bq_kv_write (K
    mean-centered to Q4_0, V to Q8_0): the oracle's bytes in either basis.
    Calls follow each other on the stream without a sync, the second writing
    the same outputs (its V launch must not overtake the first call's): the
    later call's bytes remain."""
    from block_quantized_weight_row_gb300 import inputs
    cfg = inputs.WORKLOADS["kv-write"]
    L = inputs.kv_layer(1, cfg["tokens"], cfg["kv_heads"], cfg["head_dim"], cfg["calib_tokens"], device=dev)
    T, H, D = L.K.shape
    Kn, Vn = _np(L.K), _np(L.V)
    v_ref = orc.kv_quantize(Q8, Vn, None, T, H, D)
    biases = [bq.kv_bias(L.K_calib, basis) for basis in (0, 1)]
    zeros_v = torch.zeros_like(L.V)
    kq = torch.empty((T, H, D // 32 * 18), dtype=torch.uint8, device=dev)
    vq = torch.empty((T, H, D // 32 * 34), dtype=torch.uint8, device=dev)
    for last in (0, 1):
        first = 1 - last
        bq.kv_write(Q4, L.K, biases[first], Q8, zeros_v, out_k=kq, out_v=vq, basis=first)
        bq.kv_write(Q4, L.K, biases[last], Q8, L.V, out_k=kq, out_v=vq, basis=last)
        assert np.array_equal(_np(kq), orc.kv_quantize(Q4, Kn, _np(biases[last]), T, H, D, basis=last))
        assert np.array_equal(_np(vq), v_ref)


def test_kv_write_layer_rejects_before_writing(bq, dev):
    """A bias with a Q8_0 K, a bias from another basis, an unknown V type or
    outputs that overlap: an error status and nothing written."""
    from block_quantized_weight_row_gb300 import binding
    K = torch.ones(4, 2, 64, device=dev)
    V = torch.ones(4, 2, 64, device=dev)
    ok_k = torch.full((4, 2, 36), 7, dtype=torch.uint8, device=dev)
    ok_v = torch.full((4, 2, 68), 7, dtype=torch.uint8, device=dev)
    shared = torch.full((1024,), 7, dtype=torch.uint8, device=dev)  # two outputs that overlap
    q8_k = torch.full((4, 2, 68), 7, dtype=torch.uint8, device=dev)
    cases = [
        (dict(k_type=Q8, bias=torch.zeros(2, 64, device=dev), v_type=Q8, out_k=q8_k), -3),
        (dict(k_type=Q4, bias=torch.zeros(2, 64, device=dev), v_type=Q8, basis=1, bias_basis=0), -8),
        (dict(k_type=Q4, bias=None, v_type=bq.Q4_1), -3),
        (dict(k_type=Q4, bias=None, v_type=Q8, out_k=shared[:288].view(4, 2, 36),
              out_v=shared[256:256 + 544].view(4, 2, 68)), -1),
    ]
    for kw, status in cases:
        kt, b, vt = kw.pop("k_type"), kw.pop("bias"), kw.pop("v_type")
        kw.setdefault("out_k", ok_k)
        kw.setdefault("out_v", ok_v)
        with pytest.raises(binding.BQError) as e:
            bq.kv_write(kt, K, b, vt, V, **kw)
        assert e.value.status == status
    torch.cuda.synchronize()
    for t in (ok_k, ok_v, shared, q8_k):
        assert bool((t == 7).all())  # nothing was written


def test_kv_mean_centering_keeps_softmax_and_helps(bq, dev):
    """GPU-written cache: adding the bias back after dequantization recovers K
    within half a scale step, and centering lowers the attention KL against
    the fp32 cache (softmax(z + c) = softmax(z) makes the bias free)."""
    from block_quantized_weight_row_gb300 import inputs
    T, H, D = 2048, 8, 128
    L = inputs.kv_layer(3, tokens=T, kv_heads=H, head_dim=D, calib_tokens=512, device=dev)
    bias = L.K_calib.double().mean(dim=0).float()
    kc = bq.kv_quantize(Q4, L.K, bias)
    kp = bq.kv_quantize(Q4, L.K, None)
    Kc = bq.dequantize_rows(Q4, kc, D).view(T, H, D) + bias
    Kp = bq.dequantize_rows(Q4, kp, D).view(T, H, D)
    d = kc.view(T * H * D // 32, 18)[:, :2].contiguous().view(torch.float16).float().view(T, H, D // 32, 1)
    err = (Kc - L.K).view(T, H, D // 32, 32).abs()
    assert bool(torch.all(err <= d / 2 * (1 + 2.0 ** -18) + 1e-6))
    q = inputs.normal((64, H, D), 1.0, 97, device=dev).double()
    ref = torch.softmax(torch.einsum("qhd,thd->hqt", q, L.K.double()) / math.sqrt(D), dim=-1)
    kl = {}
    for name, Kq in (("centered", Kc), ("plain", Kp)):
        p = torch.softmax(torch.einsum("qhd,thd->hqt", q, Kq.double()) / math.sqrt(D), dim=-1)
        kl[name] = float((ref * (ref.log() - p.log())).sum(-1).mean())
    assert kl["centered"] < kl["plain"]


def test_kv_bias_with_q8_0_rejected(bq, dev):
    from block_quantized_weight_row_gb300 import binding
    with pytest.raises(binding.BQError) as e:
        bq.kv_quantize(Q8, torch.zeros(2, 2, 64, device=dev), torch.zeros(2, 64, device=dev))
    assert e.value.status == -3


# ------------------------------------------- weight prefetch across kernels --

def test_gemv_prefetch_chain_respects_war_and_raw(bq, orc, dev):
    """With weight prefetch on, a GEMV starts streaming W before the previous
    GEMV has finished. Chain: g1 reads A and writes B; g2 reads C and writes A
    (g2 must not overwrite A before g1 read it); g3 reads B (g1's output) and
    writes D (it must see g1's finished y). g1 and g2 are checked against the
    oracle on the generator's inputs; g3 against the same chain without
    prefetch."""
    from block_quantized_weight_row_gb300 import binding, inputs
    K = 4096
    Ws = [inputs.weight(K, K, seed=1300 + i) for i in range(3)]
    wq = [orc.quantize_rows(Q4, W.numpy()) for W in Ws]
    wq_d = [torch.from_numpy(w).to(dev) for w in wq]
    A0 = inputs.activation(K, seed=1310)
    C0 = inputs.activation(K, seed=1311)

    def chain(prefetch):
        A, C = A0.to(dev), C0.to(dev)
        B, D = torch.empty(K, device=dev), torch.empty(K, device=dev)
        torch.cuda.synchronize()
        binding.set_weight_prefetch(prefetch)
        try:
            for _ in range(3):  # repeat so the three launches overlap in steady state
                A.copy_(A0.to(dev, non_blocking=True))
                bq.gemv(Q4, wq_d[0], A, K, K, out=B)
                bq.gemv(Q4, wq_d[1], C, K, K, out=A)
                bq.gemv(Q4, wq_d[2], B, K, K, out=D)
        finally:
            binding.set_weight_prefetch(False)
        torch.cuda.synchronize()
        return _np(B), _np(A), _np(D)

    B1, A1, D1 = chain(True)
    y_ref, mag = orc.gemv(Q4, wq[0], A0.numpy(), K, K, with_mag=True)
    _check_float(B1, y_ref, mag, "g1 (reads A before g2 overwrites it)")
    y_ref, mag = orc.gemv(Q4, wq[1], C0.numpy(), K, K, with_mag=True)
    _check_float(A1, y_ref, mag, "g2")
    _B0, _A0, D0 = chain(False)
    assert np.array_equal(D1, D0), "g3 differs when it may start before g1 finished"


# ------------------------------------------------------ batched GEMV ---------

@pytest.mark.parametrize("t", [Q4, Q8])
@pytest.mark.parametrize("Ms,K", [([4096, 1024, 1024], 4096), ([11008, 11008], 4096), ([5, 0, 17, 1, 3, 64, 2, 9], 4096),
                                  ([33, 7], 96), ([1], 256), ([300, 200, 100], 2304)])
def test_gemv_multi_matches_oracle(bq, orc, dev, t, Ms, K):
    from block_quantized_weight_row_gb300 import inputs
    x = inputs.activation(K, seed=K + 77)
    wq = [orc.quantize_rows(t, inputs.weight(m, K, seed=1000 + 17 * i + m).numpy()) if m else
          np.zeros((0, K // 32 * (18 if t == Q4 else 34)), np.uint8) for i, m in enumerate(Ms)]
    w_dev = [torch.from_numpy(w).to(dev) if w.size else torch.empty(16, dtype=torch.uint8, device=dev) for w in wq]
    outs = bq.gemv_multi(t, w_dev, x.to(dev), Ms, K)
    for i, (m, w) in enumerate(zip(Ms, wq)):
        if m == 0:
            continue
        y_ref, mag = orc.gemv(t, w, x.numpy(), m, K, with_mag=True)
        _check_float(_np(outs[i]), y_ref, mag, f"matrix {i} of the batch")


def test_gemv_multi_rejects_bad_batches(bq, dev):
    from block_quantized_weight_row_gb300 import binding
    w = torch.zeros(64 * 18, dtype=torch.uint8, device=dev)
    x = torch.zeros(64, device=dev)
    with pytest.raises(binding.BQError) as e:
        bq.gemv_multi(Q4, [w] * 9, x, [1] * 9, 64)
    assert e.value.status == -2
    y = torch.zeros(8, device=dev)
    with pytest.raises(binding.BQError) as e:  # two outputs on the same buffer
        bq.gemv_multi(Q4, [w, w], x, [4, 4], 64, outs=[y, y])
    assert e.value.status == -1


@pytest.mark.parametrize("t", [Q4, Q8])
@pytest.mark.parametrize("with_ws", [True, False])
@pytest.mark.parametrize("Ms,K", [([4096, 1024], 4096), ([3, 700], 11008), ([257], 2304),
                                  ([33, 500], 4128), ([5], 96)])  # K % 256 != 0: the generic kernel
def test_gemv_both_activation_paths(bq, orc, dev, t, with_ws, Ms, K):
    """x quantized once by the prep kernel into the workspace, or by every
    GEMV CTA: both must match the oracle (and hence each other)."""
    import ctypes
    from block_quantized_weight_row_gb300 import binding, inputs
    L = binding.lib()
    x = inputs.activation(K, seed=K + 5)
    wq = [orc.quantize_rows(t, inputs.weight(m, K, seed=2000 + 3 * i + m).numpy()) for i, m in enumerate(Ms)]
    w_dev = [torch.from_numpy(w).to(dev) for w in wq]
    outs = [torch.full((m,), float("nan"), device=dev) for m in Ms]
    xd = x.to(dev)
    ws = torch.empty(max(256, int(L.bq_gemv_workspace_size(t, K))), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    assert L.bq_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    if with_ws:
        assert L.bq_set_workspace(ctypes.c_void_p(ws.data_ptr()), ws.numel()) == 0
    else:
        assert L.bq_set_workspace(None, 0) == 0
    n, W, Y, M = binding.gemv_multi_args(w_dev, outs, Ms)
    assert L.bq_gemv_multi(t, n, W, Y, M, ctypes.c_void_p(xd.data_ptr()), K) == 0, L.bq_last_error()
    torch.cuda.synchronize()
    L.bq_set_workspace(None, 0)
    for i, (m, w) in enumerate(zip(Ms, wq)):
        y_ref, mag = orc.gemv(t, w, x.numpy(), m, K, with_mag=True)
        _check_float(_np(outs[i]), y_ref, mag, f"matrix {i}, workspace={with_ws}")


@pytest.mark.parametrize("t", [Q4, Q8, 3, 6, 7])
# K = 16416: Q8_0 rows of 17.4 KB leave no room for two row buffers per
# warp, so Q8_0 takes the generic kernel there (the other types still stage)
@pytest.mark.parametrize("Ms,K", [([33, 500], 4128), ([5], 96), ([4096], 4128), ([3, 1], 32), ([7, 40], 16416)])
def test_gemv_unaligned_rows_both_paths_bit_identical(bq, orc, dev, t, Ms, K):
    """Rows that are not multiples of 16 bytes (K % 256 != 0): with a
    workspace, x's records come from the 8-lane prep launch and the rows are
    staged in shared memory (or, for rows too long to stage, read by the
    generic kernel); without, every CTA quantizes x one block per thread and
    reads the rows from global memory. The same records and the same order
    of terms: identical bits, and the oracle's products within tolerance."""
    import ctypes
    from block_quantized_weight_row_gb300 import binding, inputs
    L = binding.lib()
    x = inputs.activation(K, seed=K + 11).to(dev)
    w_dev = [bq.quantize_rows(t, inputs.weight(m, K, seed=3000 + 7 * i + m, device=dev)) for i, m in enumerate(Ms)]
    ws = torch.empty(max(256, int(L.bq_gemv_workspace_size(t, K))), dtype=torch.uint8, device=dev)
    res = []
    for with_ws in (True, False):
        outs = [torch.full((m,), float("nan"), device=dev) for m in Ms]
        torch.cuda.synchronize()
        assert L.bq_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        assert L.bq_set_workspace(ctypes.c_void_p(ws.data_ptr()) if with_ws else None, ws.numel() if with_ws else 0) == 0
        n, W, Y, M = binding.gemv_multi_args(w_dev, outs, Ms)
        assert L.bq_gemv_multi(t, n, W, Y, M, ctypes.c_void_p(x.data_ptr()), K) == 0, L.bq_last_error()
        torch.cuda.synchronize()
        res.append(outs)
    L.bq_set_workspace(None, 0)
    for a, b in zip(*res):
        assert torch.equal(a, b)
    y_ref, mag = orc.gemv(t, _np(w_dev[0]), _np(x), Ms[0], K, with_mag=True)
    _check_float(_np(res[0][0]), y_ref, mag, "with the workspace")


def test_gemv_with_weight_prefetch_right_after_quantizing_its_weights(bq, orc, dev):
    """With weight prefetch on, a GEMV may stream its weights before the
    previous launch has completed; a row quantization of those weights just
    before it must still have finished first (it lets no dependent start
    early). Four rounds quantize new weights into the same buffer and run the
    GEMV at once, without a sync: each output matches the oracle for its
    round's weights."""
    from block_quantized_weight_row_gb300 import binding, inputs
    M, K = 4096, 4096
    x = inputs.activation(K, seed=91, device=dev)
    wq = torch.empty((M, K // 32 * 18), dtype=torch.uint8, device=dev)
    ws = [inputs.weight(M, K, seed=900 + i, device=dev) for i in range(4)]
    ys = [torch.full((M,), float("nan"), device=dev) for _ in ws]
    torch.cuda.synchronize()
    binding.set_weight_prefetch(True)
    try:
        for W, y in zip(ws, ys):
            bq.quantize_rows(Q4, W, out=wq)
            bq.gemv(Q4, wq, x, M, K, out=y)
        torch.cuda.synchronize()
    finally:
        binding.set_weight_prefetch(False)
    xn = _np(x)
    for i, (W, y) in enumerate(zip(ws, ys)):
        w_ref = orc.quantize_rows(Q4, _np(W))
        y_ref, mag = orc.gemv(Q4, w_ref, xn, M, K, with_mag=True)
        _check_float(_np(y), y_ref, mag, f"round {i}")


def test_gemv_large_launch_three_stage_ring(bq, orc, dev):
    """A launch of more than 64 MB of weights (three 11008 x 4096 Q4_0
    matrices, 76 MB) runs with a three-stage ring: it matches the oracle and
    is bit-identical to the same matrices launched one per call (two-stage
    ring; each row is computed the same way whatever the stage size)."""
    from block_quantized_weight_row_gb300 import inputs
    M, K = 11008, 4096
    x = inputs.activation(K, seed=77)
    wq = [orc.quantize_rows(Q4, inputs.weight(M, K, seed=7700 + i).numpy()) for i in range(3)]
    w_dev = [torch.from_numpy(w).to(dev) for w in wq]
    xd = x.to(dev)
    ys = bq.gemv_multi(Q4, w_dev, xd, [M] * 3, K)
    singles = [bq.gemv(Q4, w, xd, M, K) for w in w_dev]
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(ys[i], singles[i]), f"matrix {i}"
    y_ref, mag = orc.gemv(Q4, wq[0], x.numpy(), M, K, with_mag=True)
    _check_float(_np(ys[0]), y_ref, mag, "matrix 0 of the large launch")


@pytest.mark.parametrize("K", [256, 2304, 11008])
def test_gemv_activation_paths_bit_identical(bq, dev, K):
    """x's records built in every GEMV CTA (two lanes per block) and by the
    prep kernel (eight lanes per block) are the same, so y is bit-identical,
    on plain, scaled, sparse, exact-tie and subnormal-scale activations."""
    import ctypes
    from block_quantized_weight_row_gb300 import binding, inputs
    L = binding.lib()
    M = 300
    w = bq.quantize_rows(Q4, inputs.weight(M, K, seed=K + 17).to(dev))
    base = inputs.activation(K, seed=K + 19)
    ties = base.clone()
    ties[0::32] = 127.0                                   # scale exactly 1.0 in every block ...
    ties[1::32] = torch.arange(1, K // 32 + 1) % 100 + 0.5  # ... and a value on a tie
    tiny = base * 1e-6                                    # scales below binary16's normal range
    cases = {"plain": base, "small": base * 1e-3, "large": base * 300.0, "ties": ties, "tiny": tiny}
    sparse = base.clone()
    sparse[::3] = 0.0
    cases["sparse"] = sparse
    ws = torch.empty(max(256, int(L.bq_gemv_workspace_size(Q4, K))), dtype=torch.uint8, device=dev)
    assert L.bq_set_stream(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    for name, x in cases.items():
        xd = x.to(dev)
        y_ws = torch.empty(M, device=dev)
        y_cta = torch.empty(M, device=dev)
        assert L.bq_set_workspace(ctypes.c_void_p(ws.data_ptr()), ws.numel()) == 0
        assert L.bq_gemv(Q4, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(xd.data_ptr()),
                         ctypes.c_void_p(y_ws.data_ptr()), M, K) == 0
        assert L.bq_set_workspace(None, 0) == 0
        assert L.bq_gemv(Q4, ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(xd.data_ptr()),
                         ctypes.c_void_p(y_cta.data_ptr()), M, K) == 0
        torch.cuda.synchronize()
        assert torch.equal(y_ws, y_cta), name


# ------------------------------------------------ GEMV sequence (one launch) --

def _seq_case(t, seed, shapes):
    """Batches of (K, [M...]) with seeded weights and inputs, quantized by the oracle."""
    from block_quantized_weight_row_gb300 import inputs
    batches = []
    for g, (K, Ms) in enumerate(shapes):
        x = inputs.activation(K, seed=seed + 100 * g)
        mats = []
        for i, M in enumerate(Ms):
            W = inputs.weight(M, K, seed=seed + 100 * g + 1 + i)
            mats.append(_orc().quantize_rows(t, W.numpy()))
        batches.append((K, Ms, x, mats))
    return batches


def _orc():
    import oracle
    return oracle


@pytest.mark.parametrize("t", [Q4, Q8])
def test_gemv_sequence_matches_oracle(bq, orc, dev, t):
    """Mixed K (one to 16 groups of 8 blocks per row, 43 for 11008), ragged
    and empty matrices, one to three matrices per batch."""
    shapes = [(256, [7]), (4096, [300, 0, 129]), (1024, [1]), (11008, [64, 33]), (2304, [200]),
              (512, [1000, 17, 5])]
    batches = _seq_case(t, 4242, shapes)
    groups = []
    for K, Ms, x, mats in batches:
        outs = [torch.full((M,), float("nan"), device=dev) for M in Ms]
        groups.append(([torch.from_numpy(w).to(dev) for w in mats], x.to(dev), Ms, K, outs))
    bq.gemv_sequence(t, groups)
    torch.cuda.synchronize()
    from block_quantized_weight_row_gb300 import binding
    assert binding.device_status() == 0, "a bounded wait ran out"
    for (K, Ms, x, mats), g in zip(batches, groups):
        for M, w, y in zip(Ms, mats, g[4]):
            if M == 0:
                continue
            y_ref, mag = orc.gemv(t, w, x.numpy(), M, K, with_mag=True)
            _check_float(_np(y), y_ref, mag, f"sequence K={K} M={M}")


def test_gemv_sequence_chain_reads_previous_outputs(bq, orc, dev):
    """x of batch g+1 is the output of batch g (square matrices): the launch
    must read it only after every CTA wrote it. The same chain run as one
    bq_gemv_multi call per batch (same device arithmetic, launches ordered by
    the stream) gives identical bits; the first product is also checked
    against the oracle."""
    from block_quantized_weight_row_gb300 import inputs
    K, G = 2048, 12
    ws = [bq.quantize_rows(Q4, inputs.weight(K, K, seed=700 + g, device=dev)) for g in range(G)]
    x0 = inputs.activation(K, seed=699, device=dev)
    ys = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    groups = [([ws[g]], x0 if g == 0 else ys[g - 1], [K], K, [ys[g]]) for g in range(G)]
    bq.gemv_sequence(Q4, groups)
    ref = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    for g in range(G):
        bq.gemv_multi(Q4, [ws[g]], x0 if g == 0 else ref[g - 1], [K], K, outs=[ref[g]])
    torch.cuda.synchronize()
    for g in range(G):
        assert torch.equal(ys[g], ref[g]), f"batch {g}"
    y_ref, mag = orc.gemv(Q4, _np(ws[0]), x0.cpu().numpy(), K, K, with_mag=True)
    _check_float(_np(ys[0]), y_ref, mag, "chain batch 0")


def test_gemv_sequence_mixed_waits_match_per_launch(bq, orc, dev):
    """20 batches, some reading the previous batch's output (RAW), one whose
    output overwrites an earlier batch's input (WAR), the rest independent:
    the record buffers rotate through every kind of batch. Identical bits to
    one bq_gemv_multi call per batch, no bounded wait runs out, and the first
    and last products match the oracle."""
    from block_quantized_weight_row_gb300 import binding, inputs
    K = 1024
    G = 20
    ws = [bq.quantize_rows(Q4, inputs.weight(K, K, seed=800 + g, device=dev)) for g in range(G)]
    xs = [inputs.activation(K, seed=850 + g, device=dev) for g in range(G)]
    spare = inputs.activation(K, seed=899, device=dev)
    reads_prev = {3, 4, 9, 14, 15, 16}
    def build(outs, x_war):
        groups = []
        for g in range(G):
            x = outs[g - 1] if g in reads_prev else (x_war if g == 7 else xs[g])
            out = x_war if g == 11 else outs[g]  # batch 11 overwrites batch 7's input
            groups.append(([ws[g]], x, [K], K, [out]))
        return groups
    outs = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    x_war = spare.clone()
    assert binding.device_status() == 0
    bq.gemv_sequence(Q4, build(outs, x_war))
    assert binding.device_status() == 0
    ref = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    x_war_ref = spare.clone()
    for w_list, x, M_list, K_, y_list in build(ref, x_war_ref):
        bq.gemv_multi(Q4, w_list, x, M_list, K_, outs=y_list)
    torch.cuda.synchronize()
    for g in range(G):
        if g != 11:
            assert torch.equal(outs[g], ref[g]), f"batch {g}"
    assert torch.equal(x_war, x_war_ref), "batch 11's output (over batch 7's input)"
    for g in (0, G - 1):
        y_ref, mag = orc.gemv(Q4, _np(ws[g]), xs[g].cpu().numpy() if g not in reads_prev else _np(ref[g - 1]),
                              K, K, with_mag=True)
        _check_float(_np(outs[g]), y_ref, mag, f"batch {g}")


def test_gemv_sequence_longer_than_one_launch(bq, orc, dev):
    """300 batches and 600 matrices: more than one launch's worth, split on
    the host; every output still matches the oracle."""
    from block_quantized_weight_row_gb300 import inputs
    K = 256
    W = inputs.weight(48, K, seed=31)
    wq = orc.quantize_rows(Q8, W.numpy())
    w_dev = torch.from_numpy(wq).to(dev)
    xs = inputs.activation(K, seed=32, rows=300)
    groups = []
    for g in range(300):
        outs = [torch.full((48,), float("nan"), device=dev) for _ in range(2)]
        groups.append(([w_dev, w_dev], xs[g].to(dev), [48, 48], K, outs))
    bq.gemv_sequence(Q8, groups)
    torch.cuda.synchronize()
    for g in (0, 1, 255, 256, 299):
        y_ref, mag = orc.gemv(Q8, wq, xs[g].numpy(), 48, K, with_mag=True)
        for y in groups[g][4]:
            _check_float(_np(y), y_ref, mag, f"batch {g}")


def test_gemv_sequence_full_decode_step_matches_per_launch(bq, orc, dev):
    """The Qwen3-0.6B-shaped decode step (28 layers, 112 batches, 196
    matrices): identical bits to one launch per batch, and sampled rows of
    the last layer against the oracle."""
    from block_quantized_weight_row_gb300 import inputs
    import bench
    step = bench.build_decode_step("qwen3-0.6b-decode", dev, bq, inputs)
    seq_out = []
    groups = []
    for g in step["groups"]:
        outs = [torch.full_like(y, float("nan")) for y in g["y"]]
        seq_out.append(outs)
        groups.append((g["w"], g["x"], g["M"], g["K"], outs))
    bq.gemv_sequence(Q4, groups)
    bench.run_step(step, bq, True)
    torch.cuda.synchronize()
    from block_quantized_weight_row_gb300 import binding
    assert binding.device_status() == 0, "a bounded wait ran out"
    for g, outs in zip(step["groups"], seq_out):
        for y_ref, y in zip(g["y"], outs):
            assert torch.equal(y, y_ref)
    g = step["groups"][-1]
    y_ref, mag = orc.gemv(Q4, _np(g["w"][0]), _np(g["x"]), g["M"][0], g["K"], with_mag=True)
    _check_float(_np(seq_out[-1][0]), y_ref, mag, "last batch")


def test_gemv_sequence_two_group_launch_matches_per_launch(bq, orc, dev):
    """Batches of 4096 x 4096 Q8_0 (17.8 MB each, more than 64 KB per CTA):
    the launch takes two consumer groups of eight warps (the 7B decode step's
    configuration, without the per-batch stage table). Batches 2 and 3 read
    the previous output, the rest are independent: identical bits to one
    bq_gemv_multi call per batch, no bounded wait runs out, and batch 0 and
    batch 3 match the oracle."""
    from block_quantized_weight_row_gb300 import binding, inputs
    K = 4096
    G = 6
    ws = [bq.quantize_rows(Q8, inputs.weight(K, K, seed=870 + g, device=dev)) for g in range(G)]
    xs = [inputs.activation(K, seed=880 + g, device=dev) for g in range(G)]
    reads_prev = {2, 3}
    def build(outs):
        return [([ws[g]], outs[g - 1] if g in reads_prev else xs[g], [K], K, [outs[g]]) for g in range(G)]
    outs = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    assert binding.device_status() == 0
    bq.gemv_sequence(Q8, build(outs))
    ref = [torch.full((K,), float("nan"), device=dev) for _ in range(G)]
    for w_list, x, M_list, K_, y_list in build(ref):
        bq.gemv_multi(Q8, w_list, x, M_list, K_, outs=y_list)
    torch.cuda.synchronize()
    assert binding.device_status() == 0, "a bounded wait ran out"
    for g in range(G):
        assert torch.equal(outs[g], ref[g]), f"batch {g}"
    for g in (0, 3):
        x = xs[g] if g not in reads_prev else ref[g - 1]
        y_ref, mag = orc.gemv(Q8, _np(ws[g]), _np(x), K, K, with_mag=True)
        _check_float(_np(outs[g]), y_ref, mag, f"batch {g}")


def test_gemv_sequence_timeout_path_returns_error(bq, orc, dev):
    """Poll budget 0: every wait gives up at once, the grid-wide abort flag
    stops the other CTAs, copies in flight are drained, the status reports
    the timeout, and the next call is correct."""
    from block_quantized_weight_row_gb300 import binding
    L = binding.lib()
    batches = _seq_case(Q4, 515, [(1024, [256]), (1024, [128])])
    groups = [([torch.from_numpy(w).to(dev) for w in mats], x.to(dev), Ms, K, None) for K, Ms, x, mats in batches]
    assert binding.device_status() == 0
    try:
        assert L.bq_set_spin_limit(0) == 0
        bq.gemv_sequence(Q4, groups)
        assert binding.device_status() == -6
    finally:
        L.bq_set_spin_limit(-1)
    outs = bq.gemv_sequence(Q4, groups)
    assert binding.device_status() == 0
    for (K, Ms, x, mats), ys in zip(batches, outs):
        y_ref, mag = orc.gemv(Q4, mats[0], x.numpy(), Ms[0], K, with_mag=True)
        _check_float(_np(ys[0]), y_ref, mag, "after timeout")


# ------------------------------------- decode attention over the KV cache --

def _attn_tol(mag, smax, D):
    """Bound for the GPU's attention output: 1e-5 of sum_t w_t |v_t| (fp32
    accumulation), plus the effect of fp32 score rounding: each score carries
    at most (blocks + 2) roundings of ~|s|, taken with a factor 8 margin, and
    moving the softmax by ds moves o by at most 2 ds sum_t w_t |v_t|."""
    ds = 8.0 * (D // 32 + 2) * 2.0 ** -24 * (1.0 + smax)[:, None]
    return (1e-5 + 2.0 * ds) * mag


def _attn_case(orc, T, H, NKV, D, kt, vt, seed, centered=False):
    rng = np.random.default_rng(seed)
    mu = rng.uniform(-2, 2, size=(NKV, D)).astype(np.float32)
    Kf = (mu + rng.normal(size=(T, NKV, D))).astype(np.float32)
    Vf = rng.normal(size=(T, NKV, D)).astype(np.float32)
    bias = Kf.astype(np.float64).mean(axis=0).astype(np.float32) if centered else None
    K = orc.kv_quantize(kt, Kf, bias, T, NKV, D)
    V = orc.kv_quantize(vt, Vf, None, T, NKV, D)
    q = rng.normal(size=(H, D)).astype(np.float32)
    return q, K, V


@pytest.mark.parametrize("T,H,NKV,D,kt,vt", [
    (1, 4, 2, 64, Q4, Q8), (7, 2, 1, 32, Q8, Q4), (33, 8, 8, 128, Q4, Q8), (1000, 16, 8, 128, Q4, Q8),
    (300, 32, 4, 64, Q8, Q8), (4097, 16, 4, 128, Q4, Q4), (130, 1, 1, 256, Q8, Q8), (70000, 8, 8, 128, Q4, Q8),
    # head_dim 96: three blocks per row; a kv-head count that is not a power
    # of two, and eight heads per kv head at head_dim 256, take the
    # block-wide kernel
    (333, 4, 4, 96, Q4, Q8), (517, 6, 3, 64, Q4, Q8), (300, 16, 2, 256, Q8, Q4),
    # over 1024 chunks: the combine takes its chunks in two rounds; exactly
    # 1024 chunks (one full round) and 1025 (a second round of one chunk
    # holding one token)
    (600000, 2, 1, 32, Q4, Q8), (524288, 2, 1, 32, Q4, Q8), (524289, 2, 1, 32, Q8, Q4)])
def test_attn_decode_matches_oracle(bq, orc, dev, T, H, NKV, D, kt, vt):
    q, K, V = _attn_case(orc, T, H, NKV, D, kt, vt, seed=T + 31 * H + D)
    scale = 1.0 / math.sqrt(D)
    o = _np(bq.attn_decode(kt, vt, torch.from_numpy(q).to(dev), torch.from_numpy(K).to(dev),
                           torch.from_numpy(V).to(dev), NKV, scale))
    o_ref, mag, smax = orc.attn_decode(kt, vt, q, K, V, T, H, NKV, D, scale, with_mag=True)
    err = np.abs(o.astype(np.float64) - o_ref)
    tol = _attn_tol(mag, smax, D)
    assert np.all(err <= tol), f"worst err/tol {float((err / tol).max()):.3g}"


def test_attn_decode_full_layer_with_mean_centered_k(bq, orc, dev):
    """A full 32768-token layer of the KV-write workload shape (8 kv heads,
    16 query heads, head_dim 128), K mean-centered before Q4_0."""
    T, H, NKV, D = 32768, 16, 8, 128
    q, K, V = _attn_case(orc, T, H, NKV, D, Q4, Q8, seed=77, centered=True)
    scale = 1.0 / math.sqrt(D)
    o = _np(bq.attn_decode(Q4, Q8, torch.from_numpy(q).to(dev), torch.from_numpy(K).to(dev),
                           torch.from_numpy(V).to(dev), NKV, scale))
    o_ref, mag, smax = orc.attn_decode(Q4, Q8, q, K, V, T, H, NKV, D, scale, with_mag=True)
    assert np.all(np.abs(o.astype(np.float64) - o_ref) <= _attn_tol(mag, smax, D))


def test_attn_decode_timeout_path_returns_error(bq, orc, dev):
    from block_quantized_weight_row_gb300 import binding
    L = binding.lib()
    T, H, NKV, D = 2000, 8, 4, 128
    q, K, V = _attn_case(orc, T, H, NKV, D, Q4, Q8, seed=5)
    args = (torch.from_numpy(q).to(dev), torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev))
    assert binding.device_status() == 0
    try:
        assert L.bq_set_spin_limit(0) == 0
        bq.attn_decode(Q4, Q8, *args, NKV, 0.1)
        assert binding.device_status() == -6
    finally:
        L.bq_set_spin_limit(-1)
    o = _np(bq.attn_decode(Q4, Q8, *args, NKV, 0.1))
    assert binding.device_status() == 0
    o_ref, mag, smax = orc.attn_decode(Q4, Q8, q, K, V, T, H, NKV, D, 0.1, with_mag=True)
    assert np.all(np.abs(o.astype(np.float64) - o_ref) <= _attn_tol(mag, smax, D))


# ------------------------------- Hadamard-rotated K cache and calibration --

ROT = 1


def _outlier_rows(rng, T, NKV, D):
    """K rows with per-channel means and a few outlier channels (where the
    rotation matters), plus near-tie values after scaling."""
    K = rng.normal(size=(T, NKV, D)) + rng.uniform(-2, 2, size=(NKV, D))
    K[..., rng.choice(D, size=max(1, D // 32), replace=False)] *= 20.0
    return K.astype(np.float32)


# (9, 5, 1024): a bias of 160 blocks, beyond the 128 staged in shared memory
@pytest.mark.parametrize("T,NKV,D", [(1, 1, 64), (33, 2, 64), (1000, 8, 128), (7, 1, 256), (130, 3, 192),
                                     (9, 5, 1024)])
def test_kv_write_rotated_bit_exact(bq, orc, dev, T, NKV, D):
    rng = np.random.default_rng(T * 7 + D)
    K = _outlier_rows(rng, T, NKV, D)
    calib = _outlier_rows(rng, 64, NKV, D)
    bias = orc.kv_bias(calib, ROT, 64, NKV, D)
    Kd = torch.from_numpy(K).to(dev)
    got = _np(bq.kv_quantize(Q4, Kd, torch.from_numpy(bias).to(dev), basis=ROT))
    assert np.array_equal(got, orc.kv_quantize(Q4, K, bias, T, NKV, D, basis=ROT))
    assert np.array_equal(_np(bq.kv_quantize(Q4, Kd, None, basis=ROT)), orc.kv_quantize(Q4, K, None, T, NKV, D, basis=ROT))
    assert np.array_equal(_np(bq.kv_quantize(Q8, Kd, None, basis=ROT)), orc.kv_quantize(Q8, K, None, T, NKV, D, basis=ROT))


def test_kv_write_rotated_full_layer(bq, orc, dev):
    """A full 32768-token layer of the KV-write workload, K rotated and
    mean-centered with a bias calibrated in the rotated basis."""
    from block_quantized_weight_row_gb300 import inputs
    cfg = inputs.WORKLOADS["kv-write"]
    L = inputs.kv_layer(0, cfg["tokens"], cfg["kv_heads"], cfg["head_dim"], cfg["calib_tokens"], device=dev)
    bias = bq.kv_bias(L.K_calib, ROT)
    assert np.array_equal(_np(bias), orc.kv_bias(_np(L.K_calib), ROT, *L.K_calib.shape))
    got = _np(bq.kv_quantize(Q4, L.K, bias, basis=ROT))
    assert np.array_equal(got, orc.kv_quantize(Q4, _np(L.K), _np(bias), *L.K.shape, basis=ROT))


@pytest.mark.parametrize("T,NKV,D,basis", [(4096, 8, 128, 0), (4096, 8, 128, 1), (37, 3, 64, 1), (5, 1, 96, 0),
                                           (1, 2, 256, 1)])
def test_kv_bias_bit_exact(bq, orc, dev, T, NKV, D, basis):
    rng = np.random.default_rng(T + D + basis)
    rows = _outlier_rows(rng, T, NKV, D)
    got = _np(bq.kv_bias(torch.from_numpy(rows).to(dev), basis))
    assert np.array_equal(got, orc.kv_bias(rows, basis, T, NKV, D))


def test_kv_bias_from_another_basis_fails_fast(bq, dev):
    from block_quantized_weight_row_gb300 import binding
    K = torch.ones(4, 2, 64, device=dev)
    out = torch.full((4, 2, 36), 7, dtype=torch.uint8, device=dev)
    for basis, bias_basis in ((1, 0), (0, 1)):
        with pytest.raises(binding.BQError) as e:
            bq.kv_quantize(Q4, K, torch.zeros(2, 64, device=dev), out=out, basis=basis, bias_basis=bias_basis)
        assert e.value.status == -8
    torch.cuda.synchronize()
    assert bool((out == 7).all())  # nothing was written


@pytest.mark.parametrize("T,H,NKV,D,kt,vt", [
    (1000, 16, 8, 128, Q4, Q8), (300, 8, 2, 64, Q8, Q8), (4097, 16, 4, 128, Q4, Q4), (130, 1, 1, 256, Q8, Q8),
    (517, 6, 3, 64, Q4, Q8), (300, 16, 2, 256, Q8, Q4)])
def test_attn_decode_rotated_matches_oracle(bq, orc, dev, T, H, NKV, D, kt, vt):
    """Attention over a rotated (and, for Q4_0, mean-centered) K cache: q is
    rotated alike by both kernels (the last two shapes take the block-wide
    kernel)."""
    rng = np.random.default_rng(T + 3 * H + D)
    Kf = _outlier_rows(rng, T, NKV, D)
    Vf = rng.normal(size=(T, NKV, D)).astype(np.float32)
    bias = orc.kv_bias(Kf, ROT, T, NKV, D) if kt == Q4 else None
    K = orc.kv_quantize(kt, Kf, bias, T, NKV, D, basis=ROT)
    V = orc.kv_quantize(vt, Vf, None, T, NKV, D)
    q = rng.normal(size=(H, D)).astype(np.float32)
    scale = 1.0 / math.sqrt(D)
    o = _np(bq.attn_decode(kt, vt, torch.from_numpy(q).to(dev), torch.from_numpy(K).to(dev),
                           torch.from_numpy(V).to(dev), NKV, scale, k_basis=ROT))
    o_ref, mag, smax = orc.attn_decode(kt, vt, q, K, V, T, H, NKV, D, scale, with_mag=True, k_basis=ROT)
    err = np.abs(o.astype(np.float64) - o_ref)
    tol = _attn_tol(mag, smax, D)
    assert np.all(err <= tol), f"worst err/tol {float((err / tol).max()):.3g}"


# ---------------------------------------------- legacy types Q4_1, Q5_0, Q5_1 --

LEGACY_TYPES = [3, 6, 7]


def _legacy_input(rng, rows, cols):
    """Normal, heavy-tailed, offset, constant and near-tie blocks, with the
    quantizer's adversarial blocks and their negations and rescalings."""
    from block_quantized_weight_row_gb300 import inputs
    x = np.concatenate([rng.normal(size=(rows, cols)), rng.standard_t(2, size=(rows, cols)) * 10,
                        rng.normal(size=(rows, cols)) * 1e-3 + 40.0]).astype(np.float32)
    adv = inputs.adversarial_blocks().numpy()
    adv = np.concatenate([adv, -adv, adv * 1e-4 + 1.0, adv * 3e3, np.full_like(adv, 2.5)]).reshape(-1)
    pad = (-adv.size) % cols
    adv = np.concatenate([adv, np.zeros(pad, np.float32)]).reshape(-1, cols)
    # near ties: x = m + (k + 0.5) d for scales d exactly representable in binary16
    k = rng.integers(0, 15, size=(rows, cols)).astype(np.float32)
    d = np.float32(2.0) ** rng.integers(-8, 4, size=(rows, 1)).astype(np.float32)
    ties = (k + np.float32(0.5)) * d - np.float32(3.0) * d
    ties[:, ::32] = np.float32(-3.0) * d[:, :1]   # every block's minimum ...
    ties[:, 1::32] = np.float32(12.0) * d[:, :1]  # ... and maximum: Q4_1's scale is d exactly, ties exact
    return np.concatenate([x, adv.astype(np.float32), ties.astype(np.float32)])


@pytest.mark.parametrize("t", LEGACY_TYPES)
def test_legacy_quantize_and_dequantize_bit_exact(bq, orc, dev, t):
    x = _legacy_input(np.random.default_rng(t), 200, 256)
    got = _np(bq.quantize_rows(t, torch.from_numpy(x).to(dev)))
    ref = orc.quantize_rows(t, x)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"
    deq = _np(bq.dequantize_rows(t, torch.from_numpy(ref).to(dev), 256))
    dref = orc.dequantize_rows(t, ref, 256)
    # bit for bit, except that NaN payloads (a block whose scale overflowed
    # binary16: outside the supported range) only need to be NaN on both sides
    bad = np.argwhere((deq.view(np.uint32) != dref.view(np.uint32)) & ~(np.isnan(deq) & np.isnan(dref)))
    assert len(bad) == 0, (f"{len(bad)} values differ; first {bad[:3].tolist()}: gpu {deq[tuple(bad[0])]!r} "
                           f"oracle {dref[tuple(bad[0])]!r}, block bytes "
                           f"{ref[bad[0][0], (bad[0][1] // 32) * ref.shape[1] // 8:][:ref.shape[1] // 8].tolist()}")


@pytest.mark.parametrize("t", LEGACY_TYPES)
@pytest.mark.parametrize("M,K", [(1, 32), (37, 96), (4096, 4096), (11008, 4096), (300, 11008)])
def test_legacy_gemv_matches_oracle(bq, orc, dev, t, M, K):
    rng = np.random.default_rng(M + K + t)
    W = (rng.normal(size=(M, K)) * 0.02 + rng.uniform(-0.01, 0.01, size=(M, 1))).astype(np.float32)
    x = rng.normal(size=K).astype(np.float32)
    wb = orc.quantize_rows(t, W)
    y = _np(bq.gemv(t, torch.from_numpy(wb).to(dev), torch.from_numpy(x).to(dev), M, K))
    y_ref, mag = orc.gemv(t, wb, x, M, K, with_mag=True)
    _check_float(y, y_ref, mag, f"type {t}")


@pytest.mark.parametrize("t", LEGACY_TYPES)
def test_legacy_kv_write_bit_exact(bq, orc, dev, t):
    rng = np.random.default_rng(30 + t)
    T, NKV, D = 1000, 8, 128
    K = (rng.normal(size=(T, NKV, D)) + rng.uniform(-2, 2, size=(NKV, D))).astype(np.float32)
    got = _np(bq.kv_quantize(t, torch.from_numpy(K).to(dev), None))
    assert np.array_equal(got, orc.kv_quantize(t, K, None, T, NKV, D))


# ------------------------------------------------------ k-quants Q4_K, Q6_K --

KQUANTS = [12, 14]


@pytest.mark.parametrize("t", KQUANTS)
def test_kquant_quantize_and_dequantize_bit_exact(bq, orc, dev, t):
    rng = np.random.default_rng(70 + t)
    x = np.concatenate([rng.normal(size=(100, 512)), rng.standard_t(2, size=(100, 512)) * 10,
                        rng.uniform(0.5, 3.0, size=(100, 512)), rng.normal(size=(100, 512)) * 1e-3 + 40.0,
                        np.zeros((4, 512)), np.full((4, 512), -2.5)]).astype(np.float32)
    got = _np(bq.quantize_rows(t, torch.from_numpy(x).to(dev)))
    ref = orc.quantize_rows(t, x)
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"
    deq = _np(bq.dequantize_rows(t, torch.from_numpy(ref).to(dev), 512))
    assert np.array_equal(deq.view(np.uint32), orc.dequantize_rows(t, ref, 512).view(np.uint32))


@pytest.mark.parametrize("t", KQUANTS)
@pytest.mark.parametrize("M,K", [(1, 256), (37, 768), (4096, 4096), (11008, 4096), (300, 11008),
                                 # Q6_K rows not a multiple of 16 bytes: bulk copies of whole
                                 # quanta of 8 (K = 768, 11008) or 4 (K = 2560) rows
                                 (96, 768), (4096, 11008), (52, 2560)])
def test_kquant_gemv_matches_oracle(bq, orc, dev, t, M, K):
    rng = np.random.default_rng(M + K + t)
    W = (rng.normal(size=(M, K)) * 0.02).astype(np.float32)
    x = rng.normal(size=K).astype(np.float32)
    wb = orc.quantize_rows(t, W)
    y = _np(bq.gemv(t, torch.from_numpy(wb).to(dev), torch.from_numpy(x).to(dev), M, K))
    y_ref, mag = orc.gemv(t, wb, x, M, K, with_mag=True)
    _check_float(y, y_ref, mag, f"type {t}")
