"""Pins of the CPU oracle to facts outside itself (runs without a GPU).

Each test checks the oracle against something it does not compute itself:
sizes printed by the pages, blocks worked out by hand, numpy's IEEE binary16
and rint, the round-trip bound that the symmetric block rule implies, brute
force fp64 products of dequantized operands, integer dots recomputed in int64
from dequantized values, numpy's fp32 subtraction for the mean-centering bias,
and the softmax shift identity the KV-cache article relies on.
"""
import math

import numpy as np
import pytest

from tests import golden

Q4, Q8 = 2, 8
TYPES = {"Q4_0": Q4, "Q8_0": Q8}


# ---------------------------------------------------------------- sizes ----

def test_block_sizes_match_pages(orc):
    s = golden.sizes()
    assert orc.block_bytes(Q4) == s["q4_0_bytes_per_32"] == 18
    assert orc.block_bytes(Q4) * 8 / 32 == s["q4_0_bits_per_weight"]
    assert orc.block_bytes(Q8) * 8 / 32 == s["q8_0_bits_per_weight"]
    assert round(32 * 2 / orc.block_bytes(Q4), 1) == s["q4_0_vs_fp16"]
    assert round(32 * 4 / orc.block_bytes(Q4), 1) == s["q4_0_vs_fp32"]
    assert round(orc.block_bytes(Q4) / 32, 2) == s["kv_q4_0_bytes_per_elem"]
    assert round(orc.block_bytes(Q8) / 32, 2) == s["kv_q8_0_bytes_per_elem"]
    # KV cache of the pages' 0.6B model: 16384 cells x 28 layers x 8 heads x 128, K and V
    elems = 16384 * 28 * 8 * 128 * 2
    assert elems * 2 / 2**20 == s["kv_f16_mib"]
    assert elems // 32 * orc.block_bytes(Q8) / 2**20 == s["kv_q8_0_mib"]
    # 7B-shaped Q4_0 projections are most of the "about 3.8 GB" file
    proj = 32 * (4 * 4096 * 4096 + 3 * 4096 * 11008) // 32 * orc.block_bytes(Q4)
    assert 0.94 * s["q4_0_7b_gb"] * 1e9 < proj < s["q4_0_7b_gb"] * 1e9


def test_output_sizes(orc):
    x = np.zeros((3, 96), np.float32)
    assert orc.quantize_rows(Q4, x).shape == (3, 3 * 18)
    assert orc.quantize_rows(Q8, x).shape == (3, 3 * 34)


# ---------------------------------------------------- hand-worked blocks ----

@pytest.mark.parametrize("case", golden.hand_blocks(), ids=lambda c: f"{c[0]}-{c[1]}")
def test_hand_worked_blocks(orc, case):
    tname, _name, vals, expected = case
    x = np.zeros((1, 32), np.float32)
    for i, v in vals.items():
        x[0, i] = v
    got = orc.quantize_rows(TYPES[tname], x).tobytes()
    assert got.hex() == expected.hex()


def test_hand_worked_dequantize(orc):
    # scale 1.0 blocks dequantize to their codes exactly
    blk = bytes.fromhex("003c5f888a8a" + "88" * 12)
    xh = orc.dequantize_rows(Q4, np.frombuffer(blk, np.uint8), 32)[0]
    exp = np.zeros(32, np.float32)
    exp[0], exp[2], exp[3], exp[16] = 7, 2, 2, -3
    np.testing.assert_array_equal(xh, exp)
    blk8 = bytes.fromhex("003c" + "81" + "40" * 2 + "00" * 29)
    xh8 = orc.dequantize_rows(Q8, np.frombuffer(blk8, np.uint8), 32)[0]
    exp8 = np.zeros(32, np.float32)
    exp8[0], exp8[1], exp8[2] = -127, 64, 64
    np.testing.assert_array_equal(xh8, exp8)


# ------------------------------------------------ IEEE binary16, rounding ----

def test_f32_to_f16_matches_numpy(orc):
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000),
        np.array([0.0, -0.0, 1.0, 65504.0, 65519.0, 65520.0, 7e5, -7e5, 6.1035156e-05,
                  6.0975552e-05, 5.9604645e-08, 2.9802322e-08, 2.9802326e-08, 8.940697e-08,
                  1.0004, 1.0006, 1.00048828125, 1.00146484375, 2049.0, 2051.0, 1e-30,
                  np.inf, -np.inf], np.float32),
    ])
    # halfway cases between consecutive binary16 values, in every binade
    h = np.arange(0, 0x7BFF, 37, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mids = ((lo + hi) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    for v in vals:
        assert orc.f32_to_f16_bits(v) == int(np.float32(v).astype(np.float16).view(np.uint16)), v


def test_f16_to_f32_matches_numpy_all_codes(orc):
    for h in range(0, 1 << 16):
        ref = np.uint16(h).view(np.float16).astype(np.float32)
        got = np.float32(orc.f16_bits_to_f32(h))
        if np.isnan(ref):
            assert np.isnan(got)
        else:
            assert got.view(np.uint32) == ref.view(np.uint32), hex(h)


def test_round_half_even_matches_rint(orc):
    vals = np.array([0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 7.5, 126.5, 127.5, 0.49999997,
                     2.5000002, 1e8 + 0.5, 3.3, -3.7], np.float32)
    for v in vals:
        assert orc.round_half_even(v) == np.rint(v), v


# -------------------------------------------------------- round trip -------

def _blocks(rng, n):
    """Random blocks over many magnitudes, plus heavy-tailed and signed cases."""
    scale = np.float32(10.0) ** rng.uniform(-3.5, 4, (n, 1)).astype(np.float32)
    x = rng.standard_normal((n, 32)).astype(np.float32) * scale
    x[::7] = rng.standard_cauchy((len(x[::7]), 32)).astype(np.float32)
    x[::11] = np.abs(x[::11])
    return x


@pytest.mark.parametrize("tname", ["Q4_0", "Q8_0"])
def test_round_trip_bound(orc, tname):
    """|x - x_hat| <= d16/2 (1 + 2^-18) whenever the fp16 scale is normal."""
    t = TYPES[tname]
    qmax = 7 if t == Q4 else 127
    rng = np.random.default_rng(2)
    x = _blocks(rng, 4000)
    x = x[np.abs(x).max(axis=1) < 60000 * qmax / 8]          # stay inside fp16 range
    q = orc.quantize_rows(t, x.reshape(-1, 32))
    xh = orc.dequantize_rows(t, q, 32)
    bb = orc.block_bytes(t)
    d16 = q.reshape(-1, bb)[:, :2].copy().view(np.uint16).reshape(-1)
    d = d16.view(np.float16).astype(np.float64)
    normal = d >= 2.0 ** -14
    assert normal.sum() > 3000
    err = np.abs(x.astype(np.float64) - xh.astype(np.float64))
    bound = d[:, None] / 2 * (1 + 2.0 ** -18)
    assert np.all(err[normal] <= bound[normal])
    # the element of largest magnitude gets code +-qmax (no clamping loss)
    codes = np.rint(xh.astype(np.float64)[normal] / d[normal, None])
    amax_idx = np.abs(x[normal]).argmax(axis=1)
    top = codes[np.arange(len(codes)), amax_idx]
    assert np.all(np.abs(top) == qmax)
    assert np.all(np.sign(top) == np.sign(x[normal][np.arange(len(codes)), amax_idx]))
    # the fp16 scale is the ties-to-even rounding of amax/qmax (numpy's binary16)
    amax = np.abs(x).max(axis=1)
    ref = (amax / np.float32(qmax)).astype(np.float32).astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(d16, ref)


@pytest.mark.parametrize("tname", ["Q4_0", "Q8_0"])
def test_codes_in_range_and_zero_blocks(orc, tname):
    t = TYPES[tname]
    import torch
    from block_quantized_weight_row_gb300 import inputs
    x = inputs.adversarial_blocks().numpy()
    q = orc.quantize_rows(t, x)
    xh = orc.dequantize_rows(t, q, 32)
    d = q.reshape(-1, orc.block_bytes(t))[:, :2].copy().view(np.uint16).view(np.float16).astype(np.float64).reshape(-1)
    lo, hi = (-8, 7) if t == Q4 else (-127, 127)
    nz = d > 0
    codes = xh.astype(np.float64)[nz] / d[nz, None]
    assert np.all(codes == np.rint(codes))
    assert codes.min() >= lo and codes.max() <= hi
    assert np.all(xh[~nz] == 0)
    del torch


# ------------------------------------------------------- integer dots ------

@pytest.mark.parametrize("tname", ["Q4_0", "Q8_0"])
def test_block_dots_vs_int64(orc, tname):
    t = TYPES[tname]
    rng = np.random.default_rng(3)
    M, K = 7, 160
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    W[0, :32] = 0
    x = rng.standard_normal(K).astype(np.float32)
    wq = orc.quantize_rows(t, W)
    xq = orc.quantize_rows(Q8, x)
    got = orc.block_dots(t, wq, xq, M, K)
    # recompute codes from the dequantized values (x_hat / scale is exact)
    def codes(blocks, tt, rows):
        xh = orc.dequantize_rows(tt, blocks, K).astype(np.float64).reshape(rows, K // 32, 32)
        d = blocks.reshape(rows, K // 32, -1)[:, :, :2].copy().view(np.uint16)
        d = d.view(np.float16).astype(np.float64).reshape(rows, K // 32, 1)
        return np.where(d > 0, xh / np.where(d > 0, d, 1), 0).astype(np.int64)
    cw = codes(wq, t, M)
    cx = codes(xq, Q8, 1)[0]
    ref = np.einsum("mbj,bj->mb", cw, cx)
    np.testing.assert_array_equal(got, ref)
    # bounds quoted in the design: |sumi| <= 32*8*127 (Q4_0) or 32*127*127 (Q8_0)
    assert np.abs(got).max() <= (32 * 8 * 127 if t == Q4 else 32 * 127 * 127)


# ------------------------------------------------ GEMV / GEMM, brute force --

def _bruteforce(orc, t, wq, X, M, K):
    """fp64 product of the dequantized operands (no blocking)."""
    Wh = orc.dequantize_rows(t, wq, K).astype(np.float64).reshape(M, K)
    Xq = orc.quantize_rows(Q8, X.reshape(-1, K))
    Xh = orc.dequantize_rows(Q8, Xq, K).astype(np.float64)
    return Xh @ Wh.T


@pytest.mark.parametrize("tname", ["Q4_0", "Q8_0"])
@pytest.mark.parametrize("M,K", [(1, 32), (3, 64), (8, 128), (5, 96)])
def test_gemv_matches_bruteforce(orc, tname, M, K):
    t = TYPES[tname]
    rng = np.random.default_rng(M * 1000 + K)
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float32)
    wq = orc.quantize_rows(t, W)
    y, mag = orc.gemv(t, wq, x, M, K, with_mag=True)
    ref = _bruteforce(orc, t, wq, x, M, K)[0]
    # the oracle rounds an (essentially exact) fp64 sum once to fp32
    assert np.all(np.abs(y.astype(np.float64) - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-30)
    assert np.all(mag >= np.abs(ref) * (1 - 1e-12))


@pytest.mark.parametrize("tname", ["Q4_0", "Q8_0"])
def test_gemm_matches_bruteforce_and_gemv(orc, tname):
    t = TYPES[tname]
    rng = np.random.default_rng(5)
    M, N, K = 6, 5, 128
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((N, K)).astype(np.float32)
    wq = orc.quantize_rows(t, W)
    Y = orc.gemm(t, wq, X, M, N, K)
    ref = _bruteforce(orc, t, wq, X, M, K)
    assert Y.shape == (N, M)
    assert np.all(np.abs(Y.astype(np.float64) - ref) <= np.abs(ref) * 2.0 ** -24 + 1e-30)
    for n in range(N):
        np.testing.assert_array_equal(Y[n], orc.gemv(t, wq, X[n], M, K))


def test_gemv_detects_transposed_operands(orc):
    """A non-square case where reading W as K x M would give a different answer."""
    rng = np.random.default_rng(6)
    M, K = 2, 64
    W = (rng.standard_normal((M, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float32)
    wq = orc.quantize_rows(Q4, W)
    y = orc.gemv(Q4, wq, x, M, K)
    Wh = orc.dequantize_rows(Q4, wq, K).astype(np.float64)
    xh = orc.dequantize_rows(Q8, orc.quantize_rows(Q8, x), K)[0].astype(np.float64)
    np.testing.assert_allclose(y, Wh @ xh, rtol=1e-6)


# ------------------------------------------------------------ KV write -----

def test_kv_bias_matches_numpy_subtraction(orc):
    rng = np.random.default_rng(7)
    T, H, D = 9, 3, 64
    K = rng.standard_normal((T, H, D)).astype(np.float32) + 1.5
    b = rng.uniform(-2, 2, (H, D)).astype(np.float32)
    got = orc.kv_quantize(Q4, K, b, T, H, D)
    centered = (K - b[None]).astype(np.float32)           # numpy IEEE fp32 subtraction
    ref = orc.quantize_rows(Q4, centered.reshape(-1, D)).reshape(T, H, -1)
    np.testing.assert_array_equal(got, ref)
    # without a bias the KV write is the plain row quantizer, for both types
    for t in (Q4, Q8):
        np.testing.assert_array_equal(orc.kv_quantize(t, K, None, T, H, D),
                                      orc.quantize_rows(t, K.reshape(-1, D)).reshape(T, H, -1))


def test_kv_bias_rejected_for_q8_0(orc):
    K = np.zeros((1, 1, 32), np.float32)
    with pytest.raises(ValueError):
        orc.kv_quantize(Q8, K, np.zeros((1, 32), np.float32), 1, 1, 32)


def _softmax(z):
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def test_softmax_shift_invariance_fp32():
    """q.k_i = q.(k_i - kbar) + q.kbar; the last term is the same for every key
    of a query row, and softmax(z + c) = softmax(z) (lpnh.cn KV-cache article,
    §解法). Unquantized fp32 K, as the article's F32-cache test does."""
    import torch
    from block_quantized_weight_row_gb300 import inputs
    L = inputs.kv_layer(0, tokens=512, kv_heads=2, head_dim=128, calib_tokens=256)
    bias = L.K_calib.double().mean(dim=0).float().numpy()
    K = L.K.numpy()
    q = inputs.normal((16, 2, 128), 1.0, 99).numpy()
    for h in range(2):
        z0 = (q[:, h] @ K[:, h].T).astype(np.float32) / np.float32(math.sqrt(128))
        z1 = (q[:, h] @ (K[:, h] - bias[h]).T).astype(np.float32) / np.float32(math.sqrt(128))
        assert np.abs(_softmax(z0) - _softmax(z1)).max() <= 1e-6
    del torch


def test_mean_centering_lowers_q4_0_attention_error(orc):
    """Expected, not proved (parity-unpinned magnitude): centering K before
    Q4_0 lowers the attention KL against the fp32 cache."""
    from block_quantized_weight_row_gb300 import inputs
    T, H, D = 1024, 4, 128
    L = inputs.kv_layer(1, tokens=T, kv_heads=H, head_dim=D, calib_tokens=512)
    K = L.K.numpy()
    bias = L.K_calib.double().mean(dim=0).float().numpy()
    q = inputs.normal((32, H, D), 1.0, 98).numpy()
    Kq_plain = orc.dequantize_rows(Q4, orc.kv_quantize(Q4, K, None, T, H, D), D).reshape(T, H, D)
    Kq_cent = orc.dequantize_rows(Q4, orc.kv_quantize(Q4, K, bias, T, H, D), D).reshape(T, H, D)
    kl = {"plain": 0.0, "cent": 0.0}
    for h in range(H):
        p = _softmax(q[:, h].astype(np.float64) @ K[:, h].T.astype(np.float64) / math.sqrt(D))
        for name, Kq in (("plain", Kq_plain), ("cent", Kq_cent)):
            r = _softmax(q[:, h].astype(np.float64) @ Kq[:, h].T.astype(np.float64) / math.sqrt(D))
            kl[name] += float(np.sum(p * (np.log(p) - np.log(r))) / len(p))
    assert kl["cent"] < kl["plain"]


# ---------------------------------------- decode attention over the cache --
# R11 (scaled dot-product attention over the dequantized cache, grouped query
# heads) and R12 (q . k as the Q8_0 block dot); [FA], [SHIFT].

def _q4_block(scale, codes):
    """A Q4_0 block from the format definition: fp16 scale (LE), then byte j =
    (q[j]+8) | (q[j+16]+8) << 4."""
    c = np.asarray(codes, np.int64) + 8
    qs = (c[:16] | (c[16:] << 4)).astype(np.uint8)
    return np.concatenate([np.array([scale], np.float16).view(np.uint8), qs])


def _q8_block(scale, codes):
    return np.concatenate([np.array([scale], np.float16).view(np.uint8),
                           np.asarray(codes, np.int8).view(np.uint8)])


def _rand_cache(orc, rng, T, H, D, kt, vt):
    K = orc.kv_quantize(kt, rng.normal(size=(T, H, D)).astype(np.float32), None, T, H, D)
    V = orc.kv_quantize(vt, rng.normal(size=(T, H, D)).astype(np.float32), None, T, H, D)
    return K, V


def test_attn_single_token_returns_its_value_row(orc):
    rng = np.random.default_rng(3)
    T, NH, NKV, D = 1, 4, 2, 64
    K, V = _rand_cache(orc, rng, T, NKV, D, Q4, Q8)
    q = rng.normal(size=(NH, D)).astype(np.float32)
    o = orc.attn_decode(Q4, Q8, q, K, V, T, NH, NKV, D, 1.0 / math.sqrt(D))
    v = orc.dequantize_rows(Q8, V.reshape(-1), D).reshape(NKV, D)
    for h in range(NH):
        assert np.array_equal(o[h], v[h // 2])  # weight 1, heads 0,1 -> kv 0; 2,3 -> kv 1


def test_attn_equal_keys_give_the_mean_value(orc):
    rng = np.random.default_rng(4)
    T, D = 3, 32
    K1, V = _rand_cache(orc, rng, T, 1, D, Q4, Q4)
    K = np.repeat(K1[:1], T, axis=0)  # the same key bytes for every token
    q = rng.normal(size=(1, D)).astype(np.float32)
    o = orc.attn_decode(Q4, Q4, q, K, V, T, 1, 1, D, 0.3)
    v = orc.dequantize_rows(Q4, V.reshape(-1), D).astype(np.float64)
    assert np.allclose(o[0], v.mean(axis=0), rtol=0, atol=1e-6 * np.abs(v).max())


def test_attn_two_tokens_closed_form(orc):
    """Hand-built blocks: q = 1.0 everywhere quantizes to codes 127 with the
    binary16 scale of 1/127; token 0 has K codes all +1 at scale 0.5, token 1
    alternates +2 / -1 at scale 0.25; V is constant per token. Scores, softmax
    and output then follow in closed form."""
    D = 32
    dq = float(np.float16(np.float32(1.0) / np.float32(127.0)))
    assert round(1.0 / dq) == 127
    K = np.stack([_q4_block(0.5, [1] * 32), _q4_block(0.25, [2, -1] * 16)]).reshape(2, 1, 18)
    V = np.stack([_q8_block(0.5, [10] * 32), _q8_block(0.125, [-20] * 32)]).reshape(2, 1, 34)
    scale = float(np.float32(1.0 / math.sqrt(D)))  # the scale is an fp32 argument
    s0 = scale * 0.5 * dq * (32 * 127 * 1)
    s1 = scale * 0.25 * dq * (16 * 127 * 2 - 16 * 127)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * 5.0 + (1.0 - w0) * (-2.5)
    q = np.ones((1, D), np.float32)
    o, mag, smax = orc.attn_decode(Q4, Q8, q, K, V, 2, 1, 1, D, scale, with_mag=True)
    assert np.allclose(o[0], expect, rtol=1e-6, atol=0)
    assert np.allclose(mag[0], w0 * 5.0 + (1.0 - w0) * 2.5, rtol=1e-12)
    assert math.isclose(smax[0], max(abs(s0), abs(s1)), rel_tol=1e-12)


def test_attn_grouped_heads_read_their_kv_head(orc):
    rng = np.random.default_rng(5)
    T, NH, NKV, D = 40, 6, 3, 64
    K, V = _rand_cache(orc, rng, T, NKV, D, Q8, Q8)
    q = rng.normal(size=(NH, D)).astype(np.float32)
    o = orc.attn_decode(Q8, Q8, q, K, V, T, NH, NKV, D, 0.125)
    for h in range(NH):
        kvh = h // 2
        o1 = orc.attn_decode(Q8, Q8, q[h:h + 1], np.ascontiguousarray(K[:, kvh:kvh + 1]),
                             np.ascontiguousarray(V[:, kvh:kvh + 1]), T, 1, 1, D, 0.125)
        assert np.array_equal(o[h], o1[0])


def test_attn_token_order_does_not_matter(orc):
    rng = np.random.default_rng(6)
    T, NH, NKV, D = 57, 4, 2, 128
    K, V = _rand_cache(orc, rng, T, NKV, D, Q4, Q8)
    q = rng.normal(size=(NH, D)).astype(np.float32)
    o, mag, _ = orc.attn_decode(Q4, Q8, q, K, V, T, NH, NKV, D, 1 / math.sqrt(D), with_mag=True)
    p = rng.permutation(T)
    o2 = orc.attn_decode(Q4, Q8, q, np.ascontiguousarray(K[p]), np.ascontiguousarray(V[p]), T, NH, NKV, D,
                         1 / math.sqrt(D))
    assert np.all(np.abs(o2 - o) <= 1e-6 * mag + 1e-30)


def test_attn_shift_of_all_scores_leaves_the_output(orc):
    """[SHIFT]: a channel block whose key bytes are the same for every token
    adds one constant to every score of a head; the other channels' output is
    unchanged."""
    rng = np.random.default_rng(7)
    T, D = 33, 64
    K, V = _rand_cache(orc, rng, T, 1, D, Q4, Q8)
    q = rng.normal(size=(1, D)).astype(np.float32)
    o = orc.attn_decode(Q4, Q8, q, K, V, T, 1, 1, D, 0.2)
    extra_k = np.tile(_q4_block(0.75, [3] * 32), (T, 1, 1))
    extra_v = np.tile(_q8_block(0.0, [0] * 32), (T, 1, 1))
    K2 = np.concatenate([K.reshape(T, 1, -1), extra_k.reshape(T, 1, -1)], axis=2)
    V2 = np.concatenate([V.reshape(T, 1, -1), extra_v.reshape(T, 1, -1)], axis=2)
    q2 = np.concatenate([q, np.full((1, 32), 2.0, np.float32)], axis=1)
    o2, _, s2 = orc.attn_decode(Q4, Q8, q2, K2, V2, T, 1, 1, D + 32, 0.2, with_mag=True)
    _, _, s1 = orc.attn_decode(Q4, Q8, q, K, V, T, 1, 1, D, 0.2, with_mag=True)
    assert s2[0] > s1[0] + 1.0  # the shift is real, and large
    assert np.allclose(o2[0, :D], o[0], rtol=1e-6, atol=1e-7)
    assert np.all(o2[0, D:] == 0.0)


# ------------------------------------- Hadamard rotation of K ([ROT], R14) --

def _h64():
    """H64 of the definition: (-1)^popcount(i & j), fp64, unnormalized."""
    i = np.arange(64)
    pc = np.vectorize(lambda v: bin(v).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


def _rot_exact(x):
    """fp64 matrix product of the definition, every group of 64 values."""
    g = np.asarray(x, np.float64).reshape(-1, 64)
    return (g @ _h64().T / 8.0).reshape(np.shape(x))


def _rot_bound(x):
    """fp32 butterflies: 6 rounded stages, each error at most 2^-24 of the
    partial sums, which never exceed the group's sum of |x|."""
    g = np.abs(np.asarray(x, np.float64)).reshape(-1, 64).sum(axis=1, keepdims=True)
    return np.broadcast_to(7.0 * 2.0 ** -24 * g / 8.0, (g.shape[0], 64)).reshape(np.shape(x))


def test_hadamard_columns_are_the_definition(orc):
    """Each unit vector maps to its column of H64 / 8, exactly (one nonzero
    input: no rounding), which fixes the order, the signs and the scaling."""
    H = _h64()
    for j in range(64):
        e = np.zeros(64, np.float32)
        e[j] = 1.0
        assert np.array_equal(orc.hadamard64(e), (H[:, j] / 8.0).astype(np.float32)), j
    assert np.array_equal(orc.hadamard64(np.ones(64, np.float32))[:2], np.array([8.0, 0.0], np.float32))


def test_hadamard_matches_the_matrix_product(orc):
    rng = np.random.default_rng(11)
    for scale in (1.0, 1e-3, 1e4):
        x = (rng.standard_t(3, size=64 * 40) * scale).astype(np.float32)
        y = orc.hadamard64(x).astype(np.float64)
        assert np.all(np.abs(y - _rot_exact(x)) <= _rot_bound(x))


def test_hadamard_is_orthonormal_and_its_own_inverse(orc):
    rng = np.random.default_rng(12)
    x = rng.normal(size=64 * 16).astype(np.float32)
    y = orc.hadamard64(x)
    g = x.astype(np.float64).reshape(-1, 64)
    assert np.allclose((y.astype(np.float64).reshape(-1, 64) ** 2).sum(1), (g ** 2).sum(1), rtol=1e-6)
    z = orc.hadamard64(y).astype(np.float64)
    assert np.all(np.abs(z - x) <= 2 * _rot_bound(x) + 2 * _rot_bound(y))


def test_hadamard_groups_are_independent(orc):
    rng = np.random.default_rng(13)
    a, b = rng.normal(size=64).astype(np.float32), rng.normal(size=64).astype(np.float32)
    assert np.array_equal(orc.hadamard64(np.concatenate([a, b])),
                          np.concatenate([orc.hadamard64(a), orc.hadamard64(b)]))
    with pytest.raises(ValueError):
        orc.hadamard64(np.zeros(96, np.float32))


def test_rotated_kv_write_of_rotated_codes_is_the_plain_write(orc):
    """K = H^T C / 8 * 8 with C exactly Q8_0-representable (power-of-two
    scales): rotating K gives C up to fp32 rounding far below half a code, so
    the rotated cache of K equals the plain cache of C byte for byte."""
    rng = np.random.default_rng(14)
    T, NKV, D = 5, 2, 128
    codes = rng.integers(-127, 128, size=(T, NKV, D))
    codes[..., ::32] = 127  # every block's extreme is 127: scale exactly 2^-6
    C = (codes * 2.0 ** -6).astype(np.float32)
    K = _rot_exact(C.reshape(-1)).reshape(T, NKV, D).astype(np.float32)  # H is its own inverse (H H / 64 = I)
    plain = orc.kv_quantize(Q8, C, None, T, NKV, D)
    rot = orc.kv_quantize(Q8, K, None, T, NKV, D, basis=1)
    assert np.array_equal(rot, plain)
    assert not np.array_equal(orc.kv_quantize(Q8, K, None, T, NKV, D), plain)


def test_rotated_kv_write_round_trip_in_the_rotated_basis(orc):
    rng = np.random.default_rng(15)
    T, NKV, D = 40, 2, 64
    K = (rng.normal(size=(T, NKV, D)) * rng.uniform(0.1, 3.0, size=(1, 1, D))).astype(np.float32)
    bias = orc.kv_bias(K, 1, T, NKV, D)
    cache = orc.kv_quantize(Q4, K, bias, T, NKV, D, basis=1)
    deq = orc.dequantize_rows(Q4, cache.reshape(T * NKV, -1), D).astype(np.float64).reshape(T, NKV, D)
    target = _rot_exact(K.reshape(-1)).reshape(T, NKV, D) - bias.astype(np.float64)[None]
    d16 = cache.reshape(-1, 18)[:, :2].copy().view(np.float16).astype(np.float64).reshape(T, NKV, D // 32)
    tol = np.repeat(d16, 32, axis=2) / 2 * (1 + 2.0 ** -18) + _rot_bound(K.reshape(-1)).reshape(T, NKV, D) + 1e-6
    assert np.all(np.abs(deq - target) <= tol)


def test_bias_from_another_basis_is_rejected(orc):
    T, NKV, D = 3, 1, 64
    K = np.ones((T, NKV, D), np.float32)
    with pytest.raises(ValueError):
        orc.kv_quantize(Q4, K, np.zeros((NKV, D), np.float32), T, NKV, D, basis=1, bias_basis=0)
    with pytest.raises(ValueError):
        orc.kv_quantize(Q4, K, np.zeros((NKV, D), np.float32), T, NKV, D, basis=0, bias_basis=1)
    with pytest.raises(ValueError):
        orc.kv_quantize(Q4, np.ones((T, NKV, 96), np.float32), None, T, NKV, 96, basis=1)


def test_plain_bias_is_the_channel_mean(orc):
    rng = np.random.default_rng(16)
    T, NKV, D = 300, 3, 96
    K = (rng.normal(size=(T, NKV, D)) + rng.uniform(-2, 2, size=(NKV, D))).astype(np.float32)
    b = orc.kv_bias(K, 0, T, NKV, D)
    ref = K.astype(np.float64).mean(axis=0).astype(np.float32)
    assert np.all(np.abs(b.view(np.int32) - ref.view(np.int32)) <= 1)  # within one fp32 ulp


def test_rotated_bias_is_the_rotation_of_the_mean(orc):
    """Linearity: the mean of the rotated rows is the rotated mean."""
    rng = np.random.default_rng(17)
    T, NKV, D = 200, 2, 128
    K = (rng.normal(size=(T, NKV, D)) + rng.uniform(-2, 2, size=(NKV, D))).astype(np.float32)
    b = orc.kv_bias(K, 1, T, NKV, D).astype(np.float64)
    ref = _rot_exact(K.astype(np.float64).mean(axis=0).reshape(-1)).reshape(NKV, D)
    bound = _rot_bound(np.abs(K).max(axis=0).reshape(-1)).reshape(NKV, D) + 2 * 2.0 ** -24 * np.abs(ref) + 1e-7
    assert np.all(np.abs(b - ref) <= bound)


def test_rotation_spreads_outlier_channels(orc):
    """Expected, not proved (parity unpinned magnitude): with a few outlier
    channels per head, Q4_0 after rotation loses less of K, measured back in
    the original basis, than Q4_0 of the raw rows."""
    rng = np.random.default_rng(18)
    T, NKV, D = 256, 2, 128
    K = rng.normal(size=(T, NKV, D)).astype(np.float32)
    K[..., [3, 40, 77, 101]] *= 25.0
    plain = orc.dequantize_rows(Q4, orc.kv_quantize(Q4, K, None, T, NKV, D).reshape(T * NKV, -1), D)
    rot = orc.dequantize_rows(Q4, orc.kv_quantize(Q4, K, None, T, NKV, D, basis=1).reshape(T * NKV, -1), D)
    back = _rot_exact(rot.reshape(-1)).reshape(T * NKV, D)  # H / 8 is its own inverse
    err_plain = np.mean((plain - K.reshape(T * NKV, D)) ** 2)
    err_rot = np.mean((back - K.reshape(T * NKV, D)) ** 2)
    assert err_rot < 0.5 * err_plain


def test_attn_over_a_rotated_cache_rotates_q(orc):
    """(Hq).(Hk) = q.k: over a rotated Q8_0 cache the output stays close to
    exact fp64 attention of the unquantized rows (quantization noise only),
    and using q unrotated is far off."""
    rng = np.random.default_rng(19)
    T, NH, NKV, D = 120, 4, 2, 128
    K = rng.normal(size=(T, NKV, D)).astype(np.float32)
    V = rng.normal(size=(T, NKV, D)).astype(np.float32)
    q = rng.normal(size=(NH, D)).astype(np.float32)
    scale = 1 / math.sqrt(D)
    Kc = orc.kv_quantize(Q8, K, None, T, NKV, D, basis=1)
    Vc = orc.kv_quantize(Q8, V, None, T, NKV, D)
    vhat = orc.dequantize_rows(Q8, Vc.reshape(T * NKV, -1), D).reshape(T, NKV, D).astype(np.float64)
    exact = np.zeros((NH, D))
    for h in range(NH):
        s = scale * (K[:, h // 2].astype(np.float64) @ q[h].astype(np.float64))
        w = np.exp(s - s.max())
        exact[h] = (w / w.sum()) @ vhat[:, h // 2]
    o = orc.attn_decode(Q8, Q8, q, Kc, Vc, T, NH, NKV, D, scale, k_basis=1)
    o_wrong = orc.attn_decode(Q8, Q8, q, Kc, Vc, T, NH, NKV, D, scale)
    err = np.abs(o - exact).max()
    assert err < 0.02
    assert np.abs(o_wrong - exact).max() > 10 * err


# ---------------------------------------------- legacy types ([LEG], R16-R19) --

Q4_1, Q5_0, Q5_1 = 3, 6, 7
LEGACY = {"Q4_1": Q4_1, "Q5_0": Q5_0, "Q5_1": Q5_1}


def _parse_legacy(t, blocks):
    """The test's own reading of R16: (d16, m16, u[32]) per block, as numpy."""
    b = np.asarray(blocks, np.uint8).reshape(-1, {Q4_1: 20, Q5_0: 22, Q5_1: 24}[t])
    d = b[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
    o = 2
    m = np.zeros_like(d)
    if t != Q5_0:
        m = b[:, 2:4].copy().view(np.float16).astype(np.float64)[:, 0]
        o = 4
    qh = np.zeros(len(b), np.uint64)
    if t != Q4_1:
        qh = b[:, o:o + 4].copy().view(np.uint32)[:, 0].astype(np.uint64)
        o += 4
    nib = b[:, o:o + 16].astype(np.int64)
    lo = np.concatenate([nib & 15, nib >> 4], axis=1)
    hi = ((qh[:, None] >> np.arange(32, dtype=np.uint64)[None, :]) & np.uint64(1)).astype(np.int64)
    return d, m, lo | (hi << 4)


def test_legacy_block_sizes(orc):
    # the "_1" types add one fp16 minimum to the scale (R16); 5-bit types add 32 high bits
    assert orc.block_bytes(Q4_1) == orc.block_bytes(Q4) + 2 == 20
    assert orc.block_bytes(Q5_0) == 2 + 4 + 16 == 22
    assert orc.block_bytes(Q5_1) == orc.block_bytes(Q5_0) + 2 == 24
    assert [orc.block_bytes(t) * 8 / 32 for t in (Q4_1, Q5_0, Q5_1)] == [5.0, 5.5, 6.0]


def test_legacy_hand_blocks(orc):
    # Q4_1: x = -1, 0.5, 1.5, 14, rest 0 -> m = -1, d = 15/15 = 1 (0x3C00);
    # (x - m) = 0, 1.5, 2.5, 15, 1 -> u = 0, 2 (half-even), 2 (half-even), 15, 1
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = [-1.0, 0.5, 1.5, 14.0]
    b = orc.quantize_rows(Q4_1, x)[0]
    assert b[:4].tolist() == [0x00, 0x3C, 0x00, 0xBC]          # d = 1.0, m = -1.0 (0xBC00)
    assert b[4:8].tolist() == [0x10, 0x12, 0x12, 0x1F]          # low nibble u[j], high nibble u[j+16] = 1
    assert b[8:].tolist() == [0x11] * 12
    # Q5_0: x0 = 15, x1 = -15, rest 0 -> d = 1, q = 15, -15, 0 -> u = 31, 1, 16
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 15.0, -15.0
    b = orc.quantize_rows(Q5_0, x)[0]
    assert b[:2].tolist() == [0x00, 0x3C]
    qh = int.from_bytes(bytes(b[2:6]), "little")
    assert qh == 0xFFFFFFFF & ~0b10                              # bit 1 clear: u1 = 1 < 16
    assert b[6:8].tolist() == [0x0F, 0x01] and b[8:].tolist() == [0x00] * 14
    # Q5_1: a constant block -> d = 0, m = 3.25 (0x4280), every u = 0, value 3.25 exactly
    x = np.full((1, 32), 3.25, np.float32)
    b = orc.quantize_rows(Q5_1, x)[0]
    assert b.tolist() == [0x00, 0x00, 0x80, 0x42] + [0] * 20
    assert np.all(orc.dequantize_rows(Q5_1, b[None], 32) == 3.25)


def _legacy_rows(rng, n):
    rows = [rng.normal(size=(n, 32)), rng.standard_t(2, size=(n, 32)) * 10, rng.uniform(3, 9, size=(n, 32)),
            rng.normal(size=(n, 32)) * 1e-4 - 50.0]
    return np.concatenate(rows).astype(np.float32)


@pytest.mark.parametrize("name", list(LEGACY))
def test_legacy_codes_are_the_rounded_quotients(orc, name):
    """Codes stored = clamp(round_half_even((x - m16) / d16)) computed by numpy
    in fp32 from the stored scale and minimum (R17/R18)."""
    t = LEGACY[name]
    x = _legacy_rows(np.random.default_rng(21), 500)
    d, m, u = _parse_legacy(t, orc.quantize_rows(t, x))
    d32, m32 = d.astype(np.float32)[:, None], m.astype(np.float32)[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        if t == Q5_0:
            q = np.rint(x / d32)
            ref = np.where(d32 == 0, 16, np.clip(q, -16, 15) + 16)
        else:
            q = np.rint((x - m32) / d32)
            ref = np.where(d32 == 0, 0, np.clip(q, 0, 15 if t == Q4_1 else 31))
    assert np.array_equal(u, ref.astype(np.int64))
    # and the scales: symmetric amax / 15, affine (max - min) / qmax and min, as binary16
    if t == Q5_0:
        assert np.array_equal(d.astype(np.float16), (np.abs(x).max(1) / np.float32(15)).astype(np.float16))
    else:
        qmax = np.float32(15 if t == Q4_1 else 31)
        assert np.array_equal(d.astype(np.float16), ((x.max(1) - x.min(1)) / qmax).astype(np.float16))
        assert np.array_equal(m.astype(np.float16), x.min(1).astype(np.float16))


@pytest.mark.parametrize("name", list(LEGACY))
def test_legacy_round_trip_bound(orc, name):
    t = LEGACY[name]
    x = _legacy_rows(np.random.default_rng(22), 800)
    blocks = orc.quantize_rows(t, x)
    xh = orc.dequantize_rows(t, blocks, 32).astype(np.float64)
    d, m, _ = _parse_legacy(t, blocks)
    xd = x.astype(np.float64)
    ulp = 4 * np.abs(xd).max(1) * 2.0 ** -23
    if t == Q5_0:
        bound = d / 2 * (1 + 2.0 ** -18) + ulp
    else:
        qmax = 15 if t == Q4_1 else 31
        dt, mt = (xd.max(1) - xd.min(1)) / qmax, xd.min(1)
        bound = d / 2 * (1 + 2.0 ** -18) + qmax * np.abs(d - dt) + np.abs(m - mt) + ulp
    assert np.all(np.abs(xh - xd) <= bound[:, None])


@pytest.mark.parametrize("name", list(LEGACY))
def test_legacy_gemv_is_the_brute_force_product(orc, name):
    """R19: y = sum over blocks of (d_w u + m_w) . (d_x qx), in fp64 from the
    test's own parse of both operands."""
    t = LEGACY[name]
    rng = np.random.default_rng(23)
    M, K = 7, 160
    W = (rng.normal(size=(M, K)) + rng.uniform(-1, 1, size=(M, 1))).astype(np.float32)
    x = rng.normal(size=K).astype(np.float32)
    wb = orc.quantize_rows(t, W)
    y, mag = orc.gemv(t, wb, x, M, K, with_mag=True)
    dw, mw, uw = _parse_legacy(t, wb)
    xq = orc.quantize_rows(Q8, x[None])[0].reshape(-1, 34)
    dx = xq[:, 0:2].copy().view(np.float16).astype(np.float64)[:, 0]
    qx = xq[:, 2:].view(np.int8).astype(np.float64)
    vw = (dw[:, None] * (uw - (16 if t == Q5_0 else 0)) + mw[:, None]).reshape(M, K // 32, 32)
    vx = (dx[:, None] * qx)[None]
    ref = (vw * vx).sum(axis=(1, 2))
    assert np.allclose(y.astype(np.float64), ref, rtol=1e-6, atol=1e-9 * mag.max())


@pytest.mark.parametrize("name", list(LEGACY))
def test_legacy_kv_write_is_the_row_quantizer(orc, name):
    t = LEGACY[name]
    rng = np.random.default_rng(24)
    T, NKV, D = 9, 3, 64
    K = rng.normal(size=(T, NKV, D)).astype(np.float32)
    assert np.array_equal(orc.kv_quantize(t, K, None, T, NKV, D).reshape(-1),
                          orc.quantize_rows(t, K.reshape(-1, D)).reshape(-1))
    with pytest.raises(ValueError):
        orc.kv_quantize(t, K, np.zeros((NKV, D), np.float32), T, NKV, D)  # bias: Q4_0 only


# ------------------------------------------------ k-quants ([KQ], R20-R24) --

Q4_K, Q6_K = 12, 14


def _parse_q4k(blocks):
    """The test's own reading of R20: d, dmin, sc[8], mn[8], u[256] per super-block."""
    b = np.asarray(blocks, np.uint8).reshape(-1, 144)
    d = b[:, 0:2].copy().view(np.float16).astype(np.float32)[:, 0]
    dm = b[:, 2:4].copy().view(np.float16).astype(np.float32)[:, 0]
    bits = np.unpackbits(b[:, 4:16], axis=1, bitorder="little")  # 96 bits, value k at 6k..6k+5
    vals = (bits.reshape(-1, 16, 6) * (1 << np.arange(6))).sum(axis=2)
    nib = b[:, 16:].reshape(-1, 8, 16).astype(np.int64)
    u = np.concatenate([nib & 15, nib >> 4], axis=2).reshape(-1, 256)
    return d, dm, vals[:, :8], vals[:, 8:], u


def _parse_q6k(blocks):
    """The test's own reading of R22: d, sc[16] (int8), u[256] (0..63)."""
    b = np.asarray(blocks, np.uint8).reshape(-1, 210)
    ql, qh = b[:, :128].astype(np.int64), b[:, 128:192].astype(np.int64)
    lo = np.concatenate([ql & 15, ql >> 4], axis=1)
    hi = np.concatenate([(qh >> (2 * k)) & 3 for k in range(4)], axis=1)
    sc = b[:, 192:208].view(np.int8).astype(np.int64)
    d = b[:, 208:210].copy().view(np.float16).astype(np.float32)[:, 0]
    return d, sc, lo | (hi << 4)


def test_kquant_sizes(orc):
    s = golden.sizes()
    # Q4_K: 256 4-bit codes + 8 sub-blocks x (6-bit scale + 6-bit minimum) + two fp16 super-scales
    assert orc.block_bytes(Q4_K) == 256 * 4 // 8 + 8 * 12 // 8 + 4 == 144 and orc.block_values(Q4_K) == 256
    # Q6_K: 210 bytes per 256 is the layout whose size ratio to Q8_0 matches the pages'
    # Llama-3-8B file sizes; 8 sub-blocks with 6-bit scales (200 bytes) would not
    ratio = s["llama3_8b_q6_k_gib"] / s["llama3_8b_q8_0_gib"]
    bpw = lambda t: orc.block_bytes(t) * 8 / orc.block_values(t)
    assert abs(bpw(Q6_K) / bpw(Q8) - ratio) < 0.005 * ratio
    assert abs((200 * 8 / 256) / bpw(Q8) - ratio) > 0.03 * ratio


@pytest.mark.parametrize("t", [Q4_K, Q6_K])
def test_kquant_values_from_an_independent_parse(orc, t):
    rng = np.random.default_rng(40 + t)
    x = np.concatenate([rng.normal(size=(20, 512)), rng.standard_t(3, size=(20, 512)) * 5,
                        rng.uniform(0.5, 3.0, size=(20, 512))]).astype(np.float32)
    q = orc.quantize_rows(t, x)
    deq = orc.dequantize_rows(t, q, 512).reshape(-1, 256)
    if t == Q4_K:
        d, dm, sc, mn, u = _parse_q4k(q)
        S = (d[:, None] * sc.astype(np.float32)).astype(np.float32)
        M = (dm[:, None] * mn.astype(np.float32)).astype(np.float32)
        ref = np.repeat(S, 32, axis=1) * u.astype(np.float32) - np.repeat(M, 32, axis=1)
        assert sc.max() <= 63 and mn.max() <= 63
    else:
        d, sc, u = _parse_q6k(q)
        S = (d[:, None] * sc.astype(np.float32)).astype(np.float32)
        ref = np.repeat(S, 16, axis=1) * (u - 32).astype(np.float32)
    assert np.array_equal(deq.view(np.uint32), ref.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("case", golden.kquant_worked(), ids=lambda c: c[0])
def test_kquant_hand_worked_factors(orc, case):
    """Super-scales and sub-block factors of hand-worked super-blocks
    (tests/golden/kquant_worked.txt): the super-scale maps the largest
    sub-block factor to the top of its 6-bit (Q4_K) or signed 8-bit (Q6_K)
    range, every other factor rounds half to even, and a code below the
    range's floor clamps to it."""
    name, tname, vals, exp = case
    t = {"Q4_K": Q4_K, "Q6_K": Q6_K}[tname]
    x = np.zeros((1, 256), np.float32)
    for i, v in vals.items():
        x[0, i] = v
    q = orc.quantize_rows(t, x)
    if t == Q4_K:
        d, dm, sc, mn, u = _parse_q4k(q)
        assert d[0] == exp["d"] and dm[0] == exp["dmin"]
        assert sc[0].tolist() == exp["sc"] and mn[0].tolist() == exp["mn"]
    else:
        d, sc, u = _parse_q6k(q)
        assert d[0] == exp["d"]
        if "sc" in exp:
            assert sc[0].tolist() == exp["sc"]
        if "sc0" in exp:
            assert sc[0][0] == exp["sc0"] and sc[0][15] == exp["sc15"]
            assert u[0][0] == exp["u0"] and u[0][240] == exp["u240"]


@pytest.mark.parametrize("t", [Q4_K, Q6_K])
def test_kquant_codes_are_nearest_under_the_stored_factors(orc, t):
    """Each code is the nearest one to its value under the factors the
    super-block stores (d * sc, dmin * mn), as a block quantizer's code is the
    rounded quotient by the stored scale: the quotient lies within half a step
    of the code, or beyond the end of the range the code clamps to."""
    rng = np.random.default_rng(70 + t)
    x = np.concatenate([rng.normal(size=(30, 256)), rng.standard_t(3, size=(30, 256)) * 3,
                        rng.uniform(0.2, 4.0, size=(30, 256))]).astype(np.float32)
    q = orc.quantize_rows(t, x)
    slop = 1e-5
    if t == Q4_K:
        d, dm, sc, mn, u = _parse_q4k(q)
        S = np.repeat((d[:, None] * sc.astype(np.float32)).astype(np.float32), 32, axis=1).astype(np.float64)
        M = np.repeat((dm[:, None] * mn.astype(np.float32)).astype(np.float32), 32, axis=1).astype(np.float64)
        live = S > 0
        r = np.where(live, (x + M) / np.where(live, S, 1.0), 0.0)
        c, lo, hi = u.astype(np.float64), 0, 15
    else:
        d, sc, u = _parse_q6k(q)
        S = np.repeat((d[:, None] * sc.astype(np.float32)).astype(np.float32), 16, axis=1).astype(np.float64)
        live = S != 0
        r = np.where(live, x / np.where(live, S, 1.0), 0.0)
        c, lo, hi = (u - 32).astype(np.float64), -32, 31
    inner = (c > lo) & (c < hi)
    assert np.all(np.abs(r - c)[inner] <= 0.5 + slop)
    assert np.all(r[c == lo] <= lo + 0.5 + slop) and np.all(r[c == hi] >= hi - 0.5 - slop)


@pytest.mark.parametrize("t", [Q4_K, Q6_K])
def test_kquant_round_trip_bound(orc, t):
    """Half a sub-block step, plus what quantizing the sub-block factors to
    6 (Q4_K) or 8 (Q6_K) bits against fp16 super-scales can cost."""
    rng = np.random.default_rng(50 + t)
    x = np.concatenate([rng.normal(size=(40, 256)), rng.standard_t(2, size=(40, 256)),
                        rng.normal(size=(40, 256)) * 0.01 + 2.0]).astype(np.float32)
    q = orc.quantize_rows(t, x)
    err = np.abs(orc.dequantize_rows(t, q, 256).astype(np.float64) - x)
    ulp = 4 * np.abs(x).max(1, keepdims=True) * 2.0 ** -23
    if t == Q4_K:
        d, dm, sc, mn, u = _parse_q4k(q)
        S = np.repeat(d[:, None].astype(np.float64) * sc, 32, axis=1)
        bound = S / 2 + 15 * np.repeat(d[:, None], 256, 1) / 2 * 1.001 + np.repeat(dm[:, None], 256, 1) / 2 * 1.001
    else:
        d, sc, u = _parse_q6k(q)
        S = np.repeat(d[:, None].astype(np.float64) * sc, 16, axis=1)
        bound = S / 2 + 31 * np.repeat(d[:, None], 256, 1) / 2 * 1.001
    assert np.all(err <= bound + ulp)


@pytest.mark.parametrize("t", [Q4_K, Q6_K])
def test_kquant_gemv_is_the_brute_force_product(orc, t):
    rng = np.random.default_rng(60 + t)
    M, K = 5, 768
    W = (rng.normal(size=(M, K)) * 0.02).astype(np.float32)
    x = rng.normal(size=K).astype(np.float32)
    wb = orc.quantize_rows(t, W)
    y, mag = orc.gemv(t, wb, x, M, K, with_mag=True)
    if t == Q4_K:
        d, dm, sc, mn, u = _parse_q4k(wb)
        S = (d[:, None] * sc.astype(np.float32)).astype(np.float64)
        Mn = (dm[:, None] * mn.astype(np.float32)).astype(np.float64)
        vw = np.repeat(S, 32, axis=1) * u - np.repeat(Mn, 32, axis=1)
    else:
        d, sc, u = _parse_q6k(wb)
        S = (d[:, None] * sc.astype(np.float32)).astype(np.float64)
        vw = np.repeat(S, 16, axis=1) * (u - 32)
    xq = orc.quantize_rows(Q8, x[None])[0].reshape(-1, 34)
    vx = (xq[:, 0:2].copy().view(np.float16).astype(np.float64) * xq[:, 2:].view(np.int8)).reshape(-1)
    ref = vw.reshape(M, K) @ vx
    assert np.allclose(y.astype(np.float64), ref, rtol=1e-6, atol=1e-9 * mag.max())
    with pytest.raises(ValueError):
        orc.gemv(t, wb, x[:640], M, 640)  # a row must hold whole super-blocks
