"""The C-ABI library loads, exports every symbol include/bq.h declares, and
rejects bad arguments on the host (no GPU needed: none of these calls reaches
a CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, SHAPE, UNSUPPORTED, ALIGN, CUDA, TIMEOUT, WORKSPACE = 0, -1, -2, -3, -4, -5, -6, -7
Q4, Q8 = 2, 8
FAKE = 0x7f0000000000  # a 256-byte aligned, never dereferenced address


def declared_functions():
    hdr = open(os.path.join(ROOT, "include", "bq.h"), encoding="utf-8").read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(bq_[a-z_0-9]+)\s*\(", hdr)))


@pytest.fixture(scope="module")
def L():
    from block_quantized_weight_row_gb300 import binding
    if not os.path.exists(binding.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return binding.lib()


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n


def test_abi_signatures_use_no_torch_types():
    hdr = open(os.path.join(ROOT, "include", "bq.h"), encoding="utf-8").read()
    assert "torch" not in hdr.lower().replace("no torch", "")
    assert "at::" not in hdr and "Tensor" not in hdr


def test_block_bytes_and_version(L):
    assert L.bq_block_bytes(Q4) == 18
    assert L.bq_block_bytes(Q8) == 34
    assert L.bq_block_bytes(5) == 0
    assert L.bq_version() >= 1


def test_workspace_size(L):
    # K a multiple of 256: binary16 codes of 128-token tiles plus one fp32 scale per block and token
    assert L.bq_workspace_size(Q8, 4096, 512, 4096) == 4 * 128 * 4096 * 2 + 4 * 128 * 128 * 4
    assert L.bq_workspace_size(Q8, 4096, 129, 256) == 2 * 128 * 256 * 2 + 2 * 8 * 128 * 4
    # other K: Q8_0 blocks of the N rows
    assert L.bq_workspace_size(Q8, 4096, 512, 4128) == 512 * 129 * 34
    assert L.bq_workspace_size(Q8, 1, 3, 96) == 512  # 3 x 3 x 34 = 306, rounded up to 256 bytes
    assert L.bq_workspace_size(Q4, 1, 3, 96) == 0
    assert L.bq_workspace_size(Q8, 1, 0, 96) == 0


def _err(L):
    return L.bq_last_error().decode()


def test_unknown_type_is_unsupported(L):
    assert L.bq_quantize_rows(4, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + 4096), 1, 32) == UNSUPPORTED
    assert "unknown type" in _err(L)
    assert L.bq_gemv(5, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1, 32) == UNSUPPORTED
    assert L.bq_kv_quantize(0, ctypes.c_void_p(FAKE), None, ctypes.c_void_p(FAKE + 4096), 1, 1, 32) == UNSUPPORTED
    assert L.bq_block_dots(1, ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 1, 32) == UNSUPPORTED


def test_legacy_types_where_they_are_not_taken(L):
    """Q4_1 (3), Q5_0 (6), Q5_1 (7) have block sizes and go through the row
    quantizer, the GEMV and the KV write; the other entry points refuse them."""
    p = ctypes.c_void_p
    assert [L.bq_block_bytes(t) for t in (3, 6, 7)] == [20, 22, 24]
    for t in (3, 6, 7):
        assert L.bq_block_dots(t, p(FAKE), p(FAKE), p(FAKE), 1, 32) == UNSUPPORTED
        assert L.bq_gemm(t, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4, 64) == UNSUPPORTED
        assert L.bq_gemv_workspace_size(t, 4096) == L.bq_gemv_workspace_size(2, 4096) > 0  # x records, as Q4_0
        # K % 256 != 0 (generic kernel): 32 code bytes, scale and code sum per block of x
        assert L.bq_gemv_workspace_size(t, 4128) == (129 * 40 + 255) // 256 * 256
        assert L.bq_gemv_workspace_size(t, 4100) == 0
        assert L.bq_kv_quantize(t, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 2, 2, 64) == UNSUPPORTED  # bias
        assert L.bq_kv_quantize_basis(t, p(FAKE), None, 1, 1, p(FAKE + (2 << 20)), 2, 2, 64) == UNSUPPORTED  # rotation
        assert L.bq_attn_decode(t, 8, p(FAKE), p(FAKE), p(FAKE), p(FAKE + (1 << 24)), 10, 8, 8, 64,
                                ctypes.c_float(0.1)) == UNSUPPORTED
        assert L.bq_quantize_rows(t, p(FAKE), p(FAKE + 4096), 2, 33) == SHAPE  # taken: a shape error, not a type error


def test_row_length_must_be_multiple_of_32(L):
    p = ctypes.c_void_p
    assert L.bq_quantize_rows(Q4, p(FAKE), p(FAKE + (1 << 20)), 2, 33) == SHAPE
    assert L.bq_dequantize_rows(Q8, p(FAKE), p(FAKE + (1 << 20)), 2, 48) == SHAPE
    assert L.bq_gemv(Q4, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 100) == SHAPE
    assert L.bq_gemm(Q8, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4, 100) == SHAPE
    assert L.bq_kv_quantize(Q4, p(FAKE), None, p(FAKE + (1 << 20)), 2, 2, 40) == SHAPE


def test_gemv_k_limit(L):
    p = ctypes.c_void_p
    assert L.bq_gemv(Q4, p(FAKE), p(FAKE + (1 << 30)), p(FAKE + (2 << 30)), 1, 65536 + 32) == SHAPE


def test_null_pointers_and_negative_sizes(L):
    p = ctypes.c_void_p
    assert L.bq_quantize_rows(Q4, None, p(FAKE), 1, 32) == INVALID
    assert L.bq_quantize_rows(Q4, p(FAKE), None, 1, 32) == INVALID
    assert L.bq_quantize_rows(Q4, p(FAKE), p(FAKE + 4096), -1, 32) == INVALID
    assert L.bq_gemv(Q4, None, p(FAKE), p(FAKE + 4096), 1, 32) == INVALID
    assert L.bq_gemm(Q8, p(FAKE), None, p(FAKE + 4096), 1, 1, 32) == INVALID
    assert L.bq_kv_quantize(Q4, None, None, p(FAKE), 1, 1, 32) == INVALID


def test_alignment(L):
    p = ctypes.c_void_p
    assert L.bq_quantize_rows(Q4, p(FAKE + 4), p(FAKE + 4096), 1, 32) == ALIGN
    assert L.bq_quantize_rows(Q4, p(FAKE), p(FAKE + 4098), 1, 32) == ALIGN
    assert L.bq_gemv(Q4, p(FAKE + 2), p(FAKE + 4096), p(FAKE + 8192), 1, 32) == ALIGN
    assert L.bq_gemv(Q4, p(FAKE), p(FAKE + 4100), p(FAKE + 8192), 1, 32) == ALIGN
    assert L.bq_kv_quantize(Q4, p(FAKE), p(FAKE + 8), p(FAKE + 8192), 1, 1, 32) == ALIGN


def test_aliasing_rejected(L):
    p = ctypes.c_void_p
    # dst inside src
    assert L.bq_quantize_rows(Q4, p(FAKE), p(FAKE + 64), 1, 64) == INVALID
    # y overlapping x
    assert L.bq_gemv(Q4, p(FAKE), p(FAKE + 4096), p(FAKE + 4096), 4, 32) == INVALID


def test_mean_centering_bias_requires_q4_0(L):
    p = ctypes.c_void_p
    rc = L.bq_kv_quantize(Q8, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 2, 64)
    assert rc == UNSUPPORTED
    assert "Q4_0" in _err(L)


def test_gemm_takes_q8_0_only_and_needs_workspace(L):
    p = ctypes.c_void_p
    assert L.bq_gemm(Q4, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4, 64) == UNSUPPORTED
    assert L.bq_set_workspace(None, 0) == OK
    assert L.bq_gemm(Q8, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4, 64) == WORKSPACE
    assert "workspace" in _err(L)
    assert L.bq_set_workspace(p(FAKE + 8), 1024) == ALIGN
    assert L.bq_set_workspace(p(FAKE), 0) == INVALID


def test_empty_calls_are_noops(L):
    p = ctypes.c_void_p
    assert L.bq_quantize_rows(Q4, None, None, 0, 32) == OK
    assert L.bq_quantize_rows(Q8, None, None, 5, 0) == OK
    assert L.bq_gemv(Q4, None, None, None, 0, 4096) == OK
    assert L.bq_gemm(Q8, None, None, None, 0, 512, 4096) == OK
    assert L.bq_kv_quantize(Q4, None, None, None, 0, 8, 128) == OK
    assert L.bq_block_dots(Q4, None, None, None, 0, 64) == OK
    assert L.bq_dequantize_rows(Q4, None, None, 0, 64) == OK
    assert _err(L) == "no error"
    del p


def test_stream_is_thread_local(L):
    import threading
    assert L.bq_set_stream(ctypes.c_void_p(0x1234)) == OK
    seen = {}

    def other():
        seen["s"] = L.bq_get_stream()

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert L.bq_get_stream() == 0x1234
    assert seen["s"] is None
    assert L.bq_set_stream(None) == OK


def test_binding_refuses_cpu_tensors():
    import torch
    import block_quantized_weight_row_gb300 as bq
    with pytest.raises(TypeError):
        bq.quantize_rows(bq.Q4_0, torch.zeros(2, 32))
    with pytest.raises(TypeError):
        bq.gemv(bq.Q4_0, torch.zeros(18, dtype=torch.uint8), torch.zeros(32), 1, 32)


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "block_quantized_weight_row_gb300")
    for dirpath, _dirs, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "bq_oracle" not in src, f


def _seq(L, n_mats, W, Y, M, X, K, t=8):
    """bq_gemv_sequence with integer stand-ins for device pointers (the calls
    below fail validation, or find no workspace, before any device work)."""
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    g = len(n_mats)
    return L.bq_gemv_sequence(t, g, (ctypes.c_int * g)(*n_mats), (vp * len(W))(*W), (vp * len(Y))(*Y),
                              (i64 * len(M))(*M), (vp * g)(*X), (i64 * g)(*K))


def test_gemv_sequence_validation(L):
    assert L.bq_set_workspace(None, 0) == 0
    base = 1 << 32
    W0, W1 = base, base + (1 << 24)
    Y0, Y1 = base + (2 << 24), base + (3 << 24)
    X0, X1 = base + (4 << 24), base + (5 << 24)
    ok = dict(n_mats=[1, 1], W=[W0, W1], Y=[Y0, Y1], M=[64, 64], X=[X0, X1], K=[512, 512])
    assert L.bq_gemv_sequence_workspace_size() >= 4 * 257  # abort flag + one counter per batch of a launch
    assert L.bq_gemv_sequence(8, 0, None, None, None, None, None, None) == 0
    assert _seq(L, **ok) == -7                               # valid, but no workspace set
    assert _seq(L, **{**ok, "K": [512, 96]}) == -2           # K not a multiple of 256
    assert _seq(L, **{**ok, "K": [512, 32768]}) == -2        # above BQ_GEMV_SEQ_MAX_K
    assert _seq(L, **{**ok, "M": [64, -1]}) == -1
    assert _seq(L, **{**ok, "n_mats": [1, -1]}) == -1
    assert _seq(L, **ok, t=5) == -3
    assert _seq(L, **{**ok, "W": [W0 + 8, W1]}) == -4        # W not 16-byte aligned
    assert _seq(L, **{**ok, "X": [X0 + 4, X1]}) == -4
    assert _seq(L, **{**ok, "Y": [Y0 + 2, Y1]}) == -4
    assert _seq(L, **{**ok, "Y": [Y0, Y0 + 128]}) == -1      # two outputs overlap
    assert _seq(L, **{**ok, "Y": [Y0, W1 + 64]}) == -1       # an output overlaps a weight matrix
    assert _seq(L, **{**ok, "X": [Y0 + 64, X1]}) == -1       # batch 0 reads its own output
    # a later batch may read an earlier batch's output: only the workspace is missing
    assert _seq(L, **{**ok, "X": [X0, Y0]}) == -7
    assert "workspace" in L.bq_last_error().decode()


def test_attn_decode_validation(L):
    assert L.bq_set_workspace(None, 0) == 0
    base = 1 << 32
    q, K, V, o = base, base + (1 << 24), base + (2 << 24), base + (3 << 24)
    f = ctypes.c_float(0.1)
    assert L.bq_attn_decode(2, 8, q, K, V, o, 100, 16, 8, 128, f) == -7   # valid, no workspace
    assert L.bq_attn_workspace_size(2, 8, 100, 16, 8, 128) > 0
    assert L.bq_attn_decode(2, 8, q, K, V, o, 100, 12, 4, 128, f) == -3   # 3 query heads per kv head
    assert L.bq_attn_decode(2, 8, q, K, V, o, 100, 16, 8, 48, f) == -2    # head_dim not a multiple of 32
    assert L.bq_attn_decode(2, 8, q, K, V, o, 0, 16, 8, 128, f) == -2     # no tokens
    assert L.bq_attn_decode(2, 8, q, K, V, o, 100, 64, 8, 128, f) == -2   # n_heads * head_dim above 4096
    assert L.bq_attn_decode(5, 8, q, K, V, o, 100, 16, 8, 128, f) == -3
    assert L.bq_attn_decode(2, 8, q + 4, K, V, o, 100, 16, 8, 128, f) == -4
    assert L.bq_attn_decode(2, 8, q, K, V, q + 256, 100, 16, 8, 128, f) == -1  # o overlaps q
    assert L.bq_attn_decode(2, 8, None, K, V, o, 100, 16, 8, 128, f) == -1


def test_rotated_kv_and_bias_validation(L):
    """The basis arguments are checked on the host before anything runs; a
    bias from another basis fails fast with BQ_ERR_BASIS (-8)."""
    base = 1 << 32
    K, bias, dst = base, base + (1 << 24), base + (2 << 24)
    # kv write
    assert L.bq_kv_quantize_basis(2, K, bias, 0, 1, dst, 10, 2, 128) == -8   # plain bias, rotated cache
    assert L.bq_kv_quantize_basis(2, K, bias, 1, 0, dst, 10, 2, 128) == -8   # rotated bias, plain cache
    assert L.bq_kv_quantize_basis(2, K, None, 0, 1, dst, 10, 2, 96) == -2    # rotation needs head_dim % 64
    assert L.bq_kv_quantize_basis(2, K, None, 0, 2, dst, 10, 2, 128) == -3   # unknown basis
    assert L.bq_kv_quantize_basis(8, K, bias, 1, 1, dst, 10, 2, 128) == -3   # bias with Q8_0
    assert L.bq_kv_quantize_basis(8, K, None, 0, 1, dst, 0, 2, 128) == 0     # empty: a no-op
    assert L.bq_kv_quantize_basis(2, K + 4, None, 0, 1, dst, 10, 2, 128) == -4
    # calibration
    assert L.bq_kv_bias(K, 2, bias, 10, 2, 128) == -3
    assert L.bq_kv_bias(K, 1, bias, 10, 2, 96) == -2
    assert L.bq_kv_bias(K, 0, bias, 10, 2, 48) == -2
    assert L.bq_kv_bias(K, 0, bias, 0, 2, 128) == -1                          # no calibration tokens
    assert L.bq_kv_bias(None, 0, bias, 10, 2, 128) == -1
    assert L.bq_kv_bias(K + 4, 0, bias, 10, 2, 128) == -4
    assert L.bq_kv_bias(K, 0, K + 1024, 10, 2, 128) == -1                     # bias inside the rows
    # attention over a rotated cache
    assert L.bq_set_workspace(None, 0) == 0
    q, o, V = base + (3 << 24), base + (4 << 24), base + (5 << 24)
    f = ctypes.c_float(0.1)
    assert L.bq_attn_decode_basis(2, 8, 1, q, K, V, o, 100, 16, 8, 128, f) == -7  # valid, no workspace
    assert L.bq_attn_decode_basis(2, 8, 1, q, K, V, o, 100, 8, 8, 96, f) == -2    # rotated, head_dim 96
    assert L.bq_attn_decode_basis(2, 8, 3, q, K, V, o, 100, 16, 8, 128, f) == -3  # unknown basis


def test_layer_kv_write_validation(L):
    """bq_kv_write checks both tensors' types, the K basis and bias, sizes,
    alignment and every overlap on the host, before anything runs."""
    base = 1 << 32
    K, V, bias = base, base + (1 << 26), base + (2 << 26)
    kd, vd = base + (3 << 26), base + (4 << 26)
    n = (10, 2, 128)
    assert L.bq_kv_write(2, K, bias, 1, 0, kd, 8, V, vd, *n) == -8     # bias basis differs from the cache's
    assert L.bq_kv_write(8, K, bias, 0, 0, kd, 8, V, vd, *n) == -3     # bias with a Q8_0 K
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 3, V, vd, *n) == -3     # legacy V type
    assert L.bq_kv_write(12, K, None, 0, 0, kd, 8, V, vd, *n) == -3    # k-quant K type
    assert L.bq_kv_write(2, K, None, 0, 2, kd, 8, V, vd, *n) == -3     # unknown basis
    assert L.bq_kv_write(2, K, None, 0, 1, kd, 8, V, vd, 10, 2, 96) == -2   # rotation needs head_dim % 64
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, vd, 10, 2, 48) == -2   # head_dim % 32
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, vd, -1, 2, 128) == -1
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, None, vd, *n) == -1
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V + 4, vd, *n) == -4
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, vd + 8, *n) == -4
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, V + 1024, *n) == -1       # V output inside V's rows
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, K + 4096, *n) == -1       # V output inside K's rows
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, kd + 16, *n) == -1        # the outputs overlap
    assert L.bq_kv_write(2, K, bias, 0, 0, bias - 16, 8, V, vd, *n) == -1      # K output over the bias
    assert L.bq_kv_write(2, K, None, 0, 0, kd, 8, V, vd, 0, 2, 128) == 0       # empty: a no-op


def test_kquants_where_they_are_taken(L):
    """Q4_K (12) and Q6_K (14): super-blocks of 256 values; rows must hold
    whole super-blocks; only the row quantizer, dequantizer and GEMV take them."""
    p = ctypes.c_void_p
    assert [L.bq_block_bytes(t) for t in (12, 14)] == [144, 210]
    assert [L.bq_block_values(t) for t in (12, 14, 2, 3)] == [256, 256, 32, 32]
    assert L.bq_block_values(99) == 0
    for t in (12, 14):
        assert L.bq_quantize_rows(t, p(FAKE), p(FAKE + (1 << 20)), 2, 96) == SHAPE
        assert L.bq_dequantize_rows(t, p(FAKE), p(FAKE + (1 << 20)), 2, 288) == SHAPE
        assert L.bq_gemv(t, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4128) == SHAPE
        assert L.bq_kv_quantize(t, p(FAKE), None, p(FAKE + (2 << 20)), 2, 2, 256) == UNSUPPORTED
        assert L.bq_block_dots(t, p(FAKE), p(FAKE), p(FAKE), 1, 256) == UNSUPPORTED
        assert L.bq_gemm(t, p(FAKE), p(FAKE + (1 << 20)), p(FAKE + (2 << 20)), 4, 4, 256) == UNSUPPORTED
