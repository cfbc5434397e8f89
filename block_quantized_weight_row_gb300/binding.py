"""Thin Python binding over libbq.so (the C ABI in include/bq.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Tensors must be CUDA tensors; the binding passes their device
pointers, the torch current stream and a torch-allocated workspace to the
library, and raises BQError on a nonzero status. There is no CPU fallback: if
libbq.so is missing or fails to load, every call raises.
"""
import ctypes
import os

import torch

Q4_0 = 2
Q8_0 = 8
Q4_1, Q5_0, Q5_1 = 3, 6, 7
Q4_K, Q6_K = 12, 14
QK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libbq.so"

_STATUS = {0: "BQ_OK", -1: "BQ_ERR_INVALID_ARG", -2: "BQ_ERR_SHAPE", -3: "BQ_ERR_UNSUPPORTED",
           -4: "BQ_ERR_ALIGN", -5: "BQ_ERR_CUDA", -6: "BQ_ERR_TIMEOUT", -7: "BQ_ERR_WORKSPACE",
           -8: "BQ_ERR_BASIS"}
BASIS_PLAIN, BASIS_HADAMARD64 = 0, 1


class BQError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


_lib = None
_ws = {}  # device index -> torch.uint8 workspace tensor


def lib():
    """Load libbq.so (built in-tree by build.py); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} is not built; run __graft_entry__.build() "
                          "(the CUDA path has no fallback)")
    L = ctypes.CDLL(path)
    i, i64, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "bq_quantize_rows": ([i, vp, vp, i64, i64], i),
        "bq_dequantize_rows": ([i, vp, vp, i64, i64], i),
        "bq_gemv": ([i, vp, vp, vp, i64, i64], i),
        "bq_gemv_multi": ([i, i, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64), vp, i64], i),
        "bq_gemv_sequence": ([i, i, ctypes.POINTER(i), ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(i64),
                              ctypes.POINTER(vp), ctypes.POINTER(i64)], i),
        "bq_gemv_sequence_workspace_size": ([], sz),
        "bq_attn_decode": ([i, i, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float], i),
        "bq_attn_decode_basis": ([i, i, i, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float], i),
        "bq_kv_quantize_basis": ([i, vp, vp, i, i, vp, i64, i64, i64], i),
        "bq_kv_bias": ([vp, i, vp, i64, i64, i64], i),
        "bq_attn_workspace_size": ([i, i, i64, i64, i64, i64], sz),
        "bq_gemm": ([i, vp, vp, vp, i64, i64, i64], i),
        "bq_kv_quantize": ([i, vp, vp, vp, i64, i64, i64], i),
        "bq_kv_write": ([i, vp, vp, i, i, vp, i, vp, vp, i64, i64, i64], i),
        "bq_block_dots": ([i, vp, vp, vp, i64, i64], i),
        "bq_set_stream": ([vp], i),
        "bq_get_stream": ([], vp),
        "bq_set_workspace": ([vp, sz], i),
        "bq_workspace_size": ([i, i64, i64, i64], sz),
        "bq_gemv_workspace_size": ([i, i64], sz),
        "bq_last_error": ([], ctypes.c_char_p),
        "bq_block_bytes": ([i], i),
        "bq_block_values": ([i], i),
        "bq_device_status": ([], i),
        "bq_version": ([], i),
        "bq_set_spin_limit": ([i64], i),
        "bq_set_weight_prefetch": ([i], i),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes, f.restype = args, res
    _lib = L
    return L


def _check(status: int, what: str):
    if status != 0:
        msg = lib().bq_last_error()
        raise BQError(status, f"{what}: {msg.decode() if msg else ''}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _prep(device):
    """Point the library at torch's current stream on `device`."""
    L = lib()
    s = torch.cuda.current_stream(device)
    _check(L.bq_set_stream(ctypes.c_void_p(s.cuda_stream)), "bq_set_stream")
    return L


def clear_workspace() -> None:
    """Detach the calling thread's workspace (GEMVs then quantize x in-kernel)."""
    _check(lib().bq_set_workspace(None, 0), "bq_set_workspace")


def _workspace(device, nbytes: int):
    """Grow (never shrink) a torch-owned workspace and hand it to the library."""
    idx = torch.device(device).index or 0
    ws = _ws.get(idx)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws[idx] = ws
    _check(lib().bq_set_workspace(_ptr(ws), ws.numel()), "bq_set_workspace")
    return ws


def _cuda(t, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def block_bytes(t: int) -> int:
    return int(lib().bq_block_bytes(t))


def block_values(t: int) -> int:
    return int(lib().bq_block_values(t))


def quantize_rows(t: int, src: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 (rows, cols) -> uint8 (rows, cols/32*block_bytes)."""
    _cuda(src, "src")
    if src.dtype != torch.float32:
        raise TypeError("src must be float32")
    x = src.reshape(-1, src.shape[-1]) if src.dim() != 2 else src
    R, C = x.shape
    if out is None:
        out = torch.empty((R, (C // max(block_values(t), 1)) * max(block_bytes(t), 1)), dtype=torch.uint8,
                          device=src.device)
    L = _prep(src.device)
    _check(L.bq_quantize_rows(t, _ptr(x), _ptr(out), R, C), "bq_quantize_rows")
    return out


def dequantize_rows(t: int, blocks: torch.Tensor, cols: int, out: torch.Tensor | None = None) -> torch.Tensor:
    _cuda(blocks, "blocks")
    nbr = (cols // max(block_values(t), 1)) * block_bytes(t)
    R = blocks.numel() // nbr if nbr else 0
    if out is None:
        out = torch.empty((R, cols), dtype=torch.float32, device=blocks.device)
    L = _prep(blocks.device)
    _check(L.bq_dequantize_rows(t, _ptr(blocks), _ptr(out), R, cols), "bq_dequantize_rows")
    return out


def gemv(t: int, w_blocks: torch.Tensor, x: torch.Tensor, M: int, K: int,
         out: torch.Tensor | None = None) -> torch.Tensor:
    """y[M] = W (M x K, blocks of type t) . x[K] (fp32, quantized to Q8_0 in-kernel)."""
    _cuda(w_blocks, "w_blocks")
    _cuda(x, "x")
    if out is None:
        out = torch.empty(M, dtype=torch.float32, device=x.device)
    L = _prep(x.device)
    _workspace(x.device, int(L.bq_gemv_workspace_size(t, K)))
    _check(L.bq_gemv(t, _ptr(w_blocks), _ptr(x), _ptr(out), M, K), "bq_gemv")
    return out


def gemv_multi_args(w_list, y_list, M_list):
    """ctypes arrays (W pointers, y pointers, row counts) for bq_gemv_multi."""
    n = len(w_list)
    W = (ctypes.c_void_p * n)(*[w.data_ptr() for w in w_list])
    Y = (ctypes.c_void_p * n)(*[y.data_ptr() for y in y_list])
    M = (ctypes.c_int64 * n)(*M_list)
    return n, W, Y, M


def gemv_multi(t: int, w_list, x: torch.Tensor, M_list, K: int, outs=None):
    """y_i = W_i . x for matrices sharing one input x, in one launch."""
    for w in w_list:
        _cuda(w, "w_blocks")
    _cuda(x, "x")
    if outs is None:
        outs = [torch.empty(m, dtype=torch.float32, device=x.device) for m in M_list]
    n, W, Y, M = gemv_multi_args(w_list, outs, M_list)
    L = _prep(x.device)
    _workspace(x.device, int(L.bq_gemv_workspace_size(t, K)))
    _check(L.bq_gemv_multi(t, n, W, Y, M, _ptr(x), K), "bq_gemv_multi")
    return outs


def gemv_sequence_args(groups):
    """ctypes arrays for bq_gemv_sequence from batches (w_list, x, M_list, K, outs).
    Building them once and passing them to gemv_sequence_call keeps the
    per-call host work to one C call."""
    n_groups = len(groups)
    n_mats = (ctypes.c_int * n_groups)(*[len(g[0]) for g in groups])
    ws = [w for g in groups for w in g[0]]
    ys = [y for g in groups for y in g[4]]
    ms = [m for g in groups for m in g[2]]
    W = (ctypes.c_void_p * len(ws))(*[w.data_ptr() for w in ws])
    Y = (ctypes.c_void_p * len(ys))(*[y.data_ptr() for y in ys])
    M = (ctypes.c_int64 * len(ms))(*ms)
    X = (ctypes.c_void_p * n_groups)(*[g[1].data_ptr() for g in groups])
    K = (ctypes.c_int64 * n_groups)(*[g[3] for g in groups])
    return (n_groups, n_mats, W, Y, M, X, K)


def gemv_sequence_call(t: int, args, device):
    L = _prep(device)
    _workspace(device, int(L.bq_gemv_sequence_workspace_size()))
    _check(L.bq_gemv_sequence(t, *args), "bq_gemv_sequence")


def gemv_sequence(t: int, groups):
    """Batches (w_list, x, M_list, K, outs) in one launch; batch g reads its x
    after the outputs of batches 0..g-1 are written. outs may be None."""
    full = []
    for w_list, x, M_list, K, outs in groups:
        for w in w_list:
            _cuda(w, "w_blocks")
        _cuda(x, "x")
        if outs is None:
            outs = [torch.empty(m, dtype=torch.float32, device=x.device) for m in M_list]
        full.append((w_list, x, M_list, K, outs))
    if full:
        gemv_sequence_call(t, gemv_sequence_args(full), full[0][1].device)
    return [g[4] for g in full]


def attn_decode(k_type: int, v_type: int, q: torch.Tensor, K_cache: torch.Tensor, V_cache: torch.Tensor,
                n_kv_heads: int, scale: float, out: torch.Tensor | None = None,
                k_basis: int = BASIS_PLAIN) -> torch.Tensor:
    """o (n_heads, head_dim) = attention of q (n_heads, head_dim) over the
    quantized caches (n_tokens, n_kv_heads, head_dim/32 blocks as bytes);
    k_basis: the basis the K cache was written in."""
    _cuda(q, "q")
    _cuda(K_cache, "K_cache")
    _cuda(V_cache, "V_cache")
    H, D = q.shape
    T = K_cache.shape[0]
    if out is None:
        out = torch.empty((H, D), dtype=torch.float32, device=q.device)
    L = _prep(q.device)
    _workspace(q.device, int(L.bq_attn_workspace_size(k_type, v_type, T, H, n_kv_heads, D)))
    _check(L.bq_attn_decode_basis(k_type, v_type, k_basis, _ptr(q), _ptr(K_cache), _ptr(V_cache), _ptr(out), T, H,
                                  n_kv_heads, D, float(scale)), "bq_attn_decode_basis")
    return out


def gemm(t: int, w_blocks: torch.Tensor, X: torch.Tensor, M: int, N: int, K: int,
         out: torch.Tensor | None = None) -> torch.Tensor:
    """Y (N x M) = X (N x K fp32, quantized to Q8_0) . W^T (W: M x K blocks)."""
    _cuda(w_blocks, "w_blocks")
    _cuda(X, "X")
    if out is None:
        out = torch.empty((N, M), dtype=torch.float32, device=X.device)
    L = _prep(X.device)
    _workspace(X.device, int(L.bq_workspace_size(t, M, N, K)))
    _check(L.bq_gemm(t, _ptr(w_blocks), _ptr(X), _ptr(out), M, N, K), "bq_gemm")
    return out


def kv_quantize(t: int, rows: torch.Tensor, bias: torch.Tensor | None,
                out: torch.Tensor | None = None, basis: int = BASIS_PLAIN,
                bias_basis: int | None = None) -> torch.Tensor:
    """rows: (n_tokens, n_kv_heads, head_dim) fp32; bias: (n_kv_heads, head_dim) or None.
    basis: the cache's basis; bias_basis: the basis the bias was calibrated in
    (default: the cache's)."""
    _cuda(rows, "rows")
    if bias is not None:
        _cuda(bias, "bias")
    T, H, D = rows.shape
    if out is None:
        out = torch.empty((T, H, (D // QK) * max(block_bytes(t), 1)), dtype=torch.uint8, device=rows.device)
    L = _prep(rows.device)
    _check(L.bq_kv_quantize_basis(t, _ptr(rows), _ptr(bias), basis if bias_basis is None else bias_basis, basis,
                                  _ptr(out), T, H, D), "bq_kv_quantize_basis")
    return out


def kv_write(k_type: int, k_rows: torch.Tensor, bias: torch.Tensor | None, v_type: int, v_rows: torch.Tensor,
             out_k: torch.Tensor | None = None, out_v: torch.Tensor | None = None, basis: int = BASIS_PLAIN,
             bias_basis: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """One layer's K and V cache write in one launch (bq_kv_write): k_rows and
    v_rows (n_tokens, n_kv_heads, head_dim) fp32; bias (n_kv_heads, head_dim)
    or None; basis: the K cache's basis. Returns (K blocks, V blocks)."""
    _cuda(k_rows, "k_rows")
    _cuda(v_rows, "v_rows")
    if bias is not None:
        _cuda(bias, "bias")
    T, H, D = k_rows.shape
    if tuple(v_rows.shape) != (T, H, D):
        raise ValueError("k_rows and v_rows must have the same shape")
    if out_k is None:
        out_k = torch.empty((T, H, (D // QK) * max(block_bytes(k_type), 1)), dtype=torch.uint8, device=k_rows.device)
    if out_v is None:
        out_v = torch.empty((T, H, (D // QK) * max(block_bytes(v_type), 1)), dtype=torch.uint8, device=v_rows.device)
    L = _prep(k_rows.device)
    _check(L.bq_kv_write(k_type, _ptr(k_rows), _ptr(bias), basis if bias_basis is None else bias_basis, basis,
                         _ptr(out_k), v_type, _ptr(v_rows), _ptr(out_v), T, H, D), "bq_kv_write")
    return out_k, out_v


def kv_bias(rows: torch.Tensor, basis: int = BASIS_PLAIN, out: torch.Tensor | None = None) -> torch.Tensor:
    """Mean-centering bias (n_kv_heads, head_dim) fp32 of calibration rows
    (n_tokens, n_kv_heads, head_dim), measured in `basis`."""
    _cuda(rows, "rows")
    T, H, D = rows.shape
    if out is None:
        out = torch.empty((H, D), dtype=torch.float32, device=rows.device)
    L = _prep(rows.device)
    _check(L.bq_kv_bias(_ptr(rows), basis, _ptr(out), T, H, D), "bq_kv_bias")
    return out


def block_dots(t: int, w_blocks: torch.Tensor, xq_blocks: torch.Tensor, M: int, K: int) -> torch.Tensor:
    """Test export: int32 (M, K/32) per-block integer dots of W against Q8_0 blocks xq."""
    _cuda(w_blocks, "w_blocks")
    _cuda(xq_blocks, "xq_blocks")
    out = torch.empty((M, K // QK), dtype=torch.int32, device=w_blocks.device)
    L = _prep(w_blocks.device)
    _check(L.bq_block_dots(t, _ptr(w_blocks), _ptr(xq_blocks), _ptr(out), M, K), "bq_block_dots")
    return out


def set_weight_prefetch(enable: bool) -> None:
    """Let the calling thread's GEMVs stream weights before the previous
    kernel on the stream has completed (only for weights no running kernel
    writes)."""
    _check(lib().bq_set_weight_prefetch(1 if enable else 0), "bq_set_weight_prefetch")


def device_status() -> int:
    """Synchronize the current stream and return (and clear) the device error word."""
    return int(lib().bq_device_status())
