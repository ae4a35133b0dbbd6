"""Q2_K decode projections on GB300: thin Python binding of ``libq2k.so``.

Argument marshalling only: every step runs in the library's CUDA kernels,
declared in ``include/q2k.h``.  PyTorch provides device memory and the
current stream.  There is no CPU fallback: if the library is not built,
every call raises.

Functions carry the C names.  Tensors are CUDA tensors: Q2_K weights as
uint8 ``[N, K/256*84]``, q8_1 activations as uint8 ``[m, K/32*36]``, bf16
activations as ``torch.bfloat16``; outputs are fp32 unless stated.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libq2k.so")

# Every entry point include/q2k.h declares.
EXPORTS = (
    "q2k_row_bytes", "q8_1_row_bytes", "q2k_dequant_rows", "q2k_engram_hash", "q2k_engram_gate", "q8_1_quantize_rows",
    "q2k_gemv_bf16",
    "q2k_mmvq_q8_1", "q2k_mmvq_pair", "q2k_mmvq_pair_bf16", "q2k_mmvq_grouped", "q2k_mmvq_experts",
    "q3k_row_bytes", "q3k_mmvq_q8_1", "q3k_mmvq_experts",
    "swiglu_q8_1_rows",
    "q2k_moe_m1_workspace_bytes", "q2k_moe_m1", "q2k_moe_m1_static_scratch", "dense_gemm_bf16", "q2k_status_string",
    "q2k_mmq_bf16", "q2k_mmq_q8_1_workspace_bytes", "q2k_mmq_q8_1",
    "q2k_last_cuda_error", "q2k_device_error",
)

Q2K_OK = 0
Q2K_ERR_NULL_ARG = 1
Q2K_ERR_BAD_SHAPE = 2
Q2K_ERR_MISALIGNED = 3
Q2K_ERR_CUDA = 4
Q2K_ERR_UNSUPPORTED = 5
Q2K_ERR_WORKSPACE = 6

_lock = threading.Lock()
_lib = None


class Q2KError(RuntimeError):
    def __init__(self, fn: str, status: int):
        L = lib()
        msg = L.q2k_status_string(status).decode()
        if status == Q2K_ERR_CUDA:
            msg += f" (cudaError {L.q2k_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library; raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m mmvq_q2_gb300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
        sigs = {
            "q2k_row_bytes": (SZ, [I64]),
            "q8_1_row_bytes": (SZ, [I64]),
            "q2k_dequant_rows": (I32, [P, I64, I64, P, I64, P, P, P]),
            "q8_1_quantize_rows": (I32, [P, I64, I64, I64, P, P]),
            "q2k_engram_hash": (I32, [P, I64, P, I64, P, I64, I64, I64, I64, I64, P, P, P, I64, P, P, I64, P, P]),
            "q2k_engram_gate": (I32, [P, P, I64, P, I64, I64, I64, ctypes.c_float, P, P]),
            "q2k_gemv_bf16": (I32, [P, I64, I64, P, I64, I64, P, I64, P]),
            "q2k_mmvq_q8_1": (I32, [P, I64, I64, P, I64, P, I64, P]),
            "q2k_mmvq_pair": (I32, [P, I64, P, P, I64, P, I64, P, I64, P]),
            "q2k_mmvq_pair_bf16": (I32, [P, I64, P, P, I64, P, I64, P, I64, P, P]),
            "q2k_mmvq_grouped": (I32, [P, I64, I64, I64, P, I64, P, P]),
            "q2k_mmvq_experts": (I32, [P, I64, I64, I64, P, I32, P, P, P, P]),
            "q3k_row_bytes": (SZ, [I64]),
            "q3k_mmvq_q8_1": (I32, [P, I64, I64, P, I64, P, I64, P]),
            "q3k_mmvq_experts": (I32, [P, I64, I64, I64, P, I32, P, P, P, P]),
            "swiglu_q8_1_rows": (I32, [P, I64, I64, P, P, P]),
            "q2k_moe_m1_workspace_bytes": (SZ, [I64, I64, I64]),
            "q2k_moe_m1": (I32, [P, I64, I64, I64, P, P, P, P, SZ, P]),
            "q2k_moe_m1_static_scratch": (I32, [P, I64, I64, I64, P, P, P, P]),
            "dense_gemm_bf16": (I32, [P, I64, I64, I64, P, I64, P, I64, P]),
            "q2k_mmq_bf16": (I32, [P, I64, I64, P, I64, I64, P, I64, P]),
            "q2k_mmq_q8_1_workspace_bytes": (SZ, [I64, I64]),
            "q2k_mmq_q8_1": (I32, [P, I64, I64, P, I64, P, I64, P, SZ, P]),
            "q2k_status_string": (ctypes.c_char_p, [I32]),
            "q2k_last_cuda_error": (I32, []),
            "q2k_device_error": (I32, [ctypes.POINTER(ctypes.c_int32), I32]),
        }
        for name, (res, args) in sigs.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
        return L


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _call(name, *args):
    st = getattr(lib(), name)(*args)
    if st != Q2K_OK:
        raise Q2KError(name, st)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")


def q2k_row_bytes(K: int) -> int:
    return lib().q2k_row_bytes(K)


def q8_1_row_bytes(K: int) -> int:
    return lib().q8_1_row_bytes(K)


def q2k_dequant_rows(table, K, ids=None, n_rows=None, out=None, err_flag=None, stream=None):
    """Gather + dequantise Q2_K rows to bf16 ``[n_rows, K]``."""
    _need_cuda(table, ids, out, err_flag)
    n_table_rows = table.numel() // q2k_row_bytes(K)
    if n_rows is None:
        n_rows = ids.numel() if ids is not None else n_table_rows
    if out is None:
        out = torch.empty((n_rows, K), dtype=torch.bfloat16, device=table.device)
    _call("q2k_dequant_rows", _ptr(table), n_table_rows, K, _ptr(ids), n_rows, _ptr(out), _ptr(err_flag),
          _stream(stream))
    return out


def q2k_engram_hash(token_map, cache, input_ids, start_pos, max_ngram, n_layers, n_heads, multipliers, primes,
                    offsets, pad_id, layer_index=None, err_flag=None, stream=None):
    """Engram row ids of ``input_ids`` at ``start_pos`` -> (out int64
    ``[seqlen, n_layers, cols]``, layer ids int32 ``[seqlen, cols]`` or
    None); ``cache`` is updated on the device."""
    _need_cuda(token_map, cache, input_ids, multipliers, primes, offsets, err_flag)
    seqlen = input_ids.numel()
    cols = (max_ngram - 1) * n_heads
    out = torch.empty((seqlen, n_layers, cols), dtype=torch.int64, device=cache.device)
    lids = None if layer_index is None else torch.empty((seqlen, cols), dtype=torch.int32, device=cache.device)
    _call("q2k_engram_hash", _ptr(token_map), token_map.numel(), _ptr(cache), cache.numel(), _ptr(input_ids), seqlen,
          start_pos, max_ngram, n_layers, n_heads, _ptr(multipliers), _ptr(primes), _ptr(offsets), pad_id, _ptr(out),
          _ptr(lids), -1 if layer_index is None else layer_index, _ptr(err_flag), _stream(stream))
    return out, lids


def q8_1_quantize_rows(x, out=None, stream=None):
    """bf16 ``[m, K]`` (row stride allowed) -> q8_1 uint8 ``[m, K/32*36]``."""
    _need_cuda(x, out)
    m, K = x.shape
    if out is None:
        out = torch.empty((m, q8_1_row_bytes(K)), dtype=torch.uint8, device=x.device)
    _call("q8_1_quantize_rows", _ptr(x), m, K, x.stride(0), _ptr(out), _stream(stream))
    return out


def q2k_engram_gate(streams, kv, qk, eps, gates=None, stream=None):
    """Engram gate in place on fp32 ``streams [T, hc, dim]`` from fp32
    ``kv [T, >= (hc+1)*dim]`` (keys, then the shared value) and fp32
    ``qk [hc, dim]``; returns ``streams`` (and fills ``gates [T, hc]`` when
    given)."""
    _need_cuda(streams, kv, qk, gates)
    T, hc, dim = streams.shape
    if not streams.is_contiguous() or kv.stride(1) != 1 or not qk.is_contiguous():
        raise ValueError("streams and qk must be contiguous, kv rows dense")
    _call("q2k_engram_gate", _ptr(streams), _ptr(kv), kv.stride(0), _ptr(qk), T, hc, dim, float(eps), _ptr(gates),
          _stream(stream))
    return streams


def q2k_gemv_bf16(W, x, out=None, stream=None):
    """Q2_K ``[N, K]`` times bf16 ``x [m, K]`` -> fp32 ``[m, N]``."""
    _need_cuda(W, x, out)
    m, K = x.shape
    N = W.numel() // q2k_row_bytes(K)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=x.device)
    _call("q2k_gemv_bf16", _ptr(W), N, K, _ptr(x), m, x.stride(0), _ptr(out), out.stride(0), _stream(stream))
    return out


def q2k_mmvq_q8_1(W, xq, K, out=None, stream=None):
    """Q2_K ``[N, K]`` times q8_1 ``xq [m, K/32*36]`` -> fp32 ``[m, N]``."""
    _need_cuda(W, xq, out)
    m = xq.shape[0]
    N = W.numel() // q2k_row_bytes(K)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=xq.device)
    _call("q2k_mmvq_q8_1", _ptr(W), N, K, _ptr(xq), m, _ptr(out), out.stride(0), _stream(stream))
    return out


def q2k_mmvq_pair(Wa, Wb, xq, K, ya=None, yb=None, stream=None):
    """Two Q2_K matrices over one q8_1 input, one launch -> (ya, yb)."""
    _need_cuda(Wa, Wb, xq, ya, yb)
    m = xq.shape[0]
    Na = Wa.numel() // q2k_row_bytes(K)
    Nb = Wb.numel() // q2k_row_bytes(K)
    if ya is None:
        ya = torch.empty((m, Na), dtype=torch.float32, device=xq.device)
    if yb is None:
        yb = torch.empty((m, Nb), dtype=torch.float32, device=xq.device)
    _call("q2k_mmvq_pair", _ptr(Wa), Na, _ptr(ya), _ptr(Wb), Nb, _ptr(yb), K, _ptr(xq), m, _stream(stream))
    return ya, yb


def q2k_mmvq_pair_bf16(Wa, Wb, x, K, ya=None, yb=None, xq=None, stream=None):
    """The pair over bf16 rows ``x [m, K]``, with the q8_1 encoding of x in
    the same call (inside the one launch for m = 1) -> (ya, yb, xq)."""
    _need_cuda(Wa, Wb, x, ya, yb, xq)
    m = x.shape[0]
    Na = Wa.numel() // q2k_row_bytes(K)
    Nb = Wb.numel() // q2k_row_bytes(K)
    if ya is None:
        ya = torch.empty((m, Na), dtype=torch.float32, device=x.device)
    if yb is None:
        yb = torch.empty((m, Nb), dtype=torch.float32, device=x.device)
    if xq is None:
        xq = torch.empty((m, q8_1_row_bytes(K)), dtype=torch.uint8, device=x.device)
    _call("q2k_mmvq_pair_bf16", _ptr(Wa), Na, _ptr(ya), _ptr(Wb), Nb, _ptr(yb), K, _ptr(x), m, _ptr(xq),
          _stream(stream))
    return ya, yb, xq


def q2k_mmvq_grouped(W, groups, rows_per_group, K_group, xq, y=None, stream=None):
    """Block-diagonal MMVQ: group g's rows of ``W`` against group g's slice of
    each q8_1 row of ``xq`` -> fp32 ``[m, groups * rows_per_group]``."""
    _need_cuda(W, xq, y)
    m = xq.shape[0]
    if y is None:
        y = torch.empty((m, groups * rows_per_group), dtype=torch.float32, device=xq.device)
    _call("q2k_mmvq_grouped", _ptr(W), groups, rows_per_group, K_group, _ptr(xq), m, _ptr(y), _stream(stream))
    return y


def pointer_table(tensors, device=None):
    """int64 device tensor holding the device addresses of ``tensors``."""
    dev = device if device is not None else tensors[0].device
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=dev)


def q2k_mmvq_experts(W_table, N, K, xq, x_per_matrix=False, y=None, route_w=None, y_sum=None,
                     want_y=True, stream=None):
    """Batched single-token MMVQ over the matrices in ``W_table`` (int64
    device tensor of addresses); optional route-weighted ``y_sum``."""
    _need_cuda(W_table, xq, y, route_w, y_sum)
    n_mat = W_table.numel()
    if y is None and want_y:
        y = torch.empty((n_mat, N), dtype=torch.float32, device=xq.device)
    _call("q2k_mmvq_experts", _ptr(W_table), n_mat, N, K, _ptr(xq), 1 if x_per_matrix else 0, _ptr(y),
          _ptr(route_w), _ptr(y_sum), _stream(stream))
    return y, y_sum


def q3k_row_bytes(K) -> int:
    return lib().q3k_row_bytes(K)


def q3k_mmvq_q8_1(W, xq, K, out=None, stream=None):
    """Q3_K ``[N, K]`` (110-byte GGUF blocks) times q8_1 ``xq [m, K/32*36]``
    -> fp32 ``[m, N]``."""
    _need_cuda(W, xq, out)
    m = xq.shape[0]
    N = W.numel() // q3k_row_bytes(K)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=xq.device)
    _call("q3k_mmvq_q8_1", _ptr(W), N, K, _ptr(xq), m, _ptr(out), out.stride(0), _stream(stream))
    return out


def q3k_mmvq_experts(W_table, N, K, xq, x_per_matrix=False, y=None, route_w=None, y_sum=None, stream=None):
    """Batched single-token Q3_K MMVQ over the matrices in ``W_table``;
    optional route-weighted ``y_sum`` -> (y, y_sum)."""
    _need_cuda(W_table, xq, y, route_w, y_sum)
    n_mat = W_table.numel()
    if y is None:
        y = torch.empty((n_mat, N), dtype=torch.float32, device=xq.device)
    _call("q3k_mmvq_experts", _ptr(W_table), n_mat, N, K, _ptr(xq), 1 if x_per_matrix else 0, _ptr(y),
          _ptr(route_w), _ptr(y_sum), _stream(stream))
    return y, y_sum


def swiglu_q8_1_rows(gate_up, h_q8=None, h_bf16=None, stream=None):
    """fp32 ``[2E, N]`` (gate rows, then up rows) -> q8_1 ``h`` (and bf16 h)."""
    _need_cuda(gate_up, h_q8, h_bf16)
    twoE, N = gate_up.shape
    E = twoE // 2
    if h_q8 is None:
        h_q8 = torch.empty((E, q8_1_row_bytes(N)), dtype=torch.uint8, device=gate_up.device)
    _call("swiglu_q8_1_rows", _ptr(gate_up), E, N, _ptr(h_q8), _ptr(h_bf16), _stream(stream))
    return h_q8, h_bf16


def q2k_moe_m1_workspace_bytes(E, dim, inter) -> int:
    return lib().q2k_moe_m1_workspace_bytes(E, dim, inter)


def q2k_moe_m1(ptrs, E, dim, inter, x, route_w, y=None, workspace=None, stream=None):
    """Routed experts for one token: ``ptrs`` holds 3E device addresses
    (gate..., up..., down...); returns fp32 ``y [dim]`` (and the workspace)."""
    _need_cuda(ptrs, x, route_w, y, workspace)
    if y is None:
        y = torch.empty(dim, dtype=torch.float32, device=x.device)
    need = q2k_moe_m1_workspace_bytes(E, dim, inter)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _call("q2k_moe_m1", _ptr(ptrs), E, dim, inter, _ptr(x), _ptr(route_w), _ptr(y), _ptr(workspace),
          workspace.numel(), _stream(stream))
    return y, workspace


def q2k_moe_m1_static_scratch(ptrs, E, dim, inter, x, route_w, y=None, stream=None):
    """As ``q2k_moe_m1`` on the library's fixed device scratch (no
    workspace); calls on one device must not overlap."""
    _need_cuda(ptrs, x, route_w, y)
    if y is None:
        y = torch.empty(dim, dtype=torch.float32, device=x.device)
    _call("q2k_moe_m1_static_scratch", _ptr(ptrs), E, dim, inter, _ptr(x), _ptr(route_w), _ptr(y),
          _stream(stream))
    return y


def q2k_mmq_q8_1_workspace_bytes(m, K) -> int:
    return lib().q2k_mmq_q8_1_workspace_bytes(m, K)


def q2k_mmq_bf16(W, x, out=None, stream=None):
    """Q2_K ``[N, K]`` times bf16 ``x [m, K]`` for many tokens (the tensor
    cores over the on-chip bf16 expansion) -> fp32 ``[m, N]``."""
    _need_cuda(W, x, out)
    m, K = x.shape
    N = W.numel() // q2k_row_bytes(K)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=x.device)
    _call("q2k_mmq_bf16", _ptr(W), N, K, _ptr(x), m, x.stride(0), _ptr(out), out.stride(0), _stream(stream))
    return out


def q2k_mmq_q8_1(W, xq, K, out=None, workspace=None, stream=None):
    """Q2_K ``[N, K]`` times q8_1 ``xq [m, K/32*36]`` for many tokens ->
    fp32 ``[m, N]`` (the q8_1 values go through a bf16 workspace)."""
    _need_cuda(W, xq, out, workspace)
    m = xq.shape[0]
    N = W.numel() // q2k_row_bytes(K)
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=xq.device)
    need = lib().q2k_mmq_q8_1_workspace_bytes(m, K)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=xq.device)
    _call("q2k_mmq_q8_1", _ptr(W), N, K, _ptr(xq), m, _ptr(out), out.stride(0), _ptr(workspace), workspace.numel(),
          _stream(stream))
    return out


def dense_gemm_bf16(x, W, out=None, stream=None):
    """bf16 ``x [m, K]`` times bf16 ``W [N, K]``^T -> fp32 ``[m, N]``."""
    _need_cuda(x, W, out)
    m, K = x.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty((m, N), dtype=torch.float32, device=x.device)
    _call("dense_gemm_bf16", _ptr(x), m, K, x.stride(0), _ptr(W), N, _ptr(out), out.stride(0), _stream(stream))
    return out


def q2k_device_error(clear=True) -> int:
    """Synchronous read of the library's device error word (0 = none)."""
    v = ctypes.c_int32(0)
    _call("q2k_device_error", ctypes.byref(v), 1 if clear else 0)
    return v.value
