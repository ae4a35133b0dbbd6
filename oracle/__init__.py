"""CPU oracle for the Q2_K decode projections -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no
code with it; the only thing both sides share is the seeded input generator
in ``synth``.

The arithmetic lives in ``q2k_oracle.c`` (plain C, fp64 unless the method
fixes a precision).  This module compiles it with gcc on first use and
wraps each function with NumPy marshalling, plus the two composite chains
(engram rows + projection, routed experts) written as plain sequences of
those primitives.  Function docstrings cite the metrale docs page and item
each step follows.

Parity unpinned: the Q2_K field layout is a reading of the GGUF Q2_K format
(the pages give only the 84-byte size and the name); no real GGUF file is
available to pin it against.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q2k_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q2K_BYTES = 84
Q2K_WEIGHTS = 256
Q8_1_BYTES = 36
Q8_1_VALUES = 32


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, no FP
    contraction, no fast-math) and return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_fp16_to_double.restype = ctypes.c_double
            lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = ctypes.c_double
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_f32_to_fp16.restype = ctypes.c_uint16
            lib.oracle_f32_to_fp16.argtypes = [ctypes.c_float]
            lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
            lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
            lib.oracle_q2k_decode_block.argtypes = [P, P]
            lib.oracle_q2k_decode_block_bf16.argtypes = [P, P]
            lib.oracle_q2k_dequant_rows.restype = I64
            lib.oracle_q2k_dequant_rows.argtypes = [P, I64, I64, P, I64, P]
            lib.oracle_q2k_decode_matrix.argtypes = [P, I64, I64, P]
            lib.oracle_q2k_matvec.argtypes = [P, I64, I64, P, I64, P]
            lib.oracle_q8_1_quantize_rows.argtypes = [P, I64, I64, I64, P]
            lib.oracle_q8_1_dequant_rows.argtypes = [P, I64, I64, P]
            lib.oracle_dense_gemm_bf16.argtypes = [P, I64, I64, I64, P, I64, P]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_swiglu.argtypes = [P, P, I64, P]
            lib.oracle_weighted_sum.argtypes = [P, P, I64, I64, P]
            lib.oracle_round_bf16.argtypes = [P, I64, P]
            lib.oracle_engram_hash.restype = ctypes.c_int
            lib.oracle_engram_hash.argtypes = [P, I64, P, I64, P, I64, I64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               P, P, P, I64, P]
            lib.oracle_engram_gate.argtypes = [P, P, I64, P, I64, I64, I64, ctypes.c_float, P, P]
            lib.oracle_q3k_decode_block.argtypes = [P, P]
            lib.oracle_q3k_decode_matrix.argtypes = [P, I64, I64, P]
            lib.oracle_q3k_matvec.argtypes = [P, I64, I64, P, I64, P]
            lib.oracle_q3k_block_bytes.restype = ctypes.c_int
            lib.oracle_block_bytes.restype = ctypes.c_int
            lib.oracle_q8_1_block_bytes.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar formats ----------------------------------------------------------

def fp16_to_double(h: int) -> float:
    return _L().oracle_fp16_to_double(int(h))


def bf16_to_double(b: int) -> float:
    return _L().oracle_bf16_to_double(int(b))


def f32_to_fp16(x: float) -> int:
    return _L().oracle_f32_to_fp16(float(np.float32(x)))


def f32_to_bf16(x: float) -> int:
    return _L().oracle_f32_to_bf16(float(np.float32(x)))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values (bit placement, no rounding)."""
    b = _c(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_bf16(v: np.ndarray) -> np.ndarray:
    """fp64 values -> bf16 bits (via fp32, each round to nearest even)."""
    v = _c(v, np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _L().oracle_round_bf16(_p(v), v.size, _p(out))
    return out


# ---- Q2_K ----------------------------------------------------------------------

def block_bytes() -> int:
    """Bytes of one Q2_K super-block (engram_v41.rs, `ENGRAM_ROW_BYTES`)."""
    return _L().oracle_block_bytes()


def decode_block(blk: np.ndarray) -> np.ndarray:
    """Exact fp64 weights of one 84-byte block (GGUF Q2_K reading)."""
    blk = _c(blk, np.uint8).reshape(Q2K_BYTES)
    out = np.empty(Q2K_WEIGHTS, dtype=np.float64)
    _L().oracle_q2k_decode_block(_p(blk), _p(out))
    return out


def decode_matrix(W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Exact fp64 ``[N, K]`` expansion of a Q2_K matrix
    (engram_v41.rs, `wkv_q2k`: `[out, in/256]` blocks, row-major)."""
    W = _c(W, np.uint8)
    assert W.size == N * (K // Q2K_WEIGHTS) * Q2K_BYTES
    out = np.empty((N, K), dtype=np.float64)
    _L().oracle_q2k_decode_matrix(_p(W), N, K, _p(out))
    return out


def dequant_rows(table: np.ndarray, n_table_rows: int, K: int, ids, n_rows: int):
    """Gather + dequantise to bf16 bits (engram_v41.rs, `rows_from_q2k` and
    `dequant_q2_k_to_bf16`).  Returns ``(out [n_rows, K] uint16, n_bad_ids)``."""
    table = _c(table, np.uint8)
    out = np.empty((n_rows, K), dtype=np.uint16)
    if ids is None:
        bad = _L().oracle_q2k_dequant_rows(_p(table), n_table_rows, K, None, n_rows, _p(out))
    else:
        ids = _c(ids, np.int32)
        bad = _L().oracle_q2k_dequant_rows(_p(table), n_table_rows, K, _p(ids), n_rows, _p(out))
    return out, int(bad)


def matvec(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    """``y[t, n] = sum_k w[n, k] x[t, k]`` with exact Q2_K weights, fp64
    (engram_v41/apply.rs, the single-token `wkv` projection; `y = x W^T`).
    ``x`` is fp64 ``[m, K]``; returns fp64 ``[m, N]``."""
    W = _c(W, np.uint8)
    x = _c(np.atleast_2d(x), np.float64)
    m = x.shape[0]
    assert x.shape[1] == K
    y = np.empty((m, N), dtype=np.float64)
    _L().oracle_q2k_matvec(_p(W), N, K, _p(x), m, _p(y))
    return y


# ---- Q3_K (moe_v41/init.rs names the kernels; the layout is GGUF's, a reading) ----

Q3K_BYTES = 110


def q3k_block_bytes() -> int:
    return _L().oracle_q3k_block_bytes()


def q3k_decode_block(blk: np.ndarray) -> np.ndarray:
    """Exact fp64 weights of one 110-byte Q3_K block
    (hmask[32] | qs[64] | scales[12] | d)."""
    blk = _c(blk, np.uint8).reshape(Q3K_BYTES)
    out = np.empty(Q2K_WEIGHTS, dtype=np.float64)
    _L().oracle_q3k_decode_block(_p(blk), _p(out))
    return out


def q3k_decode_matrix(W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Exact fp64 ``[N, K]`` expansion of a Q3_K matrix (``[out, in/256]``
    blocks, row-major)."""
    W = _c(W, np.uint8)
    assert W.size == N * (K // Q2K_WEIGHTS) * Q3K_BYTES
    out = np.empty((N, K), dtype=np.float64)
    _L().oracle_q3k_decode_matrix(_p(W), N, K, _p(out))
    return out


def q3k_matvec(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    """``y[t, n] = sum_k w[n, k] x[t, k]`` with exact Q3_K weights, fp64
    (moe_v41/init.rs, `kquant_mmvq_q3_k_w`).  ``x`` fp64 ``[m, K]``."""
    W = _c(W, np.uint8)
    x = _c(np.atleast_2d(x), np.float64)
    m = x.shape[0]
    assert x.shape[1] == K and W.size == N * (K // Q2K_WEIGHTS) * Q3K_BYTES
    y = np.empty((m, N), dtype=np.float64)
    _L().oracle_q3k_matvec(_p(W), N, K, _p(x), m, _p(y))
    return y


# ---- q8_1 ------------------------------------------------------------------------

def q8_1_quantize(x_bf16: np.ndarray) -> np.ndarray:
    """bf16 ``[m, K]`` -> q8_1 bytes ``[m, K/32*36]``
    (attn_v41/decode.rs, `kquant_q8_1_rows`; the block encoding is a reading)."""
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    m, K = x.shape
    out = np.empty((m, (K // Q8_1_VALUES) * Q8_1_BYTES), dtype=np.uint8)
    _L().oracle_q8_1_quantize_rows(_p(x), m, K, K, _p(out))
    return out


def q8_1_dequant(xq: np.ndarray, m: int, K: int) -> np.ndarray:
    """q8_1 bytes -> the fp64 values they encode, ``f32(d) * q``."""
    xq = _c(xq, np.uint8)
    out = np.empty((m, K), dtype=np.float64)
    _L().oracle_q8_1_dequant_rows(_p(xq), m, K, _p(out))
    return out


# ---- dense and elementwise -----------------------------------------------------------

def dense_gemm(x_bf16: np.ndarray, W_bf16: np.ndarray) -> np.ndarray:
    """``y = x W^T`` with bf16 inputs, fp64 accumulation
    (engram_v41/apply.rs, `ops::dense_gemm` for several tokens)."""
    x = _c(np.atleast_2d(x_bf16), np.uint16)
    W = _c(W_bf16, np.uint16)
    m, K = x.shape
    N = W.shape[0]
    assert W.shape[1] == K
    y = np.empty((m, N), dtype=np.float64)
    _L().oracle_dense_gemm_bf16(_p(x), m, K, K, _p(W), N, _p(y))
    return y


def silu(z: float) -> float:
    return _L().oracle_silu(float(z))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """``silu(g) * u`` in fp64 (moe_v41/init.rs, `moe_v41_swiglu`)."""
    g = _c(g, np.float64)
    u = _c(u, np.float64)
    assert g.shape == u.shape
    h = np.empty(g.shape, dtype=np.float64)
    _L().oracle_swiglu(_p(g), _p(u), g.size, _p(h))
    return h


def weighted_sum(v: np.ndarray, w: np.ndarray) -> np.ndarray:
    """``y = sum_e w[e] v[e]`` in e order, fp64
    (moe_v41/init.rs, `moe_v41_accumulate` into the f32 `acc`)."""
    v = _c(v, np.float64)
    w = _c(w, np.float32)
    E, N = v.shape
    y = np.empty(N, dtype=np.float64)
    _L().oracle_weighted_sum(_p(v), _p(w), E, N, _p(y))
    return y


# ---- composite chains --------------------------------------------------------------

def engram_rows_projection(table, n_table_rows, ids, tokens, cols, wkv_bf16):
    """Engram single step: gather + dequantise ``tokens*cols`` rows (one
    block each, `[token][col]` order), view them as ``[tokens, cols*256]``
    and project through ``wkv`` (engram_v41.rs module doc, steps 2-3;
    engram_v41/apply.rs).  Returns ``(rows_bf16, y fp64 [tokens, N])``."""
    rows, bad = dequant_rows(table, n_table_rows, Q2K_WEIGHTS, ids, tokens * cols)
    assert bad == 0
    x = rows.reshape(tokens, cols * Q2K_WEIGHTS)
    return rows, dense_gemm(x, wkv_bf16)


def moe_m1(x_bf16, gate, up, down, route_w, dim, inter, quantized=False):
    """Routed experts for one token (moe_v41/init.rs: gate and up as one
    expert batch, SwiGLU fused with q8_1 requantisation of `h`, the down
    batch, then the route-weighted sum).

    ``gate``/``up`` are lists of ``[inter, dim]`` Q2_K matrices, ``down`` a
    list of ``[dim, inter]`` ones, ``route_w`` fp32 ``[E]``.

    Steps: g, u = W x for each expert, each rounded to bf16 (the page's
    expert buffers are bf16); h = silu(g) * u in fp64, rounded to bf16;
    down_e = W_down,e h_e; y = sum_e w_e down_e in fp64.  With
    ``quantized=True`` the activations entering each projection are first
    passed through the q8_1 encoding (x and every h_e), which is what the
    path feeds its integer dot products.
    """
    E = len(gate)
    x = np.atleast_2d(x_bf16)
    xin = q8_1_dequant(q8_1_quantize(x), 1, dim) if quantized else bf16_to_f64(x)
    g = np.stack([matvec(gate[e], inter, dim, xin)[0] for e in range(E)])
    u = np.stack([matvec(up[e], inter, dim, xin)[0] for e in range(E)])
    g16 = bf16_to_f64(round_bf16(g))
    u16 = bf16_to_f64(round_bf16(u))
    h_bits = round_bf16(swiglu(g16, u16))
    if quantized:
        hin = q8_1_dequant(q8_1_quantize(h_bits), E, inter)
    else:
        hin = bf16_to_f64(h_bits)
    dn = np.stack([matvec(down[e], dim, inter, hin[e:e + 1])[0] for e in range(E)])
    y = weighted_sum(dn, route_w)
    return {"g": g, "u": u, "h_bits": h_bits, "down": dn, "y": y}


def engram_hash(token_map, cache, input_ids, start_pos, max_ngram, n_layers, n_heads, multipliers, primes,
                offsets, pad_id):
    """engram_v41.rs `EngramHasher::hash`: row ids [seqlen, n_layers,
    (max_ngram-1)*n_heads] (int64); ``cache`` (int64 [max_seq]) is updated in
    place.  Raises on a token outside token_map or past the cache, as the
    page does (the cache entries before a bad token are written)."""
    token_map = _c(token_map, np.int64)
    assert cache.dtype == np.int64 and cache.flags.c_contiguous
    ids = _c(input_ids, np.uint32)
    mults = _c(multipliers, np.int64)
    pr = _c(primes, np.int64)
    off = _c(offsets, np.int64)
    cols = (max_ngram - 1) * n_heads
    out = np.zeros((len(ids), n_layers, cols), dtype=np.int64)
    st = _L().oracle_engram_hash(_p(token_map), len(token_map), _p(cache), len(cache), _p(ids), len(ids), start_pos,
                                 max_ngram, n_layers, n_heads, _p(mults), _p(pr), _p(off), pad_id, _p(out))
    if st == -1:
        raise ValueError("token outside the engram token_map")
    if st == -2:
        raise ValueError("positions past the hash cache")
    return out


def engram_gate(streams, kv, qk, eps):
    """The engram gate (engram_v41.rs module doc, step 4; engram_v41/apply.rs,
    the `gate_k` launch): ``streams`` fp32 ``[T, hc, dim]``, ``kv`` fp32
    ``[T, (hc+1)*dim]`` (keys, then the shared value; rounded to bf16 on
    use), ``qk`` fp32 ``[hc, dim]``.  Returns ``(new streams fp64 [T, hc,
    dim], gates fp64 [T, hc])``; the readings are in q2k_oracle.c."""
    st = _c(streams, np.float32)
    T, hc, dim = st.shape
    kv = _c(kv, np.float32)
    assert kv.shape[0] == T and kv.shape[1] >= (hc + 1) * dim
    q = _c(qk, np.float32)
    assert q.shape == (hc, dim)
    out = np.empty((T, hc, dim), dtype=np.float64)
    g = np.empty((T, hc), dtype=np.float64)
    _L().oracle_engram_gate(_p(st), _p(kv), kv.shape[1], _p(q), T, hc, dim, float(np.float32(eps)), _p(out), _p(g))
    return out, g


def layer_row_ids(hashes, layer):
    """engram_v41.rs `layer_row_ids`: one layer's row ids in [token][col] order."""
    return np.ascontiguousarray(hashes[:, layer, :]).reshape(-1)
