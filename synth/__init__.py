"""Seeded synthetic inputs for the Q2_K decode projections.

This module is shared by the CPU oracle's tests and by the CUDA path (tests,
bench, smoke).  It holds no arithmetic of the method itself: it only draws
random bytes and random activations and packs them into the layouts the
method consumes.  Every tensor comes from its own named sub-stream of
``numpy.random.default_rng`` so that adding a tensor never shifts another.

Recipe (the workloads of the engram / attention / MoE decode pages):

* Q2_K bytes: ``scales`` uniform u8 (both nibbles uniform 0..15), ``qs``
  uniform u8, ``d`` and ``dmin`` uniform in [1e-3, 1e-2] drawn in fp32 and
  rounded to fp16 (round to nearest even).  Block layout
  ``scales[16] | qs[64] | d (fp16 LE) | dmin (fp16 LE)`` = 84 bytes.
* Q3_K bytes (GGUF layout ``hmask[32] | qs[64] | scales[12] | d``, 110
  bytes): the first 108 bytes uniform u8 (so every 6-bit scale and every
  3-bit code is uniform), ``d`` of either sign with magnitude uniform in
  [1e-3, 1e-2], rounded to fp16.
* Activations: bf16 from N(0, 1) (fp32 draw, round to nearest even).
* Dense bf16 weights: N(0, 0.02).
* Engram row ids: uniform integers in [0, n_table_rows), with replacement.
* Routed experts: distinct expert ids, N(0, 1) logits, softmax route weights
  in fp32.
"""
from __future__ import annotations

import zlib

import numpy as np

Q2K_BLOCK_BYTES = 84
Q2K_BLOCK_WEIGHTS = 256
Q3K_BLOCK_BYTES = 110


def rng(seed: int, name: str) -> np.random.Generator:
    """Independent generator for tensor ``name`` under ``seed``."""
    key = zlib.crc32(name.encode("utf-8"))
    return np.random.default_rng(np.random.SeedSequence(int(seed), spawn_key=(key,)))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Pack fp32 values into bf16 bit patterns, round to nearest even.

    Only used to build inputs; NaN never occurs in the drawn data."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    # finite values stay below 0xFF800000, so the 32-bit sum cannot wrap
    u = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return u.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def q2k_blocks(seed: int, name: str, n_blocks: int) -> np.ndarray:
    """``n_blocks`` random Q2_K super-blocks as a ``[n_blocks, 84]`` uint8 array."""
    g = rng(seed, name)
    out = np.empty((n_blocks, Q2K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:80] = g.integers(0, 256, size=(n_blocks, 80), dtype=np.uint8)
    dd = g.uniform(1e-3, 1e-2, size=(n_blocks, 2)).astype(np.float32).astype(np.float16)
    out[:, 80:84] = dd.view(np.uint8).reshape(n_blocks, 4)
    return out


def q2k_matrix(seed: int, name: str, n_rows: int, k: int) -> np.ndarray:
    """A row-major ``[n_rows, k]`` Q2_K weight as ``[n_rows, k/256*84]`` bytes."""
    if k % Q2K_BLOCK_WEIGHTS:
        raise ValueError(f"K={k} is not a multiple of 256")
    nb = k // Q2K_BLOCK_WEIGHTS
    return q2k_blocks(seed, name, n_rows * nb).reshape(n_rows, nb * Q2K_BLOCK_BYTES)


def q3k_matrix(seed: int, name: str, n_rows: int, k: int) -> np.ndarray:
    """A row-major ``[n_rows, k]`` Q3_K weight as ``[n_rows, k/256*110]`` bytes."""
    if k % Q2K_BLOCK_WEIGHTS:
        raise ValueError(f"K={k} is not a multiple of 256")
    n_blocks = n_rows * (k // Q2K_BLOCK_WEIGHTS)
    g = rng(seed, name)
    out = np.empty((n_blocks, Q3K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:108] = g.integers(0, 256, size=(n_blocks, 108), dtype=np.uint8)
    d = g.uniform(1e-3, 1e-2, size=n_blocks) * np.where(g.integers(0, 2, size=n_blocks) == 1, 1.0, -1.0)
    out[:, 108:110] = d.astype(np.float32).astype(np.float16).view(np.uint8).reshape(n_blocks, 2)
    return out.reshape(n_rows, -1)


def bf16_normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, std) draws."""
    g = rng(seed, name)
    v = (g.standard_normal(size=shape) * std).astype(np.float32)
    return f32_to_bf16_bits(v)


def row_ids(seed: int, name: str, n: int, n_table_rows: int) -> np.ndarray:
    return rng(seed, name).integers(0, n_table_rows, size=n, dtype=np.int64).astype(np.int32)


def expert_route(seed: int, n_experts: int, topk: int):
    """Distinct selected expert ids and their softmax route weights (fp32)."""
    g = rng(seed, "route")
    ids = g.choice(n_experts, size=topk, replace=False).astype(np.int32)
    logits = g.standard_normal(size=topk).astype(np.float32)
    e = np.exp(logits - logits.max())
    w = (e / e.sum()).astype(np.float32)
    return ids, w
