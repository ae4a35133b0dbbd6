"""GPU parity at the configurations' full sizes, through the C ABI.

* The Q2_K sweep (N = K in {4096, 8192, 16384}, m in {1, 2, 4, 8}, bf16 and
  q8_1 activations): every output row against the oracle.
* The dense bf16 GEMM at m in {64, 256} and the same N = K: sampled weight
  rows that include the first and last row of every 128-row tile (at least
  256 of them).  Every output sums all K splits, so each sample also covers
  the split-K boundaries.
* The page's single-token engram path as one chain (engram_v41/apply.rs,
  `apply`: one token reads `wkv_q2k`): n-gram hash -> one layer's row ids ->
  q2k_dequant_rows -> q2k_gemv_bf16 against a Q2_K `wkv` [20480, 2048].
* Edge cases of the single-token kernel (rows of 32..128 blocks): ragged row
  counts, fewer rows than multiprocessors, padded lanes (rows whose blocks
  are not a power of two), K = 32768, and the pair with its matrix boundary
  inside a stage.

Bars as in test_gpu_parity.py: 2e-3 (bf16) and 1e-2 (q8_1, against the bf16
activations) of each token row's L2 norm; 1e-4 against the exact projection
of the q8_1 values; bit-exact rows and ids.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-3
TOL_Q8 = 1e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    from mmvq_q2_gb300 import build
    build.build()
    import mmvq_q2_gb300 as q
    q.lib()
    yield q
    torch.cuda.synchronize()
    assert q.q2k_device_error(clear=True) == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_dev(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def x_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def rel_err_rows(y, ref):
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    return max(np.max(np.abs(y[t] - ref[t])) / max(np.linalg.norm(ref[t]), 1e-300) for t in range(ref.shape[0]))


def oracle_matvec(W, N, K, x, threads=16):
    """The oracle's matvec over row ranges run side by side (each range is
    one unchanged oracle call)."""
    bounds = np.linspace(0, N, min(threads, N) + 1).astype(int)
    rb = W.reshape(N, -1)

    def one(ab):
        a, b = ab
        return oracle.matvec(np.ascontiguousarray(rb[a:b]), b - a, K, x)

    parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        return np.concatenate(list(ex.map(one, parts)), axis=1)


def close_to_q8_projection(y, W, N, K, xq_h):
    """y against the exact projection of the values the q8_1 row encodes:
    1e-4 of the row's L2 norm; for rows of fewer than 32 outputs, where one
    cancelling dot product can be small against its own terms, 1e-5 of
    sum_k |w_k x_k| per output (an fp32 accumulation bound)."""
    xhat = oracle.q8_1_dequant(xq_h, 1, K)
    ref = oracle_matvec(W, N, K, xhat)
    if N >= 32:
        return rel_err_rows(y, ref) <= 1e-4
    scale = np.abs(oracle.decode_matrix(W, N, K)) @ np.abs(xhat[0])
    return bool(np.all(np.abs(np.asarray(y, np.float64).reshape(-1) - ref.reshape(-1)) <= 1e-5 * scale))


# ---- the Q2_K sweep, every row ----------------------------------------------------

_SWEEP = {}


def sweep_matrix(N):
    if N not in _SWEEP:
        W = synth.q2k_matrix(0, f"sweep.W{N}x{N}", N, N)
        _SWEEP.clear()  # one resident matrix at a time
        _SWEEP[N] = (W, dev(W))
    return _SWEEP[N]


@pytest.mark.parametrize("m", [1, 2, 4, 8])
@pytest.mark.parametrize("N", [4096, 8192, 16384])
def test_sweep_every_row_both_activation_types(lib, N, m):
    W, Wd = sweep_matrix(N)
    x = synth.bf16_normal(0, f"sweep.x{m}.{N}", (m, N))
    ref = oracle_matvec(W, N, N, x_f64(x))
    y = lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy()
    assert np.all(np.isfinite(y))
    assert rel_err_rows(y, ref) <= TOL_BF16
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    xq_h = xq.cpu().numpy()
    np.testing.assert_array_equal(xq_h, oracle.q8_1_quantize(x))
    y8 = lib.q2k_mmvq_q8_1(Wd, xq, N).cpu().numpy()
    assert rel_err_rows(y8, ref) <= TOL_Q8
    assert rel_err_rows(y8, oracle_matvec(W, N, N, oracle.q8_1_dequant(xq_h, m, N))) <= 1e-4


# ---- dense GEMM at the configuration sizes ---------------------------------------------

_DENSE = {}


def dense_matrix(N):
    if N not in _DENSE:
        _DENSE.clear()
        W = synth.bf16_normal(0, f"sweep.dense.W{N}", (N, N), std=0.02)
        _DENSE[N] = (W, bf16_dev(W))
    return _DENSE[N]


@pytest.mark.parametrize("m", [64, 256])
@pytest.mark.parametrize("N", [4096, 8192, 16384])
def test_dense_gemm_config_tile_edges(lib, N, m):
    W, Wd = dense_matrix(N)
    x = synth.bf16_normal(0, f"sweep.dense.x{m}.{N}", (m, N))
    y = lib.dense_gemm_bf16(bf16_dev(x), Wd).cpu().numpy()
    edges = np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)])
    others = np.setdiff1d(np.arange(N), edges)
    extra = np.random.default_rng(N + m).choice(others, max(0, 256 - len(edges)), replace=False)
    rows = np.unique(np.concatenate([edges, extra]))
    assert len(rows) >= 256
    ref = oracle.dense_gemm(x, np.ascontiguousarray(W[rows]))
    assert rel_err_rows(y[:, rows], ref) <= TOL_BF16


# ---- the page's single-token engram path ------------------------------------------------

def test_engram_single_token_q2k_wkv_chain(lib):
    """One token: hash -> the layer's 8 row ids -> 8 rows of 256 bf16 ->
    [1, 2048] -> the Q2_K GEMV against wkv_q2k [dim*(hc+1), cols*256] =
    [20480, 2048] (dim 4096, hc 4, cols 8), all on the device."""
    rng = np.random.default_rng(21)
    ng, nl, nh, n_table = 3, 2, 4, 1 << 20
    tm = rng.integers(0, 1 << 40, size=4096).astype(np.int64)
    mults = rng.integers(-(1 << 62), 1 << 62, size=(nl, ng)).astype(np.int64)
    primes = np.full((nl, ng - 1, nh), 131071, np.int64)
    offsets = (np.arange(nl * (ng - 1) * nh, dtype=np.int64) % 8 * 65536).reshape(nl, (ng - 1) * nh)
    args = dict(max_ngram=ng, n_layers=nl, n_heads=nh, multipliers=mults, primes=primes, offsets=offsets, pad_id=7)
    # a prefill of 5 tokens, then the decode step: the one token of interest
    prefill = rng.integers(0, len(tm), size=5).astype(np.uint32)
    step = rng.integers(0, len(tm), size=1).astype(np.uint32)
    cache_h = np.zeros(64, np.int64)
    oracle.engram_hash(tm, cache_h, prefill, 0, **args)
    ref_hash = oracle.engram_hash(tm, cache_h, step, 5, **args)
    ids_ref = oracle.layer_row_ids(ref_hash, 0).astype(np.int32)
    assert len(ids_ref) == 8 and ids_ref.max() < n_table

    hdev = lambda a: dev(np.asarray(a))  # noqa: E731
    cache = torch.zeros(64, dtype=torch.int64, device="cuda")
    lib.q2k_engram_hash(hdev(tm), cache, hdev(prefill), 0, ng, nl, nh, hdev(mults), hdev(primes), hdev(offsets), 7)
    _, lid = lib.q2k_engram_hash(hdev(tm), cache, hdev(step), 5, ng, nl, nh, hdev(mults), hdev(primes), hdev(offsets),
                                 7, layer_index=0)
    np.testing.assert_array_equal(lid.cpu().numpy().reshape(-1), ids_ref)

    table = synth.q2k_blocks(0, "cfg1.table", n_table)
    wkv_q = synth.q2k_matrix(0, "engram.wkv_q2k", 20480, 2048)
    rows = lib.q2k_dequant_rows(dev(table), 256, ids=lid.view(-1))
    y = lib.q2k_gemv_bf16(dev(wkv_q), rows.view(1, 2048)).cpu().numpy()
    ref_rows, bad = oracle.dequant_rows(table, n_table, 256, ids_ref, 8)
    assert bad == 0
    np.testing.assert_array_equal(host_bits(rows), ref_rows)
    ref_y = oracle_matvec(wkv_q, 20480, 2048, oracle.bf16_to_f64(ref_rows.reshape(1, 2048)))
    assert rel_err_rows(y, ref_y) <= TOL_BF16


# ---- the single-token kernel's edge cases ---------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 8192), (5, 16384), (151, 8192), (153, 9216), (1000, 10240), (4097, 16384),
                                 (300, 32768), (777, 12288)])
def test_single_token_kernel_shapes(lib, N, K):
    W = synth.q2k_matrix(13, f"m1.{N}.{K}", N, K)
    x = synth.bf16_normal(13, f"m1.x.{K}", (1, K))
    Wd = dev(W)
    ref = oracle_matvec(W, N, K, x_f64(x))
    y = lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy()
    if N >= 32:
        assert rel_err_rows(y, ref) <= TOL_BF16
    else:  # a handful of cancelling dot products: bound against their terms
        scale = np.abs(oracle.decode_matrix(W, N, K)) @ np.abs(x_f64(x)[0])
        assert np.all(np.abs(y.reshape(-1) - ref.reshape(-1)) <= 1e-4 * scale)
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    y8 = lib.q2k_mmvq_q8_1(Wd, xq, K).cpu().numpy()
    assert close_to_q8_projection(y8, W, N, K, xq.cpu().numpy())
    # a repeat gives the same bits
    assert np.array_equal(y, lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy())


@pytest.mark.parametrize("Na,Nb,K", [(1027, 517, 8192), (3, 2000, 16384), (160, 1, 12288)])
def test_single_token_pair_boundary_inside_a_stage(lib, Na, Nb, K):
    """The pair's rows are one row space (Wa's, then Wb's); a stage may hold
    rows of both matrices (two copies into one slot).  Each output equals
    the single call bit for bit and the oracle within the q8_1 bars."""
    Wa = synth.q2k_matrix(14, f"pm1.a.{Na}.{K}", Na, K)
    Wb = synth.q2k_matrix(14, f"pm1.b.{Nb}.{K}", Nb, K)
    x = synth.bf16_normal(14, f"pm1.x.{K}", (1, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    Wad, Wbd = dev(Wa), dev(Wb)
    ya, yb = lib.q2k_mmvq_pair(Wad, Wbd, xq, K)
    assert torch.equal(ya, lib.q2k_mmvq_q8_1(Wad, xq, K))
    assert torch.equal(yb, lib.q2k_mmvq_q8_1(Wbd, xq, K))
    xq_h = xq.cpu().numpy()
    assert close_to_q8_projection(ya.cpu().numpy(), Wa, Na, K, xq_h)
    assert close_to_q8_projection(yb.cpu().numpy(), Wb, Nb, K, xq_h)


def test_single_token_kernel_and_general_kernel_agree(lib):
    """Activations off a 16-byte boundary take the general kernel; aligned
    ones the single-token kernel.  Both within the bf16 bar of the oracle,
    and within rounding of each other."""
    N, K = 600, 16384
    W = synth.q2k_matrix(15, "m1g.W", N, K)
    x = synth.bf16_normal(15, "m1g.x", (1, K))
    Wd = dev(W)
    buf = torch.zeros(K + 8, dtype=torch.int16, device="cuda")
    buf[1:1 + K] = torch.from_numpy(x.view(np.int16).reshape(-1)).cuda()
    x_off = buf[1:1 + K].view(1, K).view(torch.bfloat16)
    y_al = lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy()
    y_un = lib.q2k_gemv_bf16(Wd, x_off).cpu().numpy()
    ref = oracle_matvec(W, N, K, x_f64(x))
    assert rel_err_rows(y_al, ref) <= TOL_BF16
    assert rel_err_rows(y_un, ref) <= TOL_BF16
    assert rel_err_rows(y_al, y_un) <= 1e-5


# ---- the engram gate and the whole engram step -------------------------------------------

@pytest.mark.parametrize("T,hc,dim,pad", [(1, 4, 4096, 0), (16, 4, 4096, 0), (3, 1, 1000, 5), (2, 2, 7, 0),
                                          (5, 3, 2048, 64)])
def test_engram_gate_against_oracle(lib, T, hc, dim, pad):
    g = np.random.default_rng(T * 100 + hc * 10 + dim)
    streams = g.standard_normal((T, hc, dim)).astype(np.float32)
    # keys correlated with their streams so the gates spread over (0, 1)
    kv = g.standard_normal((T, (hc + 1) * dim + pad)).astype(np.float32)
    for c in range(hc):
        kv[:, c * dim:(c + 1) * dim] += (g.uniform(-2, 2, (T, 1)) * streams[:, c, :]).astype(np.float32)
    qk = g.uniform(0.5, 1.5, (hc, dim)).astype(np.float32)
    ref, ref_g = oracle.engram_gate(streams, kv, qk, 1e-6)
    sd = dev(streams)
    gates = torch.empty((T, hc), dtype=torch.float32, device="cuda")
    lib.q2k_engram_gate(sd, dev(kv), dev(qk), 1e-6, gates=gates)
    got = sd.cpu().numpy().astype(np.float64)
    for t in range(T):
        for c in range(hc):
            assert np.max(np.abs(got[t, c] - ref[t, c])) <= 1e-5 * np.linalg.norm(ref[t, c])
    np.testing.assert_allclose(gates.cpu().numpy(), ref_g, rtol=0, atol=2e-6)
    if T * hc > 4:
        assert ref_g.min() < 0.4 and ref_g.max() > 0.6  # the gates did spread
    # in place and deterministic: a second call on a fresh copy gives the same bits
    sd2 = dev(streams)
    lib.q2k_engram_gate(sd2, dev(kv), dev(qk), 1e-6)
    assert torch.equal(sd2, sd)


def _engram_tables(seed):
    rng = np.random.default_rng(seed)
    ng, nl, nh = 3, 2, 4
    tm = rng.integers(0, 1 << 40, size=4096).astype(np.int64)
    mults = rng.integers(-(1 << 62), 1 << 62, size=(nl, ng)).astype(np.int64)
    primes = np.full((nl, ng - 1, nh), 131071, np.int64)
    offsets = (np.arange(nl * (ng - 1) * nh, dtype=np.int64) % 8 * 65536).reshape(nl, (ng - 1) * nh)
    return rng, dict(max_ngram=ng, n_layers=nl, n_heads=nh, multipliers=mults, primes=primes, offsets=offsets,
                     pad_id=7), tm


@pytest.mark.parametrize("T", [16, 1])
def test_engram_step_hash_rows_projection_gate(lib, T):
    """The whole engram step on the device (engram_v41.rs module doc, steps
    1-4; engram_v41/apply.rs `apply`): hash -> one layer's row ids -> rows
    -> projection (16 tokens: the bf16 GEMM over wkv; one token: the Q2_K
    GEMV over wkv_q2k) -> gate on the fp32 streams [T, 4, 4096], against
    the oracle's chain."""
    dim, hc, cols, n_table, eps = 4096, 4, 8, 1 << 20, 1e-6
    rng, args, tm = _engram_tables(40 + T)
    toks = rng.integers(0, len(tm), size=T).astype(np.uint32)
    ref_hash = oracle.engram_hash(tm, np.zeros(64, np.int64), toks, 0, **args)
    ids_ref = oracle.layer_row_ids(ref_hash, 1).astype(np.int32)
    table = synth.q2k_blocks(0, "cfg1.table", n_table)
    streams = rng.standard_normal((T, hc, dim)).astype(np.float32)
    qk = rng.uniform(0.5, 1.5, (hc, dim)).astype(np.float32)

    hdev = lambda a: dev(np.asarray(a))  # noqa: E731
    _, lid = lib.q2k_engram_hash(hdev(tm), torch.zeros(64, dtype=torch.int64, device="cuda"), hdev(toks), 0,
                                 args["max_ngram"], args["n_layers"], args["n_heads"], hdev(args["multipliers"]),
                                 hdev(args["primes"]), hdev(args["offsets"]), args["pad_id"], layer_index=1)
    rows = lib.q2k_dequant_rows(dev(table), 256, ids=lid.view(-1))
    ref_rows, bad = oracle.dequant_rows(table, n_table, 256, ids_ref, T * cols)
    assert bad == 0
    np.testing.assert_array_equal(host_bits(rows), ref_rows)
    xr = oracle.bf16_to_f64(ref_rows.reshape(T, cols * 256))
    if T > 1:
        wkv = synth.bf16_normal(0, "cfg1.wkv", (dim * (hc + 1), cols * 256), std=0.02)
        kv = lib.dense_gemm_bf16(rows.view(T, cols * 256), bf16_dev(wkv))
        kv_ref = oracle.dense_gemm(ref_rows.reshape(T, cols * 256), wkv)
    else:
        wq = synth.q2k_matrix(0, "engram.wkv_q2k", dim * (hc + 1), cols * 256)
        kv = lib.q2k_gemv_bf16(dev(wq), rows.view(1, cols * 256))
        kv_ref = oracle_matvec(wq, dim * (hc + 1), cols * 256, xr)
    assert rel_err_rows(kv.cpu().numpy(), kv_ref) <= TOL_BF16
    sd = dev(streams)
    lib.q2k_engram_gate(sd, kv, dev(qk), eps)
    ref, _ = oracle.engram_gate(streams, kv_ref.astype(np.float32), qk, eps)
    got = sd.cpu().numpy().astype(np.float64)
    for t in range(T):
        for c in range(hc):
            assert np.max(np.abs(got[t, c] - ref[t, c])) <= TOL_BF16 * np.linalg.norm(ref[t, c])
