"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (from the method's statement of tolerances):
  * dequantised bf16 rows and the row gather: bit-exact;
  * q8_1 encoding: q, d and s bit-exact;
  * bf16-activation projections: max|y - y_ref| / ||y_ref[t]||_2 <= 2e-3 per
    token row;
  * q8_1-activation projections: the same metric <= 1e-2 against the
    projection of the original bf16 activations;
  * dense GEMM: 2e-3 of each row's L2 norm.
The configurations at their full sizes (every row of the Q2_K sweep, GEMM
tile edges, the single-token engram chain) are in test_gpu_configs.py.
"""
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


def rel_err_rows(y, ref):
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    return max(np.max(np.abs(y[t] - ref[t])) / max(np.linalg.norm(ref[t]), 1e-300) for t in range(ref.shape[0]))


def x_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# ---- a1: gather + dequantise -------------------------------------------------

def test_dequant_rows_contiguous_cfg0(lib):
    W = synth.q2k_matrix(0, "cfg0.W", 512, 4096)
    out = lib.q2k_dequant_rows(dev(W), 4096)
    ref, bad = oracle.dequant_rows(W, 512, 4096, None, 512)
    assert bad == 0
    np.testing.assert_array_equal(host_bits(out), ref)


def test_dequant_rows_gather_cfg1_bitexact_and_equal_to_contiguous_copy(lib):
    n_table = 1 << 20
    table = synth.q2k_blocks(0, "cfg1.table", n_table)
    ids = synth.row_ids(0, "cfg1.ids", 16 * 8, n_table)
    dt = dev(table)
    out = lib.q2k_dequant_rows(dt, 256, ids=dev(ids))
    ref, bad = oracle.dequant_rows(table, n_table, 256, ids, len(ids))
    assert bad == 0
    got = host_bits(out)
    np.testing.assert_array_equal(got, ref)
    copy = lib.q2k_dequant_rows(dev(table[ids]), 256)
    np.testing.assert_array_equal(host_bits(copy), got)


def test_dequant_rows_bad_ids_zero_rows_and_flag(lib):
    table = synth.q2k_blocks(1, "bad.table", 64)
    ids = np.array([3, -1, 64, 3, 63], dtype=np.int32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = lib.q2k_dequant_rows(dev(table), 256, ids=dev(ids), err_flag=flag)
    ref, bad = oracle.dequant_rows(table, 64, 256, ids, len(ids))
    assert bad == 2 and flag.item() == 1
    np.testing.assert_array_equal(host_bits(out), ref)
    flag.zero_()
    lib.q2k_dequant_rows(dev(table), 256, ids=dev(ids[[0, 4]]), err_flag=flag)
    torch.cuda.synchronize()
    assert flag.item() == 0


@pytest.mark.parametrize("K", [256, 512, 768, 1280])
def test_dequant_rows_odd_widths_and_unaligned_output(lib, K):
    W = synth.q2k_matrix(2, f"odd.{K}", 7, K)
    full = torch.empty(7 * K + 1, dtype=torch.bfloat16, device="cuda")
    out = full[1:].view(7, K)  # 2-byte aligned only
    lib.q2k_dequant_rows(dev(W), K, out=out)
    ref, _ = oracle.dequant_rows(W, 7, K, None, 7)
    np.testing.assert_array_equal(host_bits(out.contiguous()), ref)


def _hash_setup(seed, ng=3, nl=2, nh=4, vocab=1000):
    rng = np.random.default_rng(seed)
    tm = rng.integers(0, 1 << 40, size=vocab).astype(np.int64)
    tm[rng.integers(0, vocab, size=5)] = -1
    args = dict(max_ngram=ng, n_layers=nl, n_heads=nh,
                multipliers=rng.integers(-(1 << 62), 1 << 62, size=(nl, ng)).astype(np.int64),
                primes=rng.integers(1 << 19, 1 << 20, size=(nl, ng - 1, nh)).astype(np.int64),
                offsets=(np.arange(nl * (ng - 1) * nh, dtype=np.int64) * (1 << 20)).reshape(nl, -1),
                pad_id=int(rng.integers(0, 1 << 40)))
    return rng, tm, args


def _hash_dev(lib, tm, cache_d, ids, start, args, layer_index=None, err=None):
    return lib.q2k_engram_hash(dev(tm), cache_d, dev(np.asarray(ids, np.uint32)), start, args["max_ngram"],
                               args["n_layers"], args["n_heads"], dev(args["multipliers"]), dev(args["primes"]),
                               dev(args["offsets"]), args["pad_id"], layer_index=layer_index, err_flag=err)


@pytest.mark.parametrize("ng,nl,nh,seqlen", [(3, 2, 4, 16), (2, 1, 1, 1), (16, 3, 2, 700)])
def test_engram_hash_against_oracle_and_incremental(lib, ng, nl, nh, seqlen):
    rng, tm, args = _hash_setup(ng * 100 + seqlen, ng, nl, nh)
    ids = rng.integers(0, len(tm), size=seqlen).astype(np.uint32)
    cache = np.zeros(seqlen + 8, np.int64)
    ref = oracle.engram_hash(tm, cache, ids, 0, **args)
    cache_d = torch.zeros(seqlen + 8, dtype=torch.int64, device="cuda")
    out, lid = _hash_dev(lib, tm, cache_d, ids, 0, args, layer_index=nl - 1)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    np.testing.assert_array_equal(lid.cpu().numpy().reshape(-1), oracle.layer_row_ids(ref, nl - 1).astype(np.int32))
    np.testing.assert_array_equal(cache_d.cpu().numpy(), cache)
    # the same tokens in two calls (decode: one at a time after a prefix)
    cut = seqlen // 2
    c2 = torch.zeros(seqlen + 8, dtype=torch.int64, device="cuda")
    a, _ = _hash_dev(lib, tm, c2, ids[:cut], 0, args)
    b, _ = _hash_dev(lib, tm, c2, ids[cut:], cut, args)
    np.testing.assert_array_equal(np.concatenate([a.cpu().numpy(), b.cpu().numpy()]), ref)


def test_engram_hash_token_outside_the_map_sets_the_flag(lib):
    rng, tm, args = _hash_setup(7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_d = torch.zeros(8, dtype=torch.int64, device="cuda")
    out, _ = _hash_dev(lib, tm, cache_d, [3, len(tm) + 5, 4], 0, args, err=err)
    assert err.item() & 1
    assert cache_d[1].item() == -1  # reads as unmapped: later n-grams that reach it see pad
    tm2 = tm.copy()
    tm2[999] = -1
    ref = oracle.engram_hash(tm2, np.zeros(8, np.int64), [3, 999, 4], 0, **args)
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def test_engram_hash_rows_projection_chain(lib):
    """hash -> one layer's ids -> q2k_dequant_rows -> dense GEMM, all on the
    device, against the oracle's chain (cfg1 shapes: 16 tokens x 8 cols)."""
    rng, tm, args = _hash_setup(11, ng=3, nl=2, nh=4)
    n_table = 1 << 20
    args["primes"] = np.full((2, 2, 4), 131071, np.int64)  # ids inside the table
    args["offsets"] = (np.arange(16, dtype=np.int64) % 8 * 65536).reshape(2, 8)  # ids below 2^20
    ids = rng.integers(0, len(tm), size=16).astype(np.uint32)
    ref_hash = oracle.engram_hash(tm, np.zeros(32, np.int64), ids, 0, **args)
    row_ids = oracle.layer_row_ids(ref_hash, 1).astype(np.int32)
    assert row_ids.max() < n_table
    table = synth.q2k_blocks(0, "cfg1.table", n_table)
    wkv = synth.bf16_normal(0, "cfg1.wkv", (4096, 2048), std=0.02)
    _, lid = _hash_dev(lib, tm, torch.zeros(32, dtype=torch.int64, device="cuda"), ids, 0, args, layer_index=1)
    rows = lib.q2k_dequant_rows(dev(table), 256, ids=lid.view(-1))
    y = lib.dense_gemm_bf16(rows.view(16, 2048), bf16_dev(wkv)).cpu().numpy()
    ref_rows, ref_y = oracle.engram_rows_projection(table, n_table, row_ids, 16, 8, wkv)
    np.testing.assert_array_equal(host_bits(rows), ref_rows)
    assert rel_err_rows(y, ref_y) <= TOL_BF16


# ---- a2: q8_1 ------------------------------------------------------------------

@pytest.mark.parametrize("m,K,pad", [(1, 32, 0), (3, 256, 8), (8, 4096, 0), (2, 16384, 32), (5, 2048, 0)])
def test_q8_1_quantize_bitexact(lib, m, K, pad):
    x = synth.bf16_normal(3, f"q8.{m}.{K}", (m, K + pad))
    x[:, :32] = 0  # an all-zero block
    xd = bf16_dev(x)[:, :K]
    got = lib.q8_1_quantize_rows(xd).cpu().numpy()
    ref = oracle.q8_1_quantize(np.ascontiguousarray(x[:, :K]))
    np.testing.assert_array_equal(got, ref)


def test_q8_1_ties_round_away_from_zero(lib):
    vals = np.zeros((1, 64), dtype=np.float32)
    vals[0, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]
    x = synth.f32_to_bf16_bits(vals)
    np.testing.assert_array_equal(lib.q8_1_quantize_rows(bf16_dev(x)).cpu().numpy(), oracle.q8_1_quantize(x))


# ---- a3: Q2_K GEMV, bf16 activations -------------------------------------------

SMALL = [(1, 256, 1), (5, 256, 8), (3, 512, 2), (7, 768, 3), (33, 1024, 4), (17, 2048, 5), (9, 4096, 8),
         (130, 1280, 1), (1537, 2048, 1), (64, 4096, 6), (40, 8192, 7)]


@pytest.mark.parametrize("N,K,m", SMALL)
def test_gemv_bf16_small(lib, N, K, m):
    W = synth.q2k_matrix(4, f"gemv.{N}.{K}", N, K)
    x = synth.bf16_normal(4, f"gemv.x.{m}.{K}", (m, K))
    y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    ref = oracle.matvec(W, N, K, x_f64(x))
    assert rel_err_rows(y, ref) <= TOL_BF16


# one token over long rows takes whole half blocks per thread (8-word
# slices): ragged row counts, K not a power of two, rows that are not 16-byte
# aligned (K = 8448: 2772-byte rows, the 4-byte copy path) and a K split into
# two chunks that add into y (40960)
LONG_M1 = [(37, 8192), (100, 8448), (257, 12288), (19, 40960)]


@pytest.mark.parametrize("N,K", LONG_M1)
def test_gemv_bf16_long_rows_one_token(lib, N, K):
    W = synth.q2k_matrix(6, f"long.{N}.{K}", N, K)
    x = synth.bf16_normal(6, f"long.x.{K}", (1, K))
    y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16


@pytest.mark.parametrize("N,K", LONG_M1)
def test_mmvq_q8_1_long_rows_one_token(lib, N, K):
    W = synth.q2k_matrix(6, f"long.{N}.{K}", N, K)
    x = synth.bf16_normal(6, f"long.x.{K}", (1, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q2k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq, 1, K))) <= 1e-4
    if N >= 32:  # the q8_1 gate against the bf16 values (see the small shapes)
        assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_Q8


# the row-team kernel's widths: one token at 16..31 blocks per row, two or
# four tokens at 8..31 (teams of a power of two of lanes: 20 and 28 blocks
# leave lanes idle), ragged row counts
TEAM_WIDTHS = [(1, 4096, 37), (1, 5120, 1000), (1, 7168, 300), (2, 2048, 300), (2, 3072, 1000), (2, 5120, 37),
               (4, 2048, 1000), (4, 3072, 300)]


@pytest.mark.parametrize("m,K,N", TEAM_WIDTHS)
def test_row_team_widths_against_oracle(lib, m, K, N):
    W = synth.q2k_matrix(30, f"team.{N}.{K}", N, K)
    x = synth.bf16_normal(30, f"team.x.{m}.{K}", (m, K))
    Wd = dev(W)
    if m <= 2:
        y = lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy()
        assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16
    xq = oracle.q8_1_quantize(x)
    y8 = lib.q2k_mmvq_q8_1(Wd, dev(xq), K).cpu().numpy()
    assert rel_err_rows(y8, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= 1e-4


def _q8_rows_at_a_rounding_edge(m, K):
    """q8_1 rows whose every 32-value block has d = 1285 * 2^-16 (exact in
    fp16) and one q = 51: a slice's group sum d*51 has the mantissa
    65535/32768, half a step below a power of two, so packing it with its
    top at 2^15 would round to 2^15 and wrap the 16-bit field."""
    nblk = K // 32
    d = np.float16(1285 * 2.0 ** -16)
    assert float(d) == 1285 * 2.0 ** -16
    blk = np.zeros((m, nblk, 36), dtype=np.uint8)
    blk[:, :, 0:2] = np.frombuffer(d.tobytes(), dtype=np.uint8)
    blk[:, :, 2:4] = np.frombuffer(np.float16(float(d) * 51).tobytes(), dtype=np.uint8)
    blk[:, :, 4] = 51
    return blk.reshape(m, nblk * 36)


@pytest.mark.parametrize("m,K", [(1, 4096), (1, 8192), (2, 4096)])
def test_mmvq_min_sums_at_a_rounding_edge(lib, m, K):
    N = 96
    W = synth.q2k_matrix(9, f"edge.{K}", N, K)
    xq = _q8_rows_at_a_rounding_edge(m, K)
    y = lib.q2k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= 1e-4


def test_grouped_min_sums_at_a_rounding_edge(lib):
    groups, R, Kg, m = 8, 64, 2048, 8  # eight tokens: the 2-word slices
    W = synth.q2k_matrix(9, "edge.grp", groups * R, Kg)
    xq = _q8_rows_at_a_rounding_edge(m, groups * Kg)
    y = lib.q2k_mmvq_grouped(dev(W), groups, R, Kg, dev(xq)).cpu().numpy()
    xf = oracle.q8_1_dequant(xq, m, groups * Kg)
    rb = W.nbytes // (groups * R)
    for g in range(groups):
        Wg = np.ascontiguousarray(W.reshape(groups * R, rb)[g * R:(g + 1) * R])
        ref = oracle.matvec(Wg, R, Kg, np.ascontiguousarray(xf[:, g * Kg:(g + 1) * Kg]))
        assert rel_err_rows(y[:, g * R:(g + 1) * R], ref) <= 1e-4, g


def test_gemv_bf16_unaligned_weights_take_the_copy_path(lib):
    N, K = 21, 4096
    W = synth.q2k_matrix(5, "unal", N, K)
    buf = torch.zeros(W.size + 4, dtype=torch.uint8, device="cuda")
    buf[4:] = dev(W.reshape(-1))
    x = synth.bf16_normal(5, "unal.x", (2, K))
    y = lib.q2k_gemv_bf16(buf[4:], bf16_dev(x)).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16


def test_gemv_bf16_cfg0(lib):
    W = synth.q2k_matrix(0, "cfg0.W", 512, 4096)
    x = synth.bf16_normal(0, "cfg0.x", (1, 4096))
    y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, 512, 4096, x_f64(x))) <= TOL_BF16


def test_gemv_bf16_output_stride_and_guard(lib):
    N, K, m = 100, 1024, 3
    W = synth.q2k_matrix(6, "guard", N, K)
    x = synth.bf16_normal(6, "guard.x", (m, K))
    buf = torch.full((m, N + 16), 7.0, dtype=torch.float32, device="cuda")
    lib.q2k_gemv_bf16(dev(W), bf16_dev(x), out=buf[:, :N])
    b = buf.cpu().numpy()
    assert np.all(b[:, N:] == 7.0)
    assert rel_err_rows(b[:, :N], oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16


@pytest.mark.parametrize("K,one_token", [(1024, False), (8192, True)])
def test_gemv_bf16_extreme_activation_ranges(lib, K, one_token):
    # groups with mixed magnitudes, tiny values and zeros; K = 8192 one row
    # at a time takes the 8-word slices (one exponent per 32 values)
    N = 16
    W = synth.q2k_matrix(7, f"ext.{K}", N, K)
    v = np.random.default_rng(7).standard_normal((2, K)).astype(np.float32)
    v[0, ::3] *= 1e-4
    v[0, 5::7] = 0.0
    v[1] *= 1e20
    v[1, :64] = 0.0
    x = synth.f32_to_bf16_bits(v)
    if one_token:
        y = np.concatenate([lib.q2k_gemv_bf16(dev(W), bf16_dev(x[t:t + 1])).cpu().numpy() for t in range(2)])
    else:
        y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16


@pytest.fixture(scope="module")
def big_w():
    W = synth.q2k_matrix(0, "sweep.W16384", 16384, 16384)
    return W, dev(W)


# ---- a4: Q2_K x q8_1 MMVQ -------------------------------------------------------

@pytest.mark.parametrize("N,K,m", SMALL)
def test_mmvq_q8_1_small(lib, N, K, m):
    W = synth.q2k_matrix(8, f"mmvq.{N}.{K}", N, K)
    x = synth.bf16_normal(8, f"mmvq.x.{m}.{K}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q2k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    # against the exact projection of the values the q8_1 rows encode
    assert rel_err_rows(y, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= 1e-4
    # against the bf16 activations: the q8_1 gate, meaningful once the
    # output row is long enough for its L2 norm to average the per-element
    # quantisation noise (a single output is one noisy dot product)
    if N >= 32:
        assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_Q8


# ---- a5: paired launch ------------------------------------------------------------

@pytest.mark.parametrize("m", [1, 4, 8])
def test_pair_cfg2_equals_two_singles_bitwise(lib, m):
    K = 4096
    Wa = synth.q2k_matrix(0, "cfg2.wq_a", 1024, K)
    Wb = synth.q2k_matrix(0, "cfg2.wkv", 512, K)
    x = synth.bf16_normal(0, f"cfg2.x{m}", (m, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    da, db = dev(Wa), dev(Wb)
    ya, yb = lib.q2k_mmvq_pair(da, db, xq, K)
    sa = lib.q2k_mmvq_q8_1(da, xq, K)
    sb = lib.q2k_mmvq_q8_1(db, xq, K)
    assert torch.equal(ya, sa) and torch.equal(yb, sb)
    assert rel_err_rows(ya.cpu().numpy(), oracle.matvec(Wa, 1024, K, x_f64(x))) <= TOL_Q8
    assert rel_err_rows(yb.cpu().numpy(), oracle.matvec(Wb, 512, K, x_f64(x))) <= TOL_Q8


@pytest.mark.parametrize("m,K,off", [(1, 4096, 0), (1, 8448, 0), (1, 4096, 1), (4, 4096, 0)])
def test_pair_bf16_equals_quantise_then_pair(lib, m, K, off):
    """The one-call pair over bf16 rows (q8_1 made inside the launch for an
    aligned single row; a launch of its own otherwise, off = 1 element)."""
    Wa = synth.q2k_matrix(7, f"pb.a.{K}", 1024, K)
    Wb = synth.q2k_matrix(7, f"pb.b.{K}", 130, K)
    x = synth.bf16_normal(7, f"pb.x.{m}.{K}", (m, K))
    buf = torch.zeros(m * K + 8, dtype=torch.int16, device="cuda")
    buf[off:off + m * K] = torch.from_numpy(x.view(np.int16).reshape(-1)).cuda()
    xd = buf[off:off + m * K].view(m, K).view(torch.bfloat16)
    ya, yb, xq = lib.q2k_mmvq_pair_bf16(dev(Wa), dev(Wb), xd, K)
    xq2 = lib.q8_1_quantize_rows(xd)
    ya2, yb2 = lib.q2k_mmvq_pair(dev(Wa), dev(Wb), xq2, K)
    assert torch.equal(xq, xq2)
    assert torch.equal(ya, ya2) and torch.equal(yb, yb2)
    np.testing.assert_array_equal(xq.cpu().numpy(), oracle.q8_1_quantize(x))


def test_pair_ragged_sizes(lib):
    K = 768
    Wa = synth.q2k_matrix(1, "pr.a", 37, K)
    Wb = synth.q2k_matrix(1, "pr.b", 5, K)
    x = synth.bf16_normal(1, "pr.x", (3, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    ya, yb = lib.q2k_mmvq_pair(dev(Wa), dev(Wb), xq, K)
    assert torch.equal(ya, lib.q2k_mmvq_q8_1(dev(Wa), xq, K))
    assert torch.equal(yb, lib.q2k_mmvq_q8_1(dev(Wb), xq, K))


@pytest.mark.parametrize("m,K", [(1, 8448), (1, 16384), (6, 8448), (8, 16384)])
def test_pair_several_tokens_long_k(lib, m, K):
    # several tokens and several K chunks (the tensor-core path): each output
    # still equals the single call bit for bit, and matches the oracle
    Wa = synth.q2k_matrix(5, f"prl.a.{K}", 45, K)
    Wb = synth.q2k_matrix(5, f"prl.b.{K}", 19, K)
    x = synth.bf16_normal(5, f"prl.x.{m}.{K}", (m, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    ya, yb = lib.q2k_mmvq_pair(dev(Wa), dev(Wb), xq, K)
    assert torch.equal(ya, lib.q2k_mmvq_q8_1(dev(Wa), xq, K))
    assert torch.equal(yb, lib.q2k_mmvq_q8_1(dev(Wb), xq, K))
    xqf = oracle.q8_1_dequant(xq.cpu().numpy(), m, K)
    for W, y in ((Wa, ya), (Wb, yb)):
        refq = oracle.matvec(W, W.shape[0], K, xqf)
        assert rel_err_rows(y.cpu().numpy(), refq) <= 1e-4
        assert rel_err_rows(y.cpu().numpy(), oracle.matvec(W, W.shape[0], K, x_f64(x))) <= TOL_Q8


# ---- seeded sweep of small problems: every slice width and token count ---------------

@pytest.mark.parametrize("seed", range(24))
def test_gemv_and_mmvq_seeded_sweep(lib, seed):
    """Random shapes (1..8 tokens, K from 1 to 40 blocks, ragged N) through
    both activation types, against the oracle: data-dependent paths (the
    activation exponents, the 16-bit sums) meet many inputs."""
    rng = np.random.default_rng(1000 + seed)
    m = int(rng.integers(1, 9))
    K = 256 * int(rng.choice([1, 2, 3, 5, 8, 16, 24, 32, 33, 40]))
    N = int(rng.integers(16, 300))  # enough outputs that the row norm is not one cancelled dot
    W = synth.q2k_matrix(10 + seed, f"sw.{seed}", N, K)
    x = synth.bf16_normal(10 + seed, f"sw.x.{seed}", (m, K))
    if seed % 3 == 0:  # wide dynamic range inside groups
        v = synth.bf16_bits_to_f32(x) * np.exp2(rng.integers(-12, 12, size=(m, K))).astype(np.float32)
        x = synth.f32_to_bf16_bits(v)
    y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16
    xq = oracle.q8_1_quantize(x)
    yq = lib.q2k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert rel_err_rows(yq, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= 1e-4


# ---- grouped (block-diagonal) MMVQ: the Q2_K wo_a path ----------------------------

@pytest.mark.parametrize("groups,R,Kg,m", [(8, 512, 2048, 1), (8, 512, 2048, 4), (8, 512, 2048, 8),
                                           (3, 45, 768, 2), (160, 16, 256, 1)])
def test_grouped_mmvq(lib, groups, R, Kg, m):
    """og[t, g*R + r] = o_g . W[g*R + r] against the oracle's projection of
    each group (the q8_1 values the input rows encode); m = 1 also against
    single calls on each group's row block, bit for bit.  (3, 45, 768): rows
    that are not 16-byte aligned; 160 groups: more groups than SMs."""
    W = synth.q2k_matrix(8, f"grp.{groups}.{R}.{Kg}", groups * R, Kg)
    x = synth.bf16_normal(8, f"grp.x.{m}.{groups * Kg}", (m, groups * Kg))
    xq = oracle.q8_1_quantize(x)
    y = lib.q2k_mmvq_grouped(dev(W), groups, R, Kg, dev(xq)).cpu().numpy()
    xf = oracle.q8_1_dequant(xq, m, groups * Kg)
    rb = W.nbytes // (groups * R)  # bytes per row
    for g in range(groups):
        Wg = W.reshape(groups * R, rb)[g * R:(g + 1) * R]
        ref = oracle.matvec(np.ascontiguousarray(Wg), R, Kg, np.ascontiguousarray(xf[:, g * Kg:(g + 1) * Kg]))
        assert rel_err_rows(y[:, g * R:(g + 1) * R], ref) <= 1e-4, g
    if m == 1:
        q8b = xq.reshape(-1)
        for g in sorted({0, groups // 2, groups - 1}):
            Wg = np.ascontiguousarray(W.reshape(groups * R, rb)[g * R:(g + 1) * R])
            xg = np.ascontiguousarray(q8b[g * (Kg // 32) * 36:(g + 1) * (Kg // 32) * 36]).reshape(1, -1)
            single = lib.q2k_mmvq_q8_1(dev(Wg), dev(xg), Kg).cpu().numpy()
            np.testing.assert_array_equal(y[:, g * R:(g + 1) * R], single)


@pytest.mark.parametrize("m,act", [(3, "bf16"), (8, "q8_1")])
def test_tensor_core_mmvq_in_waves(lib, m, act):
    """1537 row tiles: more than eight per CTA on one CTA per SM, so the
    tensor-core MMVQ runs more CTAs than SMs, in waves; a ragged last tile."""
    N, K = 24577, 2048
    W = synth.q2k_matrix(14, "mt.waves", N, K)
    x = synth.bf16_normal(14, f"mt.waves.x{m}", (m, K))
    rows = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 40, N)]))
    Ws = np.ascontiguousarray(W[rows])
    if act == "bf16":
        y = lib.q2k_gemv_bf16(dev(W), bf16_dev(x)).cpu().numpy()
        assert rel_err_rows(y[:, rows], oracle.matvec(Ws, len(rows), K, x_f64(x))) <= TOL_BF16
    else:
        xq = lib.q8_1_quantize_rows(bf16_dev(x))
        y = lib.q2k_mmvq_q8_1(dev(W), xq, K).cpu().numpy()
        ref = oracle.matvec(Ws, len(rows), K, oracle.q8_1_dequant(xq.cpu().numpy(), m, K))
        assert rel_err_rows(y[:, rows], ref) <= 1e-4


# ---- a6: routed experts -------------------------------------------------------------

@pytest.mark.parametrize("per_matrix", [False, True])
def test_experts_rows_equal_singles_and_weighted_sum(lib, per_matrix):
    n_mat, N, K = 5, 300, 512
    mats = [dev(synth.q2k_matrix(2, f"ex.{e}", N, K)) for e in range(n_mat)]
    rows = n_mat if per_matrix else 1
    x = synth.bf16_normal(2, f"ex.x{rows}", (rows, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    w = np.float32([0.1, 0.3, 0.05, 0.25, 0.3])
    wt = dev(w)
    tbl = lib.pointer_table(mats)
    ysum = torch.empty(N, dtype=torch.float32, device="cuda")
    y, _ = lib.q2k_mmvq_experts(tbl, N, K, xq, x_per_matrix=per_matrix, route_w=wt, y_sum=ysum)
    for e in range(n_mat):
        xe = xq[e:e + 1] if per_matrix else xq
        assert torch.equal(y[e:e + 1], lib.q2k_mmvq_q8_1(mats[e], xe, K)), e
    yh = y.cpu().numpy().astype(np.float64)
    ref = (w.astype(np.float64)[:, None] * yh).sum(0)
    assert np.max(np.abs(ysum.cpu().numpy() - ref)) <= 1e-5 * np.linalg.norm(ref)
    # only the sum
    ys2 = torch.empty(N, dtype=torch.float32, device="cuda")
    lib.q2k_mmvq_experts(tbl, N, K, xq, x_per_matrix=per_matrix, route_w=wt, y_sum=ys2, want_y=False)
    assert torch.equal(ys2, ysum)


@pytest.mark.parametrize("n_mat,N,K,fused", [(160, 64, 256, False), (3, 4096, 2048, True), (24, 300, 1024, True),
                                             (4, 200, 8192, True), (5, 700, 3840, True), (3, 333, 2304, False)])
def test_experts_one_matrix_per_cta_equals_fused_sum(lib, n_mat, N, K, fused):
    """Per-matrix inputs with y given take one matrix per group of CTAs (more
    matrices than SMs: several waves) and a separate weighted sum; without y
    the sum is fused into the GEMV.  Same bits where both apply (the fused
    path keeps every matrix's partial sums of its rows in shared memory, so
    it does not take 160 matrices)."""
    mats = [dev(synth.q2k_matrix(4, f"exm.{n_mat}.{e}", N, K)) for e in range(n_mat)]
    x = synth.bf16_normal(4, f"exm.x{n_mat}", (n_mat, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    w = np.random.default_rng(n_mat).random(n_mat).astype(np.float32)
    wt = dev(w)
    tbl = lib.pointer_table(mats)
    ysum = torch.empty(N, dtype=torch.float32, device="cuda")
    y, _ = lib.q2k_mmvq_experts(tbl, N, K, xq, x_per_matrix=True, route_w=wt, y_sum=ysum)
    for e in sorted({0, n_mat // 2, n_mat - 1}):
        assert torch.equal(y[e:e + 1], lib.q2k_mmvq_q8_1(mats[e], xq[e:e + 1], K)), e
    if fused:
        ys2 = torch.empty(N, dtype=torch.float32, device="cuda")
        lib.q2k_mmvq_experts(tbl, N, K, xq, x_per_matrix=True, route_w=wt, y_sum=ys2, want_y=False)
        assert torch.equal(ys2, ysum)
    ref = (w.astype(np.float64)[:, None] * y.cpu().numpy().astype(np.float64)).sum(0)
    assert np.max(np.abs(ysum.cpu().numpy() - ref)) <= 1e-5 * np.linalg.norm(ref)
    # matrix 0's rows against the oracle (8-word slices from 8 blocks per row
    # for one q8_1 token, 4-word below)
    W0 = mats[0].cpu().numpy()
    x0 = oracle.q8_1_dequant(xq[0:1].cpu().numpy(), 1, K)
    assert rel_err_rows(y[0:1].cpu().numpy(), oracle.matvec(W0, N, K, x0)) <= 1e-4


def test_experts_fused_sum_too_big_is_refused_before_any_launch(lib):
    """Without y the fused sum keeps every matrix's partial sums of a CTA's
    rows in shared memory; a batch whose partials cannot fit returns
    Q2K_ERR_WORKSPACE at the call, and y_sum is left untouched."""
    import ctypes
    n_mat, N, K = 160, 64, 256
    mats = [dev(synth.q2k_matrix(4, f"exm.{n_mat}.{e}", N, K)) for e in range(n_mat)]
    xq = lib.q8_1_quantize_rows(bf16_dev(synth.bf16_normal(4, f"exm.x{n_mat}", (n_mat, K))))
    wt = torch.full((n_mat,), 0.5, dtype=torch.float32, device="cuda")
    tbl = lib.pointer_table(mats)
    ysum = torch.full((N,), 7.0, dtype=torch.float32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.lib().q2k_mmvq_experts(P(tbl), n_mat, N, K, P(xq), 1, None, P(wt), P(ysum),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 6  # Q2K_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(ysum == 7.0)
    # with y as the workspace the same batch runs
    y, _ = lib.q2k_mmvq_experts(tbl, N, K, xq, x_per_matrix=True, route_w=wt, y_sum=ysum)
    ref = 0.5 * y.double().sum(0)
    assert torch.max(torch.abs(ysum.double() - ref)) <= 1e-5 * torch.linalg.norm(ref)


def test_swiglu_q8_1_against_oracle(lib):
    E, N = 3, 2048
    g = np.random.default_rng(3).standard_normal((2 * E, N)).astype(np.float32) * 2
    gu = dev(g)
    h16 = torch.empty((E, N), dtype=torch.bfloat16, device="cuda")
    hq, _ = lib.swiglu_q8_1_rows(gu, h_bf16=h16)
    got16 = host_bits(h16)
    gb = x_f64(oracle.round_bf16(g[:E].astype(np.float64)))
    ub = x_f64(oracle.round_bf16(g[E:].astype(np.float64)))
    ref16 = oracle.round_bf16(oracle.swiglu(gb, ub))
    # silu in fp32 vs fp64: at most one bf16 step apart
    diff = np.abs(got16.astype(np.int32) - ref16.astype(np.int32))
    same_sign = (got16 >> 15) == (ref16 >> 15)
    assert np.all((diff <= 1) & same_sign | (got16 == ref16))
    np.testing.assert_array_equal(hq.cpu().numpy(), oracle.q8_1_quantize(got16))


@pytest.fixture(scope="module")
def cfg3():
    E_all, topk, dim, inter = 256, 8, 4096, 2048
    mats = {}
    dev_mats = {}
    for e in range(E_all):
        for kind, shape in (("gate", (inter, dim)), ("up", (inter, dim)), ("down", (dim, inter))):
            a = synth.q2k_matrix(0, f"cfg3.{kind}{e}", *shape)
            dev_mats[(kind, e)] = dev(a)
            mats[(kind, e)] = a
    ids, w = synth.expert_route(0, E_all, topk)
    x = synth.bf16_normal(0, "cfg3.x", (1, dim))
    return dict(mats=mats, dev=dev_mats, ids=ids, w=w, x=x, dim=dim, inter=inter, topk=topk)


def test_moe_m1_cfg3(lib, cfg3):
    c = cfg3
    ids, w = c["ids"], c["w"]
    ptrs = [c["dev"][("gate", int(e))] for e in ids] + [c["dev"][("up", int(e))] for e in ids] + \
           [c["dev"][("down", int(e))] for e in ids]
    tbl = lib.pointer_table(ptrs)
    y, ws = lib.q2k_moe_m1(tbl, len(ids), c["dim"], c["inter"], bf16_dev(c["x"][0]), dev(w))
    y = y.cpu().numpy()
    gate = [c["mats"][("gate", int(e))] for e in ids]
    up = [c["mats"][("up", int(e))] for e in ids]
    down = [c["mats"][("down", int(e))] for e in ids]
    ref = oracle.moe_m1(c["x"], gate, up, down, w, c["dim"], c["inter"])
    assert rel_err_rows(y, ref["y"]) <= TOL_Q8
    refq = oracle.moe_m1(c["x"], gate, up, down, w, c["dim"], c["inter"], quantized=True)
    assert rel_err_rows(y, refq["y"]) <= 2e-3
    # the chain equals its steps run one by one
    xq = lib.q8_1_quantize_rows(bf16_dev(c["x"]))
    gu, _ = lib.q2k_mmvq_experts(lib.pointer_table(ptrs[:16]), c["inter"], c["dim"], xq)
    hq, _ = lib.swiglu_q8_1_rows(gu)
    ys = torch.empty(c["dim"], dtype=torch.float32, device="cuda")
    lib.q2k_mmvq_experts(lib.pointer_table(ptrs[16:]), c["dim"], c["inter"], hq, x_per_matrix=True,
                         route_w=dev(w), y_sum=ys, want_y=False)
    np.testing.assert_array_equal(ys.cpu().numpy(), y)


def _moe_steps(lib, ptrs, E, dim, inter, x, w):
    """The step run one call at a time: q8_1 of x, the gate/up batch, SwiGLU
    + q8_1, the down batch with the route-weighted sum."""
    xq = lib.q8_1_quantize_rows(x.view(1, dim))
    gu, _ = lib.q2k_mmvq_experts(lib.pointer_table(ptrs[:2 * E]), inter, dim, xq)
    hq, _ = lib.swiglu_q8_1_rows(gu)
    ys = torch.empty(dim, dtype=torch.float32, device="cuda")
    lib.q2k_mmvq_experts(lib.pointer_table(ptrs[2 * E:]), dim, inter, hq, x_per_matrix=True, route_w=w,
                         y_sum=ys, want_y=False)
    return ys


# (E, dim, inter): both batches on 8-word slices (rows of 9 and 8 blocks, and
# the configuration's 16 and 8), and on 4-word slices (rows of 4 and 2 blocks)
@pytest.mark.parametrize("E,dim,inter", [(5, 2304, 2048), (8, 4096, 2048), (3, 1024, 512)])
def test_moe_m1_equals_its_steps_and_the_oracle(lib, E, dim, inter):
    gate = [synth.q2k_matrix(21, f"moe.g{E}.{e}", inter, dim) for e in range(E)]
    up = [synth.q2k_matrix(21, f"moe.u{E}.{e}", inter, dim) for e in range(E)]
    down = [synth.q2k_matrix(21, f"moe.d{E}.{e}", dim, inter) for e in range(E)]
    ptrs = [dev(a) for a in gate + up + down]
    tbl = lib.pointer_table(ptrs)
    x = synth.bf16_normal(21, f"moe.x{E}", (1, dim))
    w = np.random.default_rng(E).dirichlet(np.ones(E)).astype(np.float32)
    xd, wd = bf16_dev(x[0]), dev(w)
    steps = _moe_steps(lib, ptrs, E, dim, inter, xd, wd)
    # a workspace holding garbage, the same workspace again, then x off a
    # 16-byte boundary (its q8_1 in a launch of its own)
    need = lib.q2k_moe_m1_workspace_bytes(E, dim, inter)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, device="cuda")
    for _ in range(3):
        y, _ = lib.q2k_moe_m1(tbl, E, dim, inter, xd, wd, workspace=ws)
        assert torch.equal(y, steps)
    xbuf = torch.zeros(dim + 8, dtype=torch.bfloat16, device="cuda")
    xbuf[1:dim + 1] = xd
    y2, _ = lib.q2k_moe_m1(tbl, E, dim, inter, xbuf[1:dim + 1], wd, workspace=ws)
    assert torch.equal(y2, steps)
    refq = oracle.moe_m1(x, gate, up, down, w, dim, inter, quantized=True)
    assert rel_err_rows(y.cpu().numpy(), refq["y"]) <= 2e-3


# ---- a7: dense GEMM -----------------------------------------------------------------

@pytest.mark.parametrize("m,N,K,pad", [(1, 8, 16, 0), (3, 65, 64, 0), (16, 130, 200, 0), (17, 64, 1024, 0),
                                       (64, 256, 512, 0), (100, 70, 136, 0), (256, 128, 256, 0), (300, 200, 2048, 8),
                                       (40, 1000, 4104, 0), (256, 384, 8192, 16), (16, 4096, 128, 0),
                                       (48, 2000, 320, 0), (600, 300, 192, 0)])
def test_dense_gemm_small(lib, m, N, K, pad):
    x = synth.bf16_normal(9, f"dg.x.{m}.{K}", (m, K + pad))
    W = synth.bf16_normal(9, f"dg.w.{N}.{K}", (N, K), std=0.02)
    xd = bf16_dev(x)[:, :K]  # row stride K + pad
    y = lib.dense_gemm_bf16(xd, bf16_dev(W)).cpu().numpy()
    assert rel_err_rows(y, oracle.dense_gemm(np.ascontiguousarray(x[:, :K]), W)) <= TOL_BF16


def test_engram_cfg1_rows_then_gemm(lib):
    n_table, T, cols, N = 1 << 20, 16, 8, 4096 * 5
    table = synth.q2k_blocks(0, "cfg1.table", n_table)
    ids = synth.row_ids(0, "cfg1.ids", T * cols, n_table)
    wkv = synth.bf16_normal(0, "cfg1.wkv", (N, cols * 256), std=0.02)
    rows = lib.q2k_dequant_rows(dev(table), 256, ids=dev(ids))
    y = lib.dense_gemm_bf16(rows.view(T, cols * 256), bf16_dev(wkv)).cpu().numpy()
    ref_rows, ref_y = oracle.engram_rows_projection(table, n_table, ids, T, cols, wkv)
    np.testing.assert_array_equal(host_bits(rows), ref_rows)
    assert rel_err_rows(y, ref_y) <= TOL_BF16


def test_q2k_gemv_matches_dense_gemm_over_the_expansion(lib):
    # engram_v41.rs `wkv_q2k`: the Q2_K GEMV and the bf16 GEMV over its bf16
    # expansion agree (bit for bit on the page's kernels; here within 2e-3,
    # the two kernels reduce in different orders and the expansion rounds
    # weights to bf16).
    N, K = 512, 4096
    W = synth.q2k_matrix(0, "cfg0.W", N, K)
    x = synth.bf16_normal(0, "cfg0.x", (1, K))
    Wd = dev(W)
    y_q = lib.q2k_gemv_bf16(Wd, bf16_dev(x)).cpu().numpy()
    W16 = lib.q2k_dequant_rows(Wd, K)
    y_d = lib.dense_gemm_bf16(bf16_dev(x), W16).cpu().numpy()
    assert rel_err_rows(y_q, y_d) <= TOL_BF16


def test_repeat_calls_are_bitwise_identical(lib, big_w):
    _, Wd = big_w
    x = bf16_dev(synth.bf16_normal(0, "sweep.x1", (1, 16384)))
    a = lib.q2k_gemv_bf16(Wd, x)
    b = lib.q2k_gemv_bf16(Wd, x)
    assert torch.equal(a, b)
