"""Pins for the CPU oracle: each check compares it with something other than
itself -- the pages' stated facts, library routines (NumPy / SciPy), exact
rational arithmetic, closed forms and invariants -- so that a dropped term,
a wrong sign, index or nibble, or a transposed operand fails one of them.

The Q2_K bit order inside ``qs`` is a reading of the GGUF Q2_K format (the
pages give only the 84-byte size, the field list and the formula); the
bijectivity and one-hot checks below pin its internal consistency, not its
agreement with a real GGUF file (parity unpinned there).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def page_facts():
    facts = {}
    with open(os.path.join(GOLDEN, "page_facts.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                facts[k] = int(v)
    return facts


def make_block(scales, qs, d, dmin):
    b = np.zeros(84, dtype=np.uint8)
    b[0:16] = np.asarray(scales, dtype=np.uint8)
    b[16:80] = np.asarray(qs, dtype=np.uint8)
    b[80:84] = np.array([d, dmin], dtype=np.float16).view(np.uint8)
    return b


# ---- exact rational reference roundings (independent of the oracle's C) ----

def frac_round_even(x: Fraction) -> int:
    fl = math.floor(x)
    r = x - fl
    if r > Fraction(1, 2):
        return fl + 1
    if r < Fraction(1, 2):
        return fl
    return fl if fl % 2 == 0 else fl + 1


def frac_to_binary(x: Fraction, sig_bits: int, emin: int):
    """Nearest value with ``sig_bits`` significand bits (ties to even),
    exponent floor ``emin`` (subnormals below), no overflow handling."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    q = Fraction(2) ** (e - (sig_bits - 1))
    return s * frac_round_even(a / q) * q


def bf16_bits_of(v: Fraction) -> int:
    f = np.float32(float(v))  # v is a bf16 value: exact in fp32
    return int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)


# ---- the pages' stated facts -------------------------------------------------

def test_block_size_is_the_pages_84_bytes():
    facts = page_facts()
    assert oracle.block_bytes() == facts["q2k_block_bytes"] == 84
    assert 16 + 64 + 2 + 2 == facts["q2k_block_bytes"]
    assert facts["q2k_block_weights"] == oracle.Q2K_WEIGHTS
    # a bf16 row of 256 weights takes 512 bytes, against the block's 84
    assert facts["bf16_bytes_per_256"] == 2 * facts["q2k_block_weights"]
    assert oracle.Q8_1_BYTES == 2 + 2 + 32


# ---- scalar formats ----------------------------------------------------------

def test_fp16_decode_matches_numpy_for_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits[finite]])
    np.testing.assert_array_equal(got, ref[finite])


def test_f32_to_fp16_matches_numpy_round_to_nearest_even():
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 5, 4000),
        np.float32(2.0) ** g.integers(-26, 16, 500).astype(np.float32),
        # exact half-way cases between consecutive fp16 values
        (np.arange(1000, 1200, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -10),
        (np.arange(0, 300, dtype=np.float32) + np.float32(0.5)) * np.float32(2.0 ** -24),
        np.array([65504.0, 65519.0, 65520.0, 0.0, -0.0, 6.1e-5, -5.9e-8], dtype=np.float32),
    ])
    vals = vals[np.abs(vals) < np.float32(65520.0)]  # overflow to inf is checked apart
    assert oracle.f32_to_fp16(65520.0) == 0x7C00 and oracle.f32_to_fp16(-1e6) == 0xFC00
    got = np.array([oracle.f32_to_fp16(float(v)) for v in vals], dtype=np.uint16)
    ref = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_f32_to_bf16_is_the_nearest_even_by_exact_arithmetic():
    g = np.random.default_rng(2)
    u = g.integers(0, 2 ** 32, 3000, dtype=np.uint64).astype(np.uint32)
    vals = u.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < np.float32(3e38))]
    ties = (np.arange(200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties[np.isfinite(ties)], np.float32([1e-40, -3e-45, 0.0])])
    for v in vals:
        ref = bf16_bits_of(frac_to_binary(Fraction(float(v)), 8, -126))
        got = oracle.f32_to_bf16(float(v))
        sign = 0x8000 if np.signbit(v) else 0
        assert got == (ref | sign), (float(v), hex(got), hex(ref))


# ---- Q2_K decode -------------------------------------------------------------

def test_all_codes_three_gives_closed_form_per_subblock():
    # Every 2-bit code = 3, so the layout of qs does not matter; sub-block j
    # (16 consecutive weights) uses scales[j]: low nibble scale, high min.
    sc = np.arange(16) % 16
    mn = (15 - np.arange(16)) % 16
    d, dmin = 0.5, 0.125
    blk = make_block((mn << 4) | sc, np.full(64, 0xFF), d, dmin)
    w = oracle.decode_block(blk)
    p = np.arange(256)
    np.testing.assert_array_equal(w, 3 * d * sc[p // 16] - dmin * mn[p // 16])


def test_all_codes_zero_gives_minus_min():
    sc = np.full(16, 7)
    mn = np.arange(16)
    blk = make_block((mn << 4) | sc, np.zeros(64), 2.0, 0.25)
    w = oracle.decode_block(blk)
    np.testing.assert_array_equal(w, -0.25 * np.repeat(mn, 16))


def test_d_and_dmin_fields_are_not_swapped():
    blk = make_block(np.full(16, (1 << 4) | 1), np.full(64, 0x55), 4.0, 1.0)  # codes 1
    assert np.all(oracle.decode_block(blk) == 4.0 * 1 * 1 - 1.0 * 1)


def test_each_qs_bit_drives_exactly_one_weight_and_all_256_are_covered():
    low, high = [], []
    for byte in range(64):
        for bit in range(8):
            qs = np.zeros(64, dtype=np.uint8)
            qs[byte] = 1 << bit
            w = oracle.decode_block(make_block(np.full(16, 1), qs, 1.0, 0.0))
            nz = np.flatnonzero(w)
            assert len(nz) == 1
            val = w[nz[0]]
            assert val == (1.0 if bit % 2 == 0 else 2.0)
            (low if bit % 2 == 0 else high).append(int(nz[0]))
            # the low and high bit of one code land on the same weight
            if bit % 2 == 1:
                assert high[-1] == low[-1]
    assert sorted(low) == list(range(256))
    assert sorted(high) == list(range(256))


def test_one_hot_code_reading():
    # Reading of the GGUF layout: weight p takes bits 2*((p%128)//32) of
    # qs[32*(p//128) + p%32].  A one-hot code decodes to the unit vector.
    for p in range(256):
        qs = np.zeros(64, dtype=np.uint8)
        qs[32 * (p // 128) + p % 32] = 1 << (2 * ((p % 128) // 32))
        w = oracle.decode_block(make_block(np.full(16, 1), qs, 1.0, 0.0))
        e = np.zeros(256)
        e[p] = 1.0
        np.testing.assert_array_equal(w, e)


def test_scale_byte_affects_sixteen_consecutive_weights():
    base = synth.q2k_blocks(0, "pin.scales", 1)[0]
    w0 = oracle.decode_block(base)
    for j in range(16):
        b = base.copy()
        b[j] ^= 0x11
        changed = np.flatnonzero(oracle.decode_block(b) != w0)
        assert set(changed) <= set(range(16 * j, 16 * j + 16))
        assert len(changed) > 0


def test_decode_bf16_is_exact_value_rounded_once_to_f32_then_bf16():
    blocks = synth.q2k_blocks(3, "pin.bf16", 6)
    # add extreme d/dmin combinations (subnormal and large fp16)
    extra = []
    for d, dm in [(6.1e-5, 60000.0), (60000.0, 5.96e-8), (1e-7, 1e-7), (1000.0, 3.0)]:
        b = blocks[0].copy()
        b[80:84] = np.array([d, dm], dtype=np.float16).view(np.uint8)
        extra.append(b)
    for blk in list(blocks) + extra:
        rows, bad = oracle.dequant_rows(blk, 1, 256, None, 1)
        assert bad == 0
        d = Fraction(float(blk[80:82].view(np.float16)[0]))
        dm = Fraction(float(blk[82:84].view(np.float16)[0]))
        w_exact = oracle.decode_block(blk)
        for p in range(0, 256, 7):
            j = p // 16
            sc, mn = int(blk[j]) & 15, int(blk[j]) >> 4
            byte = int(blk[16 + 32 * (p // 128) + p % 32])
            q = (byte >> (2 * ((p % 128) // 32))) & 3
            exact = d * sc * q - dm * mn
            f32 = frac_to_binary(exact, 24, -126)
            ref = bf16_bits_of(frac_to_binary(f32, 8, -126))
            if exact < 0 and ref == 0:
                ref = 0x8000
            assert int(rows[0, p]) == ref, (p, float(exact))
            # the fp64 decode is exact whenever the products span <= 53 bits
            if abs(float(d)) > 0 and abs(float(dm)) > 0 and max(d, dm) / min(d, dm) < 2 ** 30:
                assert Fraction(w_exact[p]) == exact


def test_dequant_rows_gather_equals_contiguous_copy_and_flags_bad_ids():
    K = 512
    table = synth.q2k_matrix(4, "pin.table", 10, K)
    ids = np.array([3, 3, 0, 9, 5], dtype=np.int32)
    got, bad = oracle.dequant_rows(table, 10, K, ids, len(ids))
    assert bad == 0
    ref, _ = oracle.dequant_rows(np.ascontiguousarray(table[ids]), len(ids), K, None, len(ids))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(got[0], got[1])
    got2, bad2 = oracle.dequant_rows(table, 10, K, np.array([1, -1, 10, 2], np.int32), 4)
    assert bad2 == 2
    assert not got2[1].any() and not got2[2].any()
    row1, _ = oracle.dequant_rows(table, 10, K, np.array([1], np.int32), 1)
    np.testing.assert_array_equal(got2[0], row1[0])


# ---- q8_1 --------------------------------------------------------------------

def q8_fields(xq, m, K):
    blk = xq.reshape(m, K // 32, 36)
    d = blk[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float32)
    s = blk[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float32)
    q = blk[..., 4:].view(np.int8).astype(np.int32)
    return d, s, q


def test_q8_1_invariants_on_random_rows():
    m, K = 3, 1024
    x = synth.bf16_normal(5, "pin.q8", (m, K))
    xq = oracle.q8_1_quantize(x)
    d, s, q = q8_fields(xq, m, K)
    xv = synth.bf16_bits_to_f32(x).reshape(m, K // 32, 32)
    amax = np.abs(xv).max(axis=-1)
    d32 = (amax / np.float32(127.0)).astype(np.float32)
    assert np.all(np.abs(q) <= 127)
    assert np.all(np.abs(q).max(axis=-1) == 127)
    # |x - d32 q| <= d32/2, up to the one fp32 rounding of x/d32 (half an
    # ulp of a value below 128, i.e. 2^-17)
    err = np.abs(xv.astype(np.float64) - d32[..., None].astype(np.float64) * q)
    assert np.all(err <= d32[..., None].astype(np.float64) * (0.5 + 2.0 ** -17))
    # stored d is fp16(d32) (NumPy's round-to-nearest-even cast)
    np.testing.assert_array_equal(d, d32.astype(np.float16).astype(np.float32))
    # s = fp16(f32(d) * sum q)
    sref = (d * q.sum(axis=-1).astype(np.float32)).astype(np.float32).astype(np.float16).astype(np.float32)
    np.testing.assert_array_equal(s, sref)


def test_q8_1_rounds_half_away_from_zero_and_zero_block():
    vals = np.zeros(64, dtype=np.float32)
    vals[:8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5]
    x = synth.f32_to_bf16_bits(vals)[None, :]
    d, s, q = q8_fields(oracle.q8_1_quantize(x), 1, 64)
    assert d[0, 0] == 1.0
    assert list(q[0, 0, :8]) == [127, 3, -3, 1, -1, 2, -2, 127]
    assert d[0, 1] == 0.0 and s[0, 1] == 0.0 and not q[0, 1].any()


def test_q8_1_power_of_two_scaling_is_exact():
    x = synth.bf16_normal(6, "pin.q8s", (2, 256))
    x2 = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x) * np.float32(2.0))
    d1, _, q1 = q8_fields(oracle.q8_1_quantize(x), 2, 256)
    d2, _, q2 = q8_fields(oracle.q8_1_quantize(x2), 2, 256)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(d2, 2 * d1)


def test_q8_1_dequant_is_d_times_q():
    x = synth.bf16_normal(7, "pin.q8d", (2, 128))
    xq = oracle.q8_1_quantize(x)
    d, _, q = q8_fields(xq, 2, 128)
    np.testing.assert_array_equal(oracle.q8_1_dequant(xq, 2, 128),
                                  (d[..., None].astype(np.float64) * q).reshape(2, 128))


# ---- projections -----------------------------------------------------------------

@pytest.mark.parametrize("N,K,m", [(1, 256, 1), (3, 512, 2), (5, 256, 8), (4, 768, 3)])
def test_matvec_equals_numpy_matmul_of_decoded_matrix(N, K, m):
    W = synth.q2k_matrix(8, f"pin.mv{N}x{K}", N, K)
    x = synth.bf16_bits_to_f32(synth.bf16_normal(8, f"pin.mvx{m}", (m, K))).astype(np.float64)
    Wd = oracle.decode_matrix(W, N, K)
    np.testing.assert_allclose(oracle.matvec(W, N, K, x), x @ Wd.T, rtol=1e-12, atol=1e-12)


def test_matvec_unit_vector_selects_one_column_exactly():
    N, K = 5, 512
    W = synth.q2k_matrix(9, "pin.col", N, K)
    Wd = oracle.decode_matrix(W, N, K)
    for k in (0, 1, 17, 255, 256, 300, 511):
        x = np.zeros((1, K))
        x[0, k] = 1.0
        np.testing.assert_array_equal(oracle.matvec(W, N, K, x)[0], Wd[:, k])


def test_matvec_rows_are_independent_blocks():
    # a row's output depends only on its own blocks: permuting rows of W
    # permutes y.
    N, K = 4, 512
    W = synth.q2k_matrix(10, "pin.perm", N, K)
    x = np.random.default_rng(0).standard_normal((2, K))
    perm = [2, 0, 3, 1]
    np.testing.assert_array_equal(oracle.matvec(W[perm], N, K, x), oracle.matvec(W, N, K, x)[:, perm])


def test_dense_gemm_matches_numpy_matmul():
    x = synth.bf16_normal(11, "pin.gx", (3, 96))
    W = synth.bf16_normal(11, "pin.gw", (7, 96), std=0.02)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(W).astype(np.float64).T
    np.testing.assert_allclose(oracle.dense_gemm(x, W), ref, rtol=1e-13, atol=1e-15)


def test_silu_matches_scipy_and_odd_identity():
    from scipy.special import expit
    z = np.linspace(-30, 30, 601)
    got = np.array([oracle.silu(v) for v in z])
    np.testing.assert_allclose(got, z * expit(z), rtol=1e-14, atol=1e-300)
    # silu(z) - silu(-z) = z
    np.testing.assert_allclose(got - got[::-1], z, atol=1e-12)
    assert oracle.silu(0.0) == 0.0


def test_weighted_sum_matches_numpy_and_one_hot_selects():
    v = np.random.default_rng(1).standard_normal((4, 9))
    w = np.array([0.1, 0.2, 0.3, 0.4], dtype=np.float32)
    np.testing.assert_allclose(oracle.weighted_sum(v, w), w.astype(np.float64) @ v, rtol=1e-14)
    np.testing.assert_array_equal(oracle.weighted_sum(v, np.float32([0, 0, 1, 0])), v[2])


def test_moe_chain_single_expert_and_quantised_agreement():
    dim, inter = 256, 256
    gate = [synth.q2k_matrix(12, f"pin.g{e}", inter, dim) for e in range(2)]
    up = [synth.q2k_matrix(12, f"pin.u{e}", inter, dim) for e in range(2)]
    down = [synth.q2k_matrix(12, f"pin.d{e}", dim, inter) for e in range(2)]
    x = synth.bf16_normal(12, "pin.x", (1, dim))
    both = oracle.moe_m1(x, gate, up, down, np.float32([1.0, 0.0]), dim, inter)
    one = oracle.moe_m1(x, gate[:1], up[:1], down[:1], np.float32([1.0]), dim, inter)
    np.testing.assert_array_equal(both["y"], one["y"])
    # swapping expert order together with the weights leaves y unchanged
    w = np.float32([0.3, 0.7])
    a = oracle.moe_m1(x, gate, up, down, w, dim, inter)["y"]
    b = oracle.moe_m1(x, gate[::-1], up[::-1], down[::-1], w[::-1], dim, inter)["y"]
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    q = oracle.moe_m1(x, gate, up, down, w, dim, inter, quantized=True)["y"]
    assert np.max(np.abs(q - a)) / np.linalg.norm(a) < 1e-2


# ---- the MoE chain on hand-built experts, written out in closed form ------------
#
# moe_v41/init.rs, MoeV41::new: gate and up form one expert batch over the
# shared x, SwiGLU of (gate, up) is requantised to q8_1, the down batch reads
# expert e's own h row, and the outputs are summed with the route weights.
# The experts below are built so that every intermediate has a closed form:
#   gate/up: every code 3, every sub-block scale 1 and min 0, dmin 0, so each
#            weight of row i is 3*d_i; with x = e_k, g[i] = 3*d_i exactly;
#            d is constant over each run of 32 rows (one q8_1 block of h);
#   down:    row r holds a single weight 1, at column perm_e[r], so
#            down_e[r] = h_e[perm_e[r]].
# The d values use the full fp16 significand, so 3*d is not a bf16 value
# and every bf16 rounding point changes the result.

def _const_rows_q2k(d_rows, K):
    nb = K // 256
    rows = len(d_rows)
    b = np.zeros((rows, nb, 84), dtype=np.uint8)
    b[:, :, 0:16] = 0x01   # scale 1, min 0
    b[:, :, 16:80] = 0xFF  # every code 3
    b[:, :, 80:82] = np.asarray(d_rows, dtype=np.float16).view(np.uint8).reshape(rows, 1, 2)
    return b.reshape(-1)


def _permutation_q2k(cols, K):
    """Row r has weight 1 at column cols[r], 0 elsewhere (d = 1, dmin = 0)."""
    nb = K // 256
    b = np.zeros((len(cols), nb, 84), dtype=np.uint8)
    for r, c in enumerate(cols):
        blk = b[r, c // 256]
        p = c % 256
        blk[p // 16] = 0x01
        blk[16 + 32 * (p // 128) + p % 32] |= np.uint8(1 << (2 * ((p % 128) // 32)))
        blk[80:82] = np.array([1.0], dtype=np.float16).view(np.uint8)
    return b.reshape(-1)


def _bf16(v: float) -> Fraction:
    """fp64 -> fp32 -> bf16, each step round to nearest even (exact rationals)."""
    return frac_to_binary(frac_to_binary(Fraction(v), 24, -126), 8, -126)


def _q8_1_const_block(v: float) -> float:
    """The value a q8_1 block whose 32 entries all equal v decodes to:
    amax = |v|, d32 = amax/127 (fp32 divide), q = round(v/d32) = +-127,
    stored d = fp16(d32); the decoded entry is f32(d) * q."""
    if v == 0.0:
        return 0.0
    d32 = np.float32(abs(v)) / np.float32(127.0)
    q = float(np.round(np.float32(v) / d32))
    assert abs(q) == 127.0
    return float(np.float16(d32)) * q


def _moe_hand_case(seed=5, E=3, dim=512, inter=512):
    g = np.random.default_rng(seed)
    groups = inter // 32
    dg = (g.uniform(0.1, 0.9, (E, groups)) * g.choice([-1.0, 1.0], (E, groups))).astype(np.float16)
    du = (g.uniform(0.1, 0.9, (E, groups)) * g.choice([-1.0, 1.0], (E, groups))).astype(np.float16)
    perms = [g.permutation(inter)[:dim] if dim <= inter else g.integers(0, inter, dim) for _ in range(E)]
    gate = [_const_rows_q2k(np.repeat(dg[e], 32), dim) for e in range(E)]
    up = [_const_rows_q2k(np.repeat(du[e], 32), dim) for e in range(E)]
    down = [_permutation_q2k(perms[e], inter) for e in range(E)]
    k = int(g.integers(0, dim))
    x = np.zeros((1, dim), dtype=np.uint16)
    x[0, k] = 0x3F80  # bf16 1.0
    w = np.array(g.dirichlet(np.ones(E)), dtype=np.float32)
    return dict(E=E, dim=dim, inter=inter, dg=dg, du=du, perms=perms, gate=gate, up=up, down=down, x=x, w=w)


def _moe_expected(c, quantized):
    """The chain written out: g, u rounded to bf16, h = bf16(silu(g) * u),
    (q8_1 of x and of h when quantized), down_e = h_e[perm_e], y = sum_e w_e down_e."""
    # x = e_k: its q8_1 block has amax 1, so x_k decodes as a constant block of 1s would
    xk = _q8_1_const_block(1.0) if quantized else 1.0
    out = {"g": [], "u": [], "h": [], "down": []}
    y = np.zeros(c["dim"])
    for e in range(c["E"]):
        g = np.repeat(3.0 * c["dg"][e].astype(np.float64) * xk, 32)
        u = np.repeat(3.0 * c["du"][e].astype(np.float64) * xk, 32)
        g16 = np.array([float(_bf16(v)) for v in g])
        u16 = np.array([float(_bf16(v)) for v in u])
        silu = g16 / (1.0 + np.exp(-g16))
        h = np.array([float(_bf16(v)) for v in silu * u16])
        hin = np.array([_q8_1_const_block(v) for v in h]) if quantized else h
        dn = hin[c["perms"][e]]
        y = y + np.float64(c["w"][e]) * dn
        for key, v in (("g", g), ("u", u), ("h", h), ("down", dn)):
            out[key].append(v)
    out["y"] = y
    return out


@pytest.mark.parametrize("quantized", [False, True])
def test_moe_chain_on_hand_built_experts_matches_closed_form(quantized):
    """Fails if silu lands on u instead of g, if a bf16 rounding of g, u or h
    is dropped, if the down batch reads another expert's h (or reads h
    through a transposed matrix), or if the route weights are misassigned."""
    c = _moe_hand_case()
    got = oracle.moe_m1(c["x"], c["gate"], c["up"], c["down"], c["w"], c["dim"], c["inter"], quantized=quantized)
    exp = _moe_expected(c, quantized)
    np.testing.assert_array_equal(got["g"], np.stack(exp["g"]))
    np.testing.assert_array_equal(got["u"], np.stack(exp["u"]))
    np.testing.assert_array_equal(oracle.bf16_to_f64(got["h_bits"]), np.stack(exp["h"]))
    np.testing.assert_array_equal(got["down"], np.stack(exp["down"]))
    np.testing.assert_allclose(got["y"], exp["y"], rtol=1e-15, atol=0)
    # every rounding point and role matters on this case: the alternatives differ
    g16 = np.array([float(_bf16(v)) for v in exp["g"][0]])
    u16 = np.array([float(_bf16(v)) for v in exp["u"][0]])
    assert not np.array_equal(g16, exp["g"][0]) and not np.array_equal(u16, exp["u"][0])
    assert not np.allclose(g16 / (1 + np.exp(-g16)) * u16, u16 / (1 + np.exp(-u16)) * g16, rtol=1e-3)


# ---- engram n-gram hash (engram_v41.rs, EngramHasher::hash) ---------------------

_HASH_ARGS = dict(max_ngram=3, n_layers=2, n_heads=2,
                  multipliers=np.array([[3, 5, 7], [11, 13, 17]], dtype=np.int64),
                  primes=np.array([[[101, 103], [107, 109]], [[113, 127], [131, 137]]], dtype=np.int64),
                  offsets=np.zeros((2, 4), dtype=np.int64), pad_id=0)


def test_engram_hash_hand_computed():
    # token_map[i] = 3i + 1; tokens 5, 7, 9 -> 16, 22, 28; pad 0.
    # pos 0: [16, pad, pad]: 16*3 = 48 for both lengths.
    # pos 1: [22, 16, pad]: 66 ^ 80 = 18.
    # pos 2: [28, 22, 16]: 84 ^ 110 = 58, then 58 ^ 112 = 74.
    tm = np.arange(100, dtype=np.int64) * 3 + 1
    out = oracle.engram_hash(tm, np.zeros(8, np.int64), [5, 7, 9], 0, **_HASH_ARGS)
    np.testing.assert_array_equal(out[:, 0, :], [[48, 48, 48, 48], [18, 18, 18, 18], [58, 58, 74, 74]])
    # layer 1, pos 0: 16*11 = 176 -> 176 mod 113 = 63, mod 127 = 49, mod 131 = 45, mod 137 = 39
    np.testing.assert_array_equal(out[0, 1, :], [63, 49, 45, 39])


def test_engram_hash_wrapping_products_and_euclidean_remainder():
    # 2^62 * 2 wraps to -2^63: the remainder is the Euclidean one, in [0, p)
    tm = np.array([1 << 62], dtype=np.int64)
    args = dict(_HASH_ARGS, max_ngram=2, n_layers=1, n_heads=1, multipliers=np.array([[2, 0]], np.int64),
                primes=np.array([[[101]]], np.int64), offsets=np.array([[7]], np.int64))
    out = oracle.engram_hash(tm, np.zeros(4, np.int64), [0], 0, **args)
    assert out[0, 0, 0] == 7 + (101 - pow(2, 63, 101)) % 101
    # 2^62 * 4 wraps to 0
    args["multipliers"] = np.array([[4, 0]], np.int64)
    assert oracle.engram_hash(tm, np.zeros(4, np.int64), [0], 0, **args)[0, 0, 0] == 7


def test_engram_hash_ranges_blocking_and_incremental_calls():
    rng = np.random.default_rng(5)
    tm = rng.integers(0, 1 << 40, size=500).astype(np.int64)
    tm[13] = -1  # an unmapped token blocks every shift that reaches it
    args = dict(_HASH_ARGS, max_ngram=4, n_layers=2, n_heads=3,
                multipliers=rng.integers(-(1 << 62), 1 << 62, size=(2, 4)).astype(np.int64),
                primes=rng.integers(1000, 1 << 30, size=(2, 3, 3)).astype(np.int64),
                offsets=rng.integers(0, 1 << 20, size=(2, 9)).astype(np.int64), pad_id=99)
    ids = rng.integers(0, 500, size=12).astype(np.uint32)
    ids[6] = 13
    out = oracle.engram_hash(tm, np.zeros(16, np.int64), ids, 0, **args)
    lo = args["offsets"][None, :, :]
    hi = lo + np.repeat(args["primes"].reshape(2, 3, 3), 1, axis=1).reshape(2, 9)[None]
    assert np.all(out >= lo) and np.all(out < hi)
    # positions 6..8 see the unmapped token at shift pos-6: shifts from there on read pad,
    # so pos 6 equals the hash of an all-pad n-gram
    pad_only = oracle.engram_hash(np.array([99], np.int64), np.zeros(4, np.int64), [0], 0, **args)
    np.testing.assert_array_equal(out[6], pad_only[0])
    # the cache carries the sequence: one call of 12 equals calls of 5 and 7
    cache = np.zeros(16, np.int64)
    a = oracle.engram_hash(tm, cache, ids[:5], 0, **args)
    b = oracle.engram_hash(tm, cache, ids[5:], 5, **args)
    np.testing.assert_array_equal(np.concatenate([a, b]), out)
    # errors as on the page
    with pytest.raises(ValueError):
        oracle.engram_hash(tm, np.zeros(16, np.int64), [600], 0, **args)
    with pytest.raises(ValueError):
        oracle.engram_hash(tm, np.zeros(4, np.int64), ids[:5], 0, **args)
    np.testing.assert_array_equal(oracle.layer_row_ids(out, 1), out[:, 1, :].reshape(-1))


# ---- Q3_K (moe_v41/init.rs, `MoeV41::new`, names the Q3_K MMVQ kernels; the
# block layout is GGUF's Q3_K, a reading: hmask[32] | qs[64] | scales[12] | d) ----

def make_q3k_block(scales6, codes, d):
    """Pack 16 six-bit scales (0..63, stored +32) and 256 codes (-4..3) the
    way GGUF's Q3_K quantiser lays them out."""
    b = np.zeros(110, dtype=np.uint8)
    for j, s in enumerate(scales6):
        s = int(s)
        if j < 8:
            b[96 + j] |= s & 15
        else:
            b[96 + j - 8] |= (s & 15) << 4
        b[96 + 8 + j % 4] |= (s >> 4) << (2 * (j // 4))
    for p, c in enumerate(codes):
        L = int(c) + 4
        if L > 3:
            b[p % 32] |= 1 << (p // 32)
        b[32 + 32 * (p // 128) + p % 32] |= (L & 3) << (2 * ((p % 128) // 32))
    b[108:110] = np.array([d], dtype=np.float16).view(np.uint8)
    return b


def test_q3k_block_is_110_bytes():
    assert oracle.q3k_block_bytes() == 32 + 64 + 12 + 2 == 110


def test_q3k_with_every_high_bit_set_is_q2k_without_a_min():
    rng = np.random.default_rng(31)
    for _ in range(20):
        qs = rng.integers(0, 256, 64, dtype=np.uint8)
        nib = rng.integers(0, 16, 16)
        d = float(np.float16(rng.uniform(-0.05, 0.05)))
        q3 = make_q3k_block(32 + nib, np.zeros(256, int), d)
        q3[0:32] = 0xFF
        q3[32:96] = qs
        q2 = make_block(nib, qs, d, 0.0)
        np.testing.assert_array_equal(oracle.q3k_decode_block(q3), oracle.decode_block(q2))


def test_q3k_with_every_high_bit_clear_is_q2k_with_min_four_d_times_scale():
    # code - 4 with the high bit clear: d*s*q - 4*d*s = Q2_K with min nibble s, dmin = 4d
    rng = np.random.default_rng(32)
    for _ in range(20):
        qs = rng.integers(0, 256, 64, dtype=np.uint8)
        nib = rng.integers(0, 16, 16)
        d = float(np.float16(2.0 ** rng.integers(-12, -4)))
        q3 = make_q3k_block(32 + nib, np.zeros(256, int), d)
        q3[0:32] = 0
        q3[32:96] = qs
        q2 = make_block(nib | (nib << 4), qs, d, 4 * d)
        np.testing.assert_array_equal(oracle.q3k_decode_block(q3), oracle.decode_block(q2))


def test_q3k_each_hmask_bit_moves_exactly_one_weight_by_four_steps():
    rng = np.random.default_rng(33)
    scales6 = rng.integers(0, 64, 16)
    codes = rng.integers(-4, 4, 256)
    d = 0.0078125
    base = make_q3k_block(scales6, codes, d)
    w0 = oracle.q3k_decode_block(base)
    hit = np.zeros(256, dtype=int)
    for byte in range(32):
        for bit in range(8):
            blk = base.copy()
            blk[byte] ^= 1 << bit
            diff = oracle.q3k_decode_block(blk) - w0
            (idx,) = np.nonzero(diff)
            step = d * (int(scales6[idx[0] // 16]) - 32) if len(idx) else None
            if scales6[(32 * bit + byte) // 16] == 32:  # a zero scale hides the change
                assert len(idx) == 0
                hit[32 * bit + byte] += 1
                continue
            assert list(idx) == [32 * bit + byte]
            was_set = (base[byte] >> bit) & 1
            assert diff[idx[0]] == (-4 if was_set else 4) * step
            hit[idx[0]] += 1
    assert (hit == 1).all()


def test_q3k_six_bit_scales_round_trip_with_every_value():
    # all 64 stored values over four blocks, each sub-block's weights = d*(s-32)
    perm = np.random.default_rng(34).permutation(64)
    d = 0.25
    for blk_i in range(4):
        s6 = perm[16 * blk_i:16 * blk_i + 16]
        w = oracle.q3k_decode_block(make_q3k_block(s6, np.ones(256, int), d))
        for j in range(16):
            assert (w[16 * j:16 * j + 16] == d * (int(s6[j]) - 32)).all()


def test_q3k_extremes_of_scale_and_code():
    d = 0.5
    w = oracle.q3k_decode_block(make_q3k_block([0] * 8 + [63] * 8, [-4] * 128 + [3] * 128, d))
    assert (w[:128] == d * 128).all()  # (-32) * (-4)
    assert (w[128:] == d * 93).all()   # 31 * 3


@pytest.mark.parametrize("N,K,m", [(1, 256, 1), (3, 512, 2), (5, 256, 8), (4, 768, 3)])
def test_q3k_matvec_equals_numpy_matmul_of_decoded_matrix(N, K, m):
    rng = np.random.default_rng(N * 100 + K + m)
    W = rng.integers(0, 256, N * (K // 256) * 110, dtype=np.uint8).reshape(N, -1)
    for n in range(N):
        for b in range(K // 256):
            W[n, b * 110 + 108:b * 110 + 110] = np.array([rng.uniform(-0.02, 0.02)], np.float16).view(np.uint8)
    x = rng.standard_normal((m, K))
    Wd = oracle.q3k_decode_matrix(W, N, K)
    np.testing.assert_allclose(oracle.q3k_matvec(W, N, K, x), x @ Wd.T, rtol=1e-12, atol=1e-12)
    # block b of row n decodes on its own
    np.testing.assert_array_equal(Wd[N - 1, K - 256:], oracle.q3k_decode_block(W[N - 1, -110:]))


def test_round_bf16_is_fp32_then_bf16_nearest_even():
    # the SwiGLU and expert rows are fp32 values rounded to bf16: the oracle's
    # fp64 -> bf16 goes through fp32 the same way (two round-to-nearest-even steps)
    rng = np.random.default_rng(41)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000),
                        [0.0, -0.0, 1.0, -1.5, 3.0e38, 1e-40]])
    # halfway cases at the bf16 step: exact ties go to the even mantissa
    base = np.float32(1.0) + np.float32(2.0 ** -7) * np.arange(8, dtype=np.float32)
    ties = (base.astype(np.float64) + 2.0 ** -8)
    v = np.concatenate([v, ties, -ties])
    got = oracle.round_bf16(v)
    want = np.array([oracle.f32_to_bf16(float(np.float32(x))) for x in v], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)
    # ties: 1 + k*2^-7 + 2^-8 rounds to the even k
    tb = oracle.round_bf16(ties)
    assert list((tb & 1).astype(int)) == [0] * 8
    assert list(tb) == [0x3F80 + k + (k & 1) for k in range(8)]


def test_engram_rows_projection_order_and_orientation():
    # engram_v41.rs: rows are gathered in [token][col] order and viewed as
    # [tokens, cols*256]; y = x wkv^T.  A permutation matrix as wkv returns
    # each token's row back with its values permuted, exactly.
    tokens, cols, n_table = 3, 2, 10
    table = synth.q2k_blocks(5, "pin.engram", n_table)
    ids = np.array([7, 2, 2, 9, 0, 5], dtype=np.int32)
    K = cols * 256
    perm = np.random.default_rng(5).permutation(K)
    wkv = np.zeros((K, K), dtype=np.uint16)
    wkv[np.arange(K), perm] = 0x3F80  # bf16 1.0: y[:, n] = x[:, perm[n]]
    rows, y = oracle.engram_rows_projection(table, n_table, ids, tokens, cols, wkv)
    for t in range(tokens):
        for c in range(cols):
            blk = table[ids[t * cols + c]]
            np.testing.assert_array_equal(rows[t * cols + c], [oracle.f32_to_bf16(float(np.float32(w)))
                                                               for w in oracle.decode_block(blk)])
    x = oracle.bf16_to_f64(rows.reshape(tokens, K))
    np.testing.assert_array_equal(y, x[:, perm])


# ---- engram gate (engram_v41.rs module doc, step 4; engram_v41/apply.rs, the
# `gate_k` launch): closed forms on built streams, keys and values ----------------

def _sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


def test_engram_gate_zero_qk_gives_half_gate_and_the_last_block_is_the_value():
    T, hc, dim = 2, 3, 8
    g = np.random.default_rng(3)
    h = (g.integers(-64, 64, (T, hc, dim)) / 16.0).astype(np.float32)
    kv = (g.integers(-64, 64, (T, (hc + 1) * dim)) / 8.0).astype(np.float32)  # bf16-exact values
    out, gates = oracle.engram_gate(h, kv, np.zeros((hc, dim), np.float32), 1e-6)
    np.testing.assert_array_equal(gates, np.full((T, hc), 0.5))
    v = kv[:, hc * dim:].astype(np.float64)
    np.testing.assert_array_equal(out, h.astype(np.float64) + 0.5 * v[:, None, :])


def test_engram_gate_rounds_kv_to_bf16():
    # values that bf16 rounds (1 + 2^-10 -> 1; 1 + 3*2^-9 -> 1 + 2^-7)
    T, hc, dim = 1, 1, 4
    h = np.zeros((T, hc, dim), np.float32)
    kv = np.zeros((T, 2 * dim), np.float32)
    kv[0, dim:] = [1 + 2.0 ** -10, 1 + 3 * 2.0 ** -9, -(1 + 2.0 ** -10), 2.0]
    out, _ = oracle.engram_gate(h, kv, np.zeros((hc, dim), np.float32), 1e-6)  # zero stream: eps keeps rms > 0
    np.testing.assert_array_equal(out[0, 0], 0.5 * np.array([1.0, 1 + 2.0 ** -7, -1.0, 2.0]))


@pytest.mark.parametrize("dim", [16, 64])
@pytest.mark.parametrize("a,b", [(2.0, 0.5), (-3.0, 1.0), (0.25, -4.0)])
def test_engram_gate_parallel_stream_and_key(dim, a, b):
    """h = a u, key = b u, qk = 1, eps = 0: the normalised dot is
    sign(ab) sqrt(dim), so the gate is sigmoid(sign(ab) dim^(1/4))."""
    u = (np.random.default_rng(dim).integers(1, 16, dim) * np.where(np.arange(dim) % 3 == 0, -1, 1)).astype(np.float64)
    h = (a * u).astype(np.float32).reshape(1, 1, dim)
    kv = np.concatenate([b * u, np.ones(dim)]).astype(np.float32).reshape(1, 2 * dim)  # bf16-exact
    out, gates = oracle.engram_gate(h, kv, np.ones((1, dim), np.float32), 0.0)
    want = _sigmoid(math.copysign(dim ** 0.25, a * b))
    assert abs(gates[0, 0] - want) < 1e-14
    np.testing.assert_allclose(out[0, 0], a * u + want, rtol=0, atol=1e-13)


def test_engram_gate_eps_enters_each_rms():
    dim, a, b, eps = 16, 0.5, 2.0, 0.75
    u = np.ones(dim)
    h = (a * u).astype(np.float32).reshape(1, 1, dim)
    kv = np.concatenate([b * u, np.zeros(dim)]).astype(np.float32).reshape(1, 2 * dim)
    _, gates = oracle.engram_gate(h, kv, np.ones((1, dim), np.float32), eps)
    # mean(u^2) = 1: s = a b dim / (sqrt(a^2 + eps) sqrt(b^2 + eps) sqrt(dim))
    s = a * b * math.sqrt(dim) / (math.sqrt(a * a + np.float32(eps)) * math.sqrt(b * b + np.float32(eps)))
    assert abs(gates[0, 0] - _sigmoid(math.sqrt(s))) < 1e-14


def test_engram_gate_each_stream_reads_its_own_key():
    """Streams on disjoint supports with their own key equal to the stream:
    each gate is sigmoid(dim^(1/4) * sqrt(...)) for its own key and exactly
    0.5 had it read another stream's key (orthogonal, dot 0)."""
    hc, dim = 4, 16
    h = np.zeros((1, hc, dim), np.float32)
    kv = np.zeros((1, (hc + 1) * dim), np.float32)
    for c in range(hc):
        h[0, c, 4 * c:4 * c + 4] = 1.0 + c
        kv[0, c * dim + 4 * c:c * dim + 4 * c + 4] = 1.0
    _, gates = oracle.engram_gate(h, kv, np.ones((hc, dim), np.float32), 0.0)
    # mean(h^2) = (1+c)^2 / 4, mean(k^2) = 1/4, dot = 4 (1+c): s = 4 sqrt(dim) / dim * 4 = ...
    for c in range(hc):
        s = 4 * (1.0 + c) / (math.sqrt((1.0 + c) ** 2 / 4) * math.sqrt(1 / 4) * math.sqrt(dim))
        assert abs(gates[0, c] - _sigmoid(math.sqrt(s))) < 1e-14
        assert gates[0, c] > 0.5 + 1e-3
