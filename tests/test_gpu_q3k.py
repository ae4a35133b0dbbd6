"""GPU parity of the Q3_K MMVQ twins (moe_v41/init.rs, `MoeV41::new`:
`kquant_mmvq_q3_k_w`, `kquant_mmvq_q3_k_experts_w*`) against the CPU oracle,
through the C ABI.

Bars: the integer dot products are exact, so against the exact projection of
the values the q8_1 rows encode the error is fp32 accumulation only
(max |y - y_ref| / ||y_ref[t]||_2 <= 1e-4 per token row); against the bf16
activations the q8_1 bar of the Q2_K path (1e-2) holds.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_EXACT_X = 1e-4
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


def rel_err_rows(y, ref):
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    return max(np.max(np.abs(y[t] - ref[t])) / max(np.linalg.norm(ref[t]), 1e-300) for t in range(ref.shape[0]))


def x_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


# slice widths 16/8/4 bytes, ragged chunks (nb not a multiple of the chunk),
# one and several chunks per warp, every token count (pairs of tokens walk the rows in turn)
CASES = [(1, 256, 1), (7, 512, 1), (33, 2048, 1), (300, 4096, 1), (65, 4864, 1), (40, 6400, 1),
         (33, 2048, 2), (300, 4096, 2), (65, 4864, 2), (31, 768, 3), (64, 4096, 4), (300, 1280, 4),
         (65, 4864, 5), (33, 2048, 6), (300, 4096, 8), (17, 256, 8)]


@pytest.mark.parametrize("N,K,m", CASES)
def test_q3k_mmvq_against_oracle(lib, N, K, m):
    W = synth.q3k_matrix(3, f"q3.{N}.{K}", N, K)
    x = synth.bf16_normal(3, f"q3.x.{m}.{K}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q3k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert y.shape == (m, N)
    assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= TOL_EXACT_X
    if N >= 32:
        assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, x_f64(x))) <= TOL_Q8


@pytest.mark.parametrize("m", [1, 3])
def test_q3k_mmvq_long_rows_many_chunks(lib, m):
    # 256 block columns: 16 (one token) or 32 chunks, more than the 8 warps
    N, K = 40, 65536
    W = synth.q3k_matrix(4, "q3.long", N, K)
    x = synth.bf16_normal(4, f"q3.long.x{m}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q3k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= TOL_EXACT_X


@pytest.mark.parametrize("m", [1, 2, 3])
def test_q3k_mmvq_largest_k(lib, m):
    # K = 2^20, the largest the boundary accepts: 4096 block columns, 256
    # (one token) or 512 chunks per row, one row per CTA
    N, K = 3, 1 << 20
    W = synth.q3k_matrix(11, "q3.maxk", N, K)
    x = synth.bf16_normal(11, f"q3.maxk.x{m}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q3k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= TOL_EXACT_X


@pytest.mark.parametrize("K,m", [(512, 2), (4096, 1), (4096, 2), (4864, 2), (4096, 4), (4864, 6), (2048, 8)])
def test_q3k_mmvq_weights_off_a_16_byte_boundary(lib, K, m):
    # the matrix starts 4 bytes into its buffer: every block's word phase
    # flips, and several tokens take warp copies instead of tensor copies;
    # one and two tokens at K = 4096 leave the row-team kernel for the
    # general one, which gives the same bits
    N = 50
    W = synth.q3k_matrix(5, f"q3.off.{K}", N, K)
    buf = torch.zeros(W.size + 4, dtype=torch.uint8, device="cuda")
    buf[4:] = dev(W.reshape(-1))
    x = synth.bf16_normal(5, f"q3.off.x.{K}.{m}", (m, K))
    xq = dev(oracle.q8_1_quantize(x))
    y = lib.q3k_mmvq_q8_1(buf[4:], xq, K).cpu().numpy()
    assert np.array_equal(y, lib.q3k_mmvq_q8_1(dev(W), xq, K).cpu().numpy())
    assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, oracle.q8_1_dequant(xq.cpu().numpy(), m, K))) <= TOL_EXACT_X


@pytest.mark.parametrize("N,K,m", [(50, 4096, 1), (50, 4096, 2), (50, 4096, 5), (40, 1280, 3)])
def test_q3k_mmvq_activations_off_a_16_byte_boundary(lib, N, K, m):
    # q8_1 rows 4 bytes into their buffer: several tokens read them from
    # global memory instead of staging them by bulk copy, and one or two
    # tokens leave the row-team kernel for the general one, with the same bits
    W = dev(synth.q3k_matrix(12, f"q3.xoff.{K}", N, K))
    xq = oracle.q8_1_quantize(synth.bf16_normal(12, f"q3.xoff.x.{K}", (m, K)))
    buf = torch.zeros(xq.size + 4, dtype=torch.uint8, device="cuda")
    buf[4:] = dev(xq.reshape(-1))
    y = lib.q3k_mmvq_q8_1(W, buf[4:].view(m, -1), K)
    assert torch.equal(y, lib.q3k_mmvq_q8_1(W, dev(xq), K))
    ref = oracle.q3k_matvec(W.cpu().numpy(), N, K, oracle.q8_1_dequant(xq, m, K))
    assert rel_err_rows(y.cpu().numpy(), ref) <= TOL_EXACT_X


def test_q3k_mmvq_output_stride_leaves_the_gap(lib):
    N, K, m = 100, 1024, 3
    W = dev(synth.q3k_matrix(6, "q3.ldy", N, K))
    xq = dev(oracle.q8_1_quantize(synth.bf16_normal(6, "q3.ldy.x", (m, K))))
    out = torch.full((m, N + 28), 7.0, dtype=torch.float32, device="cuda")
    lib.q3k_mmvq_q8_1(W, xq, K, out=out[:, :N])
    assert torch.equal(out[:, :N], lib.q3k_mmvq_q8_1(W, xq, K))
    assert (out[:, N:] == 7.0).all()


@pytest.mark.parametrize("m", [3, 8])
def test_q3k_several_tokens_in_waves(lib, m):
    # 1537 row tiles: more than eight per CTA on one CTA per SM, so the
    # tensor-core kernel runs more CTAs than SMs, in waves; a ragged last tile
    N, K = 24577, 2048
    W = synth.q3k_matrix(13, "q3.waves", N, K)
    x = synth.bf16_normal(13, f"q3.waves.x{m}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q3k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, N, 97), np.arange(N - 40, N)]))
    ref = oracle.q3k_matvec(np.ascontiguousarray(W[rows]), len(rows), K, oracle.q8_1_dequant(xq, m, K))
    assert rel_err_rows(y[:, rows], ref) <= TOL_EXACT_X


@pytest.fixture(scope="module")
def big_w3():
    W = synth.q3k_matrix(0, "q3.W16384", 16384, 16384)
    return W, dev(W)


@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_q3k_mmvq_16384_sampled(lib, big_w3, m):
    W, Wd = big_w3
    x = synth.bf16_normal(0, f"q3.sweep.x{m}", (m, 16384))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    y = lib.q3k_mmvq_q8_1(Wd, xq, 16384).cpu().numpy()
    rows = np.sort(np.random.default_rng(20 + m).choice(16384, 48, replace=False))
    Ws = np.ascontiguousarray(W[rows])
    ref = oracle.q3k_matvec(Ws, len(rows), 16384, oracle.q8_1_dequant(xq.cpu().numpy(), m, 16384))
    assert rel_err_rows(y[:, rows], ref) <= TOL_EXACT_X
    assert rel_err_rows(y[:, rows], oracle.q3k_matvec(Ws, len(rows), 16384, x_f64(x))) <= TOL_Q8


def test_q3k_repeat_calls_are_bitwise_identical(lib, big_w3):
    _, Wd = big_w3
    xq = lib.q8_1_quantize_rows(bf16_dev(synth.bf16_normal(1, "q3.rep", (1, 16384))))
    y0 = lib.q3k_mmvq_q8_1(Wd, xq, 16384)
    for _ in range(3):
        assert torch.equal(lib.q3k_mmvq_q8_1(Wd, xq, 16384), y0)


@pytest.mark.parametrize("per_matrix", [False, True])
def test_q3k_experts_rows_equal_singles_and_weighted_sum(lib, per_matrix):
    n_mat, N, K = 5, 300, 512
    mats = [dev(synth.q3k_matrix(7, f"q3ex.{e}", N, K)) for e in range(n_mat)]
    rows = n_mat if per_matrix else 1
    xq = lib.q8_1_quantize_rows(bf16_dev(synth.bf16_normal(7, f"q3ex.x{rows}", (rows, K))))
    w = np.float32([0.1, 0.3, 0.05, 0.25, 0.3])
    ysum = torch.empty(N, dtype=torch.float32, device="cuda")
    y, _ = lib.q3k_mmvq_experts(lib.pointer_table(mats), N, K, xq, x_per_matrix=per_matrix, route_w=dev(w),
                                y_sum=ysum)
    for e in range(n_mat):
        xe = xq[e:e + 1] if per_matrix else xq
        assert torch.equal(y[e:e + 1], lib.q3k_mmvq_q8_1(mats[e], xe, K)), e
    ref = (w.astype(np.float64)[:, None] * y.cpu().numpy().astype(np.float64)).sum(0)
    assert np.max(np.abs(ysum.cpu().numpy() - ref)) <= 1e-5 * np.linalg.norm(ref)


# one or two tokens over long rows (K a multiple of 2048 from 4096 to 32768,
# W and x on 16-byte boundaries) run the row-team kernel: teams of 32 to 512
# lanes, lanes past the row (K = 6144: 48 of 64 for one token, 96 of 128 for
# two), fewer rows than SMs, a row more on some CTAs, many stages per CTA
@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("N,K", [(1, 4096), (153, 6144), (300, 8192), (2000, 4096), (400, 32768)])
def test_q3k_row_team_kernel_against_oracle(lib, N, K, m):
    W = synth.q3k_matrix(12, f"q3.rt.{N}.{K}", N, K)
    x = synth.bf16_normal(12, f"q3.rt.x{m}.{K}", (m, K))
    xq = oracle.q8_1_quantize(x)
    y = lib.q3k_mmvq_q8_1(dev(W), dev(xq), K).cpu().numpy()
    assert y.shape == (m, N)
    assert rel_err_rows(y, oracle.q3k_matvec(W, N, K, oracle.q8_1_dequant(xq, m, K))) <= TOL_EXACT_X


# the expert batches keep the general kernel; their rows still equal single
# calls bit for bit where a single call takes the row-team kernel
@pytest.mark.parametrize("K", [4096, 6144, 16384])
@pytest.mark.parametrize("per_matrix", [False, True])
def test_q3k_experts_equal_singles_on_row_team_shapes(lib, K, per_matrix):
    n_mat, N = 3, 300
    mats = [dev(synth.q3k_matrix(13, f"q3rt.{K}.{e}", N, K)) for e in range(n_mat)]
    rows = n_mat if per_matrix else 1
    xq = lib.q8_1_quantize_rows(bf16_dev(synth.bf16_normal(13, f"q3rt.x{rows}.{K}", (rows, K))))
    y, _ = lib.q3k_mmvq_experts(lib.pointer_table(mats), N, K, xq, x_per_matrix=per_matrix)
    for e in range(n_mat):
        xe = xq[e:e + 1] if per_matrix else xq
        assert torch.equal(y[e:e + 1], lib.q3k_mmvq_q8_1(mats[e], xe, K)), e


def test_q3k_experts_row_team_table_entries_off_16_and_off_a_word(lib):
    # a shared input over rows of 16 blocks takes the row-team kernel: the
    # entry 4 bytes past a 16-byte boundary is copied by the lanes (word by
    # word), the entry off a word is skipped and flagged; stages straddle
    # the matrices (200 rows each, about 4 rows a CTA)
    N, K = 200, 4096
    mats = [synth.q3k_matrix(14, f"q3tab.{e}", N, K) for e in range(3)]
    good = dev(mats[0])
    buf4 = torch.zeros(mats[1].size + 16, dtype=torch.uint8, device="cuda")
    buf4[4:4 + mats[1].size] = dev(mats[1].reshape(-1))
    bad = torch.zeros(mats[2].size + 16, dtype=torch.uint8, device="cuda")
    tbl = torch.tensor([good.data_ptr(), buf4.data_ptr() + 4, bad.data_ptr() + 2], dtype=torch.int64, device="cuda")
    xq = dev(oracle.q8_1_quantize(synth.bf16_normal(14, "q3tab.x", (1, K))))
    y = torch.full((3, N), 5.0, dtype=torch.float32, device="cuda")
    lib.q2k_device_error(clear=True)
    lib.q3k_mmvq_experts(tbl, N, K, xq, y=y)
    torch.cuda.synchronize()
    assert lib.q2k_device_error(clear=True) == 2
    assert torch.equal(y[0:1], lib.q3k_mmvq_q8_1(good, xq, K))
    assert torch.equal(y[1:2], lib.q3k_mmvq_q8_1(dev(mats[1]), xq, K))
    assert (y[2] == 5.0).all()


def test_q3k_experts_moe_shapes_against_oracle(lib):
    # gate/up batch: 16 matrices [2048, 4096] over one row; down batch:
    # 8 matrices [4096, 2048], one row each (sampled output rows)
    dim, inter, E = 4096, 2048, 8
    gu = [synth.q3k_matrix(8, f"q3moe.gu.{e}", inter, dim) for e in range(2 * E)]
    dn = [synth.q3k_matrix(8, f"q3moe.dn.{e}", dim, inter) for e in range(E)]
    x = synth.bf16_normal(8, "q3moe.x", (1, dim))
    h = synth.bf16_normal(8, "q3moe.h", (E, inter))
    xq = oracle.q8_1_quantize(x)
    hq = oracle.q8_1_quantize(h)
    y_gu, _ = lib.q3k_mmvq_experts(lib.pointer_table([dev(a) for a in gu]), inter, dim, dev(xq))
    w = synth.expert_route(8, 256, E)[1]
    ysum = torch.empty(dim, dtype=torch.float32, device="cuda")
    y_dn, _ = lib.q3k_mmvq_experts(lib.pointer_table([dev(a) for a in dn]), dim, inter, dev(hq), x_per_matrix=True,
                                   route_w=dev(w), y_sum=ysum)
    rs = np.random.default_rng(9)
    xd = oracle.q8_1_dequant(xq, 1, dim)
    hd = oracle.q8_1_dequant(hq, E, inter)
    for e in (0, 5, 11, 15):
        rows = np.sort(rs.choice(inter, 24, replace=False))
        ref = oracle.q3k_matvec(np.ascontiguousarray(gu[e][rows]), len(rows), dim, xd)
        assert rel_err_rows(y_gu[e:e + 1, rows].cpu().numpy(), ref) <= TOL_EXACT_X, e
    full = np.zeros(dim)
    for e in range(E):
        ye = oracle.q3k_matvec(dn[e], dim, inter, hd[e:e + 1])
        assert rel_err_rows(y_dn[e:e + 1].cpu().numpy(), ye) <= TOL_EXACT_X, e
        full += float(w[e]) * ye[0]
    assert rel_err_rows(ysum.cpu().numpy()[None], full[None]) <= TOL_EXACT_X


def test_q3k_experts_skip_a_table_entry_off_a_word_and_flag_it(lib):
    # the kernel checks each table entry before reading it; the host made
    # the bad entry, so nothing is read from it
    N, K = 64, 512
    good = dev(synth.q3k_matrix(9, "q3bad.0", N, K))
    buf = torch.zeros(good.numel() + 16, dtype=torch.uint8, device="cuda")
    tbl = torch.tensor([good.data_ptr(), buf.data_ptr() + 2], dtype=torch.int64, device="cuda")
    xq = dev(oracle.q8_1_quantize(synth.bf16_normal(9, "q3bad.x", (1, K))))
    y = torch.full((2, N), 5.0, dtype=torch.float32, device="cuda")
    lib.q2k_device_error(clear=True)
    lib.q3k_mmvq_experts(tbl, N, K, xq, y=y)
    torch.cuda.synchronize()
    assert lib.q2k_device_error(clear=True) == 2
    assert torch.equal(y[0:1], lib.q3k_mmvq_q8_1(good, xq, K))
    assert (y[1] == 5.0).all()
