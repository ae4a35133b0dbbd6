"""GPU parity of the Q2_K matmul for many tokens (q2k_mmq_bf16 and
q2k_mmq_q8_1) against the oracle, through the C ABI.

Bars:
  * bf16 activations: 2e-3 of each token row's L2 norm against the exact
    projection (the weights' on-chip bf16 rounding, 2^-9 relative per
    weight, stays far below it);
  * the same call equals dense_gemm_bf16 over q2k_dequant_rows' expansion
    within 1e-5 of the row norm (the same bf16 operands, only the order of
    the fp32 sums differs);
  * q8_1 activations: 1e-2 against the projection of the bf16 activations
    (the q8_1 bar), and 1e-3 against the exact projection of the q8_1 values
    (the tensor cores multiply the weights and those values after one bf16
    rounding each: <= 2^-8 relative per product, averaged over K).
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


def x_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def rel_err_rows(y, ref):
    y = np.atleast_2d(np.asarray(y, dtype=np.float64))
    ref = np.atleast_2d(np.asarray(ref, dtype=np.float64))
    return max(np.max(np.abs(y[t] - ref[t])) / max(np.linalg.norm(ref[t]), 1e-300) for t in range(ref.shape[0]))


@pytest.mark.parametrize("m,N,K", [(9, 300, 2048), (16, 128, 1024), (17, 1000, 4096), (64, 4096, 4096),
                                   (256, 513, 2048), (300, 256, 3072), (64, 64, 16384), (33, 2000, 8192)])
def test_mmq_bf16_against_oracle_and_the_dense_gemm_of_the_expansion(lib, m, N, K):
    W = synth.q2k_matrix(20, f"mmq.W.{N}.{K}", N, K)
    x = synth.bf16_normal(20, f"mmq.x.{m}.{K}", (m, K))
    Wd, xd = dev(W), bf16_dev(x)
    y = lib.q2k_mmq_bf16(Wd, xd).cpu().numpy()
    assert np.all(np.isfinite(y))
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_BF16
    yd = lib.dense_gemm_bf16(xd, lib.q2k_dequant_rows(Wd, K)).cpu().numpy()
    assert rel_err_rows(y, yd) <= 1e-5


@pytest.mark.parametrize("m,N,K", [(20, 51200, 1024), (140, 20000, 1024), (48, 30000, 3072)])
def test_mmq_many_pieces_per_cta(lib, m, N, K):
    """More (tile, 1024-K) units than SMs: CTAs finish several tiles in turn,
    so the accumulators are reused (two of them up to 128 tokens, one
    above) and tiles straddle CTAs.  Every row against the dense GEMM of the
    expansion, sampled rows (two per 128-row tile) against the oracle."""
    W = synth.q2k_matrix(23, f"mmq.pieces.W.{N}.{K}", N, K)
    x = synth.bf16_normal(23, f"mmq.pieces.x.{m}.{K}", (m, K))
    Wd, xd = dev(W), bf16_dev(x)
    y = lib.q2k_mmq_bf16(Wd, xd).cpu().numpy()
    yd = lib.dense_gemm_bf16(xd, lib.q2k_dequant_rows(Wd, K)).cpu().numpy()
    assert rel_err_rows(y, yd) <= 1e-5
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.minimum(np.arange(127, N + 127, 128), N - 1)]))
    ref = oracle.matvec(np.ascontiguousarray(W.reshape(N, -1)[rows]), len(rows), K, x_f64(x))
    assert rel_err_rows(y[:, rows], ref) <= TOL_BF16


@pytest.mark.parametrize("m,N,K", [(9, 300, 2048), (64, 1024, 4096), (256, 384, 2048)])
def test_mmq_q8_1_against_oracle(lib, m, N, K):
    W = synth.q2k_matrix(21, f"mmq8.W.{N}.{K}", N, K)
    x = synth.bf16_normal(21, f"mmq8.x.{m}.{K}", (m, K))
    xq = lib.q8_1_quantize_rows(bf16_dev(x))
    xq_h = xq.cpu().numpy()
    np.testing.assert_array_equal(xq_h, oracle.q8_1_quantize(x))
    y = lib.q2k_mmq_q8_1(dev(W), xq, K).cpu().numpy()
    assert rel_err_rows(y, oracle.matvec(W, N, K, x_f64(x))) <= TOL_Q8
    assert rel_err_rows(y, oracle.matvec(W, N, K, oracle.q8_1_dequant(xq_h, m, K))) <= 1e-3


def test_mmq_output_stride_and_unaligned_row_stride_rejected(lib):
    import ctypes
    N, K, m = 200, 2048, 20
    W = dev(synth.q2k_matrix(22, "mmq.st.W", N, K))
    x = synth.bf16_normal(22, "mmq.st.x", (m, K))
    y = torch.full((m, N + 8), 7.0, dtype=torch.float32, device="cuda")
    lib.q2k_mmq_bf16(W, bf16_dev(x), out=y[:, :N])
    ref = oracle.matvec(synth.q2k_matrix(22, "mmq.st.W", N, K), N, K, x_f64(x))
    assert rel_err_rows(y[:, :N].cpu().numpy(), ref) <= TOL_BF16
    assert torch.all(y[:, N:] == 7.0)  # the gap between rows is left alone
    # a row stride that is not 16 bytes is refused before any launch
    xs = torch.zeros((m, K + 4), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.lib().q2k_mmq_bf16(P(W), N, K, P(xs), m, K + 4, P(y), N + 8, None) == 2


@pytest.mark.parametrize("m", [64, 256])
def test_mmq_config_16384_tile_edges(lib, m):
    """The sweep's dense shapes with Q2_K weights: N = K = 16384, rows at
    every 128-row tile edge."""
    N = K = 16384
    W = synth.q2k_matrix(0, "sweep.W16384x16384", N, K)
    x = synth.bf16_normal(0, f"sweep.dense.x{m}.{N}", (m, K))
    y = lib.q2k_mmq_bf16(dev(W), bf16_dev(x)).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, N, 128), np.arange(127, N, 128)]))
    ref = oracle.matvec(np.ascontiguousarray(W.reshape(N, -1)[rows]), len(rows), K, x_f64(x))
    assert rel_err_rows(y[:, rows], ref) <= TOL_BF16
