"""CPU-side checks of the C ABI: the library loads, exports every entry point
include/q2k.h declares, and rejects bad arguments with a status code before
touching the GPU (the pages' `ensure!` checks before any launch:
engram_v41/apply.rs `apply`, engram_v41.rs `rows_from_q2k`,
moe_v41/init.rs `MoeV41::new`).  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q2k.h")


@pytest.fixture(scope="module")
def L():
    from mmvq_q2_gb300 import build
    build.build()
    import mmvq_q2_gb300 as q
    return q.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?[\s\*]+([a-z][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary_calls():
    names = declared_functions()
    for want in ["q2k_dequant_rows", "q8_1_quantize_rows", "q2k_gemv_bf16", "q2k_mmvq_q8_1", "q2k_mmvq_pair",
                 "q2k_mmvq_experts", "dense_gemm_bf16", "swiglu_q8_1_rows", "q2k_moe_m1", "q2k_mmvq_grouped",
                 "q2k_engram_hash", "q2k_engram_gate", "q3k_mmvq_q8_1", "q3k_mmvq_experts", "q2k_mmq_bf16",
                 "q2k_mmq_q8_1"]:
        assert want in names


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_is_plain_c_and_cpp(lang, std, tmp_path):
    # the boundary is usable from C: no C++ or CUDA types in the signatures
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "q2k.h"\nint main(void) { return (int)q2k_row_bytes(256) + (int)q3k_row_bytes(256); }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.dirname(HEADER), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(L):
    import mmvq_q2_gb300 as q
    names = declared_functions()
    assert sorted(q.EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_size_helpers(L):
    assert L.q2k_row_bytes(256) == 84
    assert L.q2k_row_bytes(16384) == 64 * 84
    assert L.q2k_row_bytes(300) == 0 and L.q2k_row_bytes(0) == 0
    assert L.q8_1_row_bytes(4096) == 128 * 36
    assert L.q8_1_row_bytes(33) == 0
    assert L.q2k_moe_m1_workspace_bytes(8, 4096, 2048) == 4608 + 2 * 8 * 2048 * 4 + 8 * 2304 + 8 * 4096 * 4


def test_status_strings(L):
    for s in range(7):
        assert L.q2k_status_string(s)
    assert L.q2k_status_string(99) == b"unknown status"


P = ctypes.c_void_p
FAKE = P(0x10000)      # never dereferenced: validation fails first
ODD = P(0x10001)


def test_gemv_validation(L):
    assert L.q2k_gemv_bf16(None, 4, 256, FAKE, 1, 256, FAKE, 4, None) == 1
    assert L.q2k_gemv_bf16(FAKE, 4, 300, FAKE, 1, 300, FAKE, 4, None) == 2   # K % 256
    assert L.q2k_gemv_bf16(FAKE, 4, 256, FAKE, 0, 256, FAKE, 4, None) == 2   # m = 0
    assert L.q2k_gemv_bf16(FAKE, 4, 256, FAKE, 9, 256, FAKE, 4, None) == 2   # m > 8
    assert L.q2k_gemv_bf16(FAKE, 0, 256, FAKE, 1, 256, FAKE, 4, None) == 2   # N = 0
    assert L.q2k_gemv_bf16(FAKE, 4, 256, FAKE, 1, 128, FAKE, 4, None) == 2   # ldx < K
    assert L.q2k_gemv_bf16(FAKE, 4, 256, FAKE, 1, 256, FAKE, 3, None) == 2   # ldy < N
    assert L.q2k_gemv_bf16(ODD, 4, 256, FAKE, 1, 256, FAKE, 4, None) == 3
    assert L.q2k_gemv_bf16(FAKE, 4, 256, ODD, 1, 256, FAKE, 4, None) == 3
    assert L.q2k_gemv_bf16(FAKE, 4, 256, FAKE, 1, 256, P(0x10002), 4, None) == 3


def test_mmvq_pair_experts_validation(L):
    assert L.q2k_mmvq_q8_1(FAKE, 4, 512, None, 1, FAKE, 4, None) == 1
    assert L.q2k_mmvq_q8_1(FAKE, 4, 512, FAKE, 9, FAKE, 4, None) == 2
    assert L.q2k_mmvq_pair(FAKE, 4, FAKE, FAKE, 4, FAKE, 512, FAKE, 0, None) == 2
    assert L.q2k_mmvq_pair(FAKE, 4, FAKE, None, 4, FAKE, 512, FAKE, 1, None) == 1
    assert L.q2k_mmvq_pair(FAKE, 4, FAKE, FAKE, -1, FAKE, 512, FAKE, 1, None) == 2
    # the engram hash: positions within the cache, 2 <= max_ngram <= 16, a layer in range
    H = lambda *a: L.q2k_engram_hash(*a)  # noqa: E731
    ok = (FAKE, 100, FAKE, 64, FAKE, 4, 0, 3, 2, 2, FAKE, FAKE, FAKE, 0, FAKE, None, 0, None, None)
    bad = list(ok); bad[0] = None
    assert H(*bad) == 1
    bad = list(ok); bad[6] = 61  # start_pos + seqlen > max_seq
    assert H(*bad) == 2
    bad = list(ok); bad[7] = 17
    assert H(*bad) == 2
    bad = list(ok); bad[15] = FAKE; bad[16] = 2  # layer_index outside n_layers
    assert H(*bad) == 2
    bad = list(ok); bad[2] = P(0x10004)  # cache not 8-byte aligned
    assert H(*bad) == 3
    # the grouped MMVQ: groups, rows, K_group (multiple of 256) and m in 1..8
    assert L.q2k_mmvq_grouped(FAKE, 8, 64, 512, None, 1, FAKE, None) == 1
    assert L.q2k_mmvq_grouped(FAKE, 0, 64, 512, FAKE, 1, FAKE, None) == 2
    assert L.q2k_mmvq_grouped(FAKE, 8, 64, 500, FAKE, 1, FAKE, None) == 2
    assert L.q2k_mmvq_grouped(FAKE, 8, 64, 512, FAKE, 9, FAKE, None) == 2
    assert L.q2k_mmvq_grouped(P(0x10002), 8, 64, 512, FAKE, 1, FAKE, None) == 3
    # the pair over bf16 rows: the q8_1 destination is required; x is 2-byte aligned
    assert L.q2k_mmvq_pair_bf16(FAKE, 4, FAKE, FAKE, 4, FAKE, 512, FAKE, 1, None, None) == 1
    assert L.q2k_mmvq_pair_bf16(FAKE, 4, FAKE, FAKE, 4, FAKE, 512, FAKE, 9, FAKE, None) == 2
    assert L.q2k_mmvq_pair_bf16(FAKE, 4, FAKE, FAKE, 4, FAKE, 500, FAKE, 1, FAKE, None) == 2
    assert L.q2k_mmvq_pair_bf16(FAKE, 4, FAKE, FAKE, 4, FAKE, 512, P(0x10001), 1, FAKE, None) == 3
    # experts: y_sum needs route weights; x_per_matrix is 0 or 1
    assert L.q2k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 0, None, None, FAKE, None) == 1
    assert L.q2k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 0, None, None, None, None) == 1
    assert L.q2k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 2, FAKE, None, None, None) == 2
    assert L.q2k_mmvq_experts(FAKE, 0, 64, 512, FAKE, 0, FAKE, None, None, None) == 2
    assert L.q2k_mmvq_experts(P(0x10004), 8, 64, 512, FAKE, 0, FAKE, None, None, None) == 3



def test_q3k_validation(L):
    assert L.q3k_row_bytes(256) == 110 and L.q3k_row_bytes(4096) == 16 * 110 and L.q3k_row_bytes(100) == 0
    # single matrix: K multiple of 256, m in 1..8, ldy >= N, 4-byte alignment
    assert L.q3k_mmvq_q8_1(None, 4, 512, FAKE, 1, FAKE, 4, None) == 1
    assert L.q3k_mmvq_q8_1(FAKE, 4, 500, FAKE, 1, FAKE, 4, None) == 2
    assert L.q3k_mmvq_q8_1(FAKE, 4, 512, FAKE, 0, FAKE, 4, None) == 2
    assert L.q3k_mmvq_q8_1(FAKE, 4, 512, FAKE, 9, FAKE, 4, None) == 2
    assert L.q3k_mmvq_q8_1(FAKE, 4, 512, FAKE, 1, FAKE, 3, None) == 2
    assert L.q3k_mmvq_q8_1(FAKE, 0, 512, FAKE, 1, FAKE, 4, None) == 2
    assert L.q3k_mmvq_q8_1(P(0x10002), 4, 512, FAKE, 1, FAKE, 4, None) == 3
    assert L.q3k_mmvq_q8_1(FAKE, 4, 512, P(0x10002), 1, FAKE, 4, None) == 3
    # experts: y required, y_sum needs route weights, x_per_matrix 0 or 1
    assert L.q3k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 0, None, None, None, None) == 1
    assert L.q3k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 0, FAKE, None, FAKE, None) == 1
    assert L.q3k_mmvq_experts(FAKE, 8, 64, 512, FAKE, 2, FAKE, None, None, None) == 2
    assert L.q3k_mmvq_experts(FAKE, 0, 64, 512, FAKE, 0, FAKE, None, None, None) == 2
    assert L.q3k_mmvq_experts(FAKE, 8, 64, 768 + 1, FAKE, 0, FAKE, None, None, None) == 2
    assert L.q3k_mmvq_experts(P(0x10004), 8, 64, 512, FAKE, 0, FAKE, None, None, None) == 3


def test_small_kernels_validation(L):
    assert L.q2k_dequant_rows(None, 4, 256, None, 1, FAKE, None, None) == 1
    assert L.q2k_dequant_rows(FAKE, 4, 200, None, 1, FAKE, None, None) == 2
    assert L.q2k_dequant_rows(FAKE, 4, 256, None, 5, FAKE, None, None) == 2  # rows past the table
    assert L.q2k_dequant_rows(FAKE, 4, 256, ODD, 2, FAKE, None, None) == 3
    assert L.q8_1_quantize_rows(FAKE, 1, 48, 48, FAKE, None) == 2
    assert L.q8_1_quantize_rows(FAKE, 1, 64, 32, FAKE, None) == 2
    assert L.q8_1_quantize_rows(FAKE, 1, 64, 64, ODD, None) == 3
    assert L.swiglu_q8_1_rows(FAKE, 1, 48, FAKE, None, None) == 2
    assert L.swiglu_q8_1_rows(None, 1, 64, FAKE, None, None) == 1


def test_moe_and_gemm_validation(L):
    ws = L.q2k_moe_m1_workspace_bytes(2, 256, 256)
    assert L.q2k_moe_m1(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, None, ws, None) == 6
    assert L.q2k_moe_m1(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, FAKE, ws - 1, None) == 6
    assert L.q2k_moe_m1(FAKE, 2, 300, 256, FAKE, FAKE, FAKE, FAKE, ws, None) == 2
    assert L.q2k_moe_m1(FAKE, 2, 256, 256, FAKE, FAKE, FAKE, P(0x10010), ws, None) == 3
    assert L.dense_gemm_bf16(FAKE, 1, 12, 12, FAKE, 4, FAKE, 4, None) == 2
    assert L.dense_gemm_bf16(P(0x10008), 1, 16, 16, FAKE, 4, FAKE, 4, None) == 3
    assert L.dense_gemm_bf16(FAKE, 0, 16, 16, FAKE, 4, FAKE, 4, None) == 2


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import mmvq_q2_gb300 as q
    monkeypatch.setattr(q, "_lib", None)
    monkeypatch.setattr(q, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        q.lib()


def test_engram_gate_validation_before_any_launch(L):
    import math
    p = ctypes.c_void_p(0x10000)
    G = lambda *a: L.q2k_engram_gate(*a)  # noqa: E731
    # streams, kv, ld_kv, qk, tokens, hc, dim, eps, gates, stream
    assert G(None, p, 20480, p, 1, 4, 4096, 1e-6, None, None) == 1
    assert G(p, p, 20480, None, 1, 4, 4096, 1e-6, None, None) == 1
    assert G(p, p, 20480, p, 1, 5, 4096, 1e-6, None, None) == 2     # hc in 1..4 (the page's limit)
    assert G(p, p, 20480, p, 1, 0, 4096, 1e-6, None, None) == 2
    assert G(p, p, 20479, p, 1, 4, 4096, 1e-6, None, None) == 2     # kv rows hold hc keys and the value
    assert G(p, p, 20480, p, 1, 4, 0, 1e-6, None, None) == 2
    assert G(p, p, 20480, p, -1, 4, 4096, 1e-6, None, None) == 2
    assert G(p, p, 20480, p, 1, 4, 4096, -1.0, None, None) == 2
    assert G(p, p, 20480, p, 1, 4, 4096, math.nan, None, None) == 2
    assert G(ctypes.c_void_p(0x10002), p, 20480, p, 1, 4, 4096, 1e-6, None, None) == 3
    assert G(p, p, 20480, p, 1, 4, 4096, 1e-6, ctypes.c_void_p(0x10001), None) == 3


def test_mmq_validation_before_any_launch(L):
    p16 = ctypes.c_void_p(0x10000)
    # W, N, K, x, m, ldx, y, ldy, stream
    assert L.q2k_mmq_bf16(None, 64, 4096, p16, 64, 4096, p16, 64, None) == 1
    assert L.q2k_mmq_bf16(p16, 64, 4352, p16, 64, 4352, p16, 64, None) == 2   # K % 1024
    assert L.q2k_mmq_bf16(p16, 64, 4096, p16, 0, 4096, p16, 64, None) == 2
    assert L.q2k_mmq_bf16(p16, 64, 4096, p16, 64, 4100, p16, 64, None) == 2   # ldx % 8
    assert L.q2k_mmq_bf16(p16, 64, 4096, p16, 64, 4096, p16, 63, None) == 2
    assert L.q2k_mmq_bf16(ctypes.c_void_p(0x10004), 64, 4096, p16, 64, 4096, p16, 64, None) == 3
    assert L.q2k_mmq_bf16(p16, 64, 4096, ctypes.c_void_p(0x10008), 64, 4096, p16, 64, None) == 3
    assert L.q2k_mmq_q8_1_workspace_bytes(64, 4096) == 64 * 4096 * 2
    assert L.q2k_mmq_q8_1_workspace_bytes(64, 4352) == 0
    need = L.q2k_mmq_q8_1_workspace_bytes(64, 4096)
    assert L.q2k_mmq_q8_1(p16, 64, 4096, p16, 64, p16, 64, p16, need - 1, None) == 6
    assert L.q2k_mmq_q8_1(p16, 64, 4096, p16, 64, p16, 64, None, need, None) == 6
