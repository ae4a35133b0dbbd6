"""The allocation-free routed-expert call (q2k_moe_m1_static_scratch)
against q2k_moe_m1 with a caller workspace.

Collected last on purpose: it must hold both alone and after every other
test has run in the same process.  The calls go through the C ABI."""
import ctypes

import numpy as np
import pytest
import torch

import synth

DIM, INTER, TOPK, E_ALL = 4096, 2048, 8, 256


@pytest.fixture(scope="module")
def L():
    from mmvq_q2_gb300 import build
    build.build()
    import mmvq_q2_gb300 as q
    return q.lib()


def test_oversized_problem_is_refused_before_any_launch(L):
    fake = ctypes.c_void_p(0x10000)
    assert L.q2k_moe_m1_workspace_bytes(64, 8192, 4096) > (1 << 20)
    assert L.q2k_moe_m1_static_scratch(fake, 64, 8192, 4096, fake, fake, fake, None) == 6
    assert L.q2k_moe_m1_static_scratch(fake, 8, 300, 2048, fake, fake, fake, None) == 2
    # shapes q2k_moe_m1 refuses are shape errors, not "too big for the scratch"
    assert L.q2k_moe_m1_static_scratch(fake, 2000, 4096, 2048, fake, fake, fake, None) == 2
    assert L.q2k_moe_m1_static_scratch(fake, 8, 4096, (1 << 20) + 256, fake, fake, fake, None) == 2
    assert L.q2k_moe_m1_static_scratch(fake, 0, 4096, 2048, fake, fake, fake, None) == 2
    assert L.q2k_moe_m1_static_scratch(None, 8, 4096, 2048, fake, fake, fake, None) == 1


def _route(seed):
    """Weights of the selected experts only, the token and its route."""
    ids, w = synth.expert_route(seed, E_ALL, TOPK)
    mats = []
    for kind, shape in (("gate", (INTER, DIM)), ("up", (INTER, DIM)), ("down", (DIM, INTER))):
        for e in ids:
            mats.append(torch.from_numpy(synth.q2k_matrix(0, f"cfg3.{kind}{int(e)}", *shape)).cuda())
    x = synth.bf16_normal(seed, "cfg3.x", (DIM,))
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    wd = torch.from_numpy(w).cuda()
    tbl = torch.tensor([m.data_ptr() for m in mats], dtype=torch.int64, device="cuda")
    return mats, tbl, xd, wd


@pytest.mark.gpu
def test_static_scratch_matches_workspace_call_twice_in_a_row(L):
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    need = L.q2k_moe_m1_workspace_bytes(TOPK, DIM, INTER)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    routes = [_route(0), _route(1)]
    outs = []
    for mats, tbl, xd, wd in routes:  # two allocation-free calls back to back
        y = torch.empty(DIM, dtype=torch.float32, device="cuda")
        assert L.q2k_moe_m1_static_scratch(P(tbl), TOPK, DIM, INTER, P(xd), P(wd), P(y), stream) == 0
        outs.append(y)
    for (mats, tbl, xd, wd), y in zip(routes, outs):
        ref = torch.empty(DIM, dtype=torch.float32, device="cuda")
        assert L.q2k_moe_m1(P(tbl), TOPK, DIM, INTER, P(xd), P(wd), P(ref), P(ws), need, stream) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(y).all()
        # the same launches on the same inputs: equal bit for bit
        assert torch.equal(y, ref)
    assert not torch.equal(outs[0], outs[1])
    v = ctypes.c_int32(0)
    assert L.q2k_device_error(ctypes.byref(v), 1) == 0 and v.value == 0
