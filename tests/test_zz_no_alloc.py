"""pa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (for example code running where its allocator or memory pool forbids
new allocations). It keeps its scratch in a fixed array inside the library
instead of a caller workspace. This file is collected last, so a run that
stops at the first failure has already run every other test.

Two calls in a row through the C ABI must each match pa_bwd (which uses a
caller-allocated workspace) within the tolerances the parity tests use, and
dims that need more scratch than the array holds must be refused."""
import ctypes

import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa
import synth

pytestmark = pytest.mark.gpu

GRAD_RELL2 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


def _inputs(w, dev):
    t = w.tensors()
    to = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)
    q, k, v, do = (to(t[x]) for x in ("q", "k", "v", "do"))
    return q, k, v, do, torch.from_numpy(w.seg).to(dev)


def _rel(a, b):
    a, b = a.float(), b.float()
    return float((a - b).norm() / b.norm())


RAGGED = synth.custom(2, 4, 2, 300, 128, [[150, 150], [1, 298, 1]], seed=32)


@pytest.mark.parametrize("name,causal", [("packed_4x4096_short", False), ("causal_2k_gqa", True),
                                         ("ragged_n300", False)])
def test_noalloc_matches_workspace_backward_twice(name, causal, cuda_dev):
    """N = 300 runs on whole tiles with a zero tail; its workspace fits in the scratch."""
    w = RAGGED if name == "ragged_n300" else synth.workload(name)
    q, k, v, do, seg = _inputs(w, cuda_dev)
    seg_arg = None if causal else seg
    out, lse = pa.forward(q, k, v, seg_arg)
    ref = pa.backward(q, k, v, out, do, lse, seg_arg)
    L = pa.lib()
    dims = pa.make_dims(w.B, w.Hq, w.Hkv, w.N, w.D)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        status = ctypes.c_uint32(0xFFFFFFFF)
        rc = L.pa_bwd_noalloc(ctypes.byref(dims), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              do.data_ptr(), lse.data_ptr(), None if causal else seg.data_ptr(), dq.data_ptr(),
                              dk.data_ptr(), dv.data_ptr(), ctypes.byref(status), stream)
        assert rc == 0, pa.pa_status_string(rc)
        assert status.value == 0, hex(status.value)
        torch.cuda.synchronize()
        for got, exp, n in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            assert torch.isfinite(got.float()).all(), (call, n)
            assert _rel(got, exp) <= GRAD_RELL2, (call, n, _rel(got, exp))


def _noalloc(L, w, q, k, v, out, do, lse, seg):
    dims = pa.make_dims(w.B, w.Hq, w.Hkv, w.N, w.D)
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
    status = ctypes.c_uint32(0xFFFFFFFF)
    rc = L.pa_bwd_noalloc(ctypes.byref(dims), q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          do.data_ptr(), lse.data_ptr(), None if seg is None else seg.data_ptr(), dq.data_ptr(),
                          dk.data_ptr(), dv.data_ptr(), ctypes.byref(status),
                          torch.cuda.current_stream().cuda_stream)
    assert rc == 0, pa.pa_status_string(rc)
    assert status.value == 0, hex(status.value)
    torch.cuda.synchronize()
    return dq, dk, dv


def test_noalloc_sequence_of_different_shapes(cuda_dev):
    """The shared array keeps whatever the previous call left in it: a large
    packed call, then a small causal one, then a ragged N that goes through
    whole tiles with a zero tail, then the large packed call again must each match
    pa_bwd with its own workspace."""
    L = pa.lib()
    runs = []
    for name, causal in (("packed_4x4096_short", False), ("causal_2k_gqa", True), ("ragged_n300", False)):
        w = RAGGED if name == "ragged_n300" else synth.workload(name)
        q, k, v, do, seg = _inputs(w, cuda_dev)
        seg_arg = None if causal else seg
        out, lse = pa.forward(q, k, v, seg_arg)
        runs.append((name, w, (q, k, v, out, do, lse, seg_arg), pa.backward(q, k, v, out, do, lse, seg_arg)))
    for name, w, args, ref in runs + runs[:1]:
        got = _noalloc(L, w, *args)
        for g, e, n in zip(got, ref, ("dq", "dk", "dv")):
            assert torch.isfinite(g.float()).all(), (name, n)
            assert _rel(g, e) <= GRAD_RELL2, (name, n, _rel(g, e))


def test_noalloc_refuses_dims_beyond_its_scratch(cuda_dev):
    L = pa.lib()
    big = pa.make_dims(4, 64, 8, 16384, 128)  # 4M query rows of delta: 16 MiB > 8 MiB
    assert L.pa_workspace_bytes(ctypes.byref(big)) > 8 << 20
    fake = 0x100000
    rc = L.pa_bwd_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, None, None)
    assert rc == 6  # PA_ERR_WORKSPACE, refused before anything touches the device
    bad = pa.make_dims(1, 4, 2, 256, 80)
    assert L.pa_bwd_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                            None, None) == 2  # PA_ERR_HEAD_DIM, from the same checks as pa_bwd
    # the same refusal without seg (plain causal): the causal checks name it too
    assert L.pa_bwd_noalloc(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, None, fake, fake, fake,
                            None, None) == 2
