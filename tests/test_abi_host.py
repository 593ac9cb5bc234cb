"""The C ABI on the host (no GPU needed): the library builds and loads, exports
every function include/pa.h declares, and refuses bad arguments with typed
statuses before touching a device (mlx-train-perf 0.5.1 README, "When it
refuses": typed refusals, never silent fallbacks)."""
import ctypes
import os
import re

import pytest

import segment_masked_causal_gb300 as pa
from segment_masked_causal_gb300 import build as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    pabuild.build()
    return pa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert set(names) == set(pa.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def d(B=1, Hq=4, Hkv=2, N=256, D=128, scale=0.0):
    return pa.make_dims(B, Hq, Hkv, N, D, scale)


FAKE = 0x100000  # a 16-byte-aligned non-null address; never dereferenced on refusal


def fwd(L, dims, q=FAKE, k=FAKE, v=FAKE, seg=FAKE, out=FAKE, lse=FAKE, ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = 1 << 40
    return L.pa_fwd(ctypes.byref(dims), q, k, v, seg, out, lse, ws, ws_bytes, None)


def test_workspace_bytes(L):
    assert L.pa_workspace_bytes(ctypes.byref(d(D=80))) == 0
    assert L.pa_workspace_bytes(ctypes.byref(d(D=96))) == L.pa_workspace_bytes(ctypes.byref(d(D=128)))
    assert L.pa_workspace_bytes(None) == 0
    n1 = L.pa_workspace_bytes(ctypes.byref(d(N=256)))
    n2 = L.pa_workspace_bytes(ctypes.byref(d(N=512)))
    assert n1 > 0 and n2 > n1
    # status word + tile table + fp32 delta and fp32 lse*log2(e) per query row
    assert n2 >= 2 * 4 * 4 * 512 + 16 * 4


@pytest.mark.parametrize("dims,code", [
    (dict(D=80), 2), (dict(D=32), 2), (dict(D=256), 2),
    (dict(Hq=6, Hkv=4), 3),
    (dict(N=0), 4), (dict(B=0), 4), (dict(Hq=0), 4), (dict(Hkv=0), 4),
    (dict(B=1024, Hq=64, N=65536), 4),  # row coordinates overflow int32
])
def test_shape_refusals(L, dims, code):
    assert fwd(L, d(**dims)) == code


def test_null_and_alignment_refusals(L):
    assert L.pa_fwd(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 1
    assert fwd(L, d(), q=None) == 1
    assert fwd(L, d(), seg=None) == 1  # the packed entry point needs segment ids
    assert fwd(L, d(), ws=None) == 1
    assert fwd(L, d(), out=FAKE + 8) == 5
    assert fwd(L, d(), seg=FAKE + 4) == 5
    assert fwd(L, d(), ws=FAKE + 2) == 5
    need = L.pa_workspace_bytes(ctypes.byref(d()))
    assert fwd(L, d(), ws_bytes=need - 1) == 6
    dims = d()
    assert L.pa_bwd(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                    1 << 40, None) == 1
    assert L.pa_bwd_causal(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 1, FAKE,
                           1 << 40, None) == 5


def strides(q_b, q_h, q_n, k_b, k_h, k_n):
    return pa.pa_strides(q_b, q_h, q_n, k_b, k_h, k_n)


def test_ragged_n_and_strided_workspace(L):
    """For N not a multiple of 128 pa_workspace_bytes also counts the staging
    copies that fp32 calls use: (B, H, Np, D) buffers for q, out, dout, dq
    (Hq heads) and k, v, dk, dv (Hkv heads), plus lse and seg, with Np = N
    rounded up to 128 (bf16 calls need less and never more)."""
    base = L.pa_workspace_bytes(ctypes.byref(d(N=256)))
    ragged = L.pa_workspace_bytes(ctypes.byref(d(N=200)))
    assert ragged == L.pa_workspace_bytes_strided(ctypes.byref(d(N=200)))
    assert ragged == L.pa_workspace_bytes_strided(ctypes.byref(d(N=256)))
    B, Hq, Hkv, Np, D = 1, 4, 2, 256, 128
    assert ragged >= base + 4 * B * Hq * Np * D * 2 + 4 * B * Hkv * Np * D * 2 + 4 * B * Hq * Np + 4 * B * Np
    assert L.pa_workspace_bytes(ctypes.byref(d(N=1))) > 0


def test_ragged_n_refusals(L):
    """The single-step calls need whole tiles; the full calls take any N and
    then need the workspace of N rounded up to whole tiles."""
    dims = d(N=200)
    assert L.pa_fwd_tiles(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 4
    assert L.pa_build_tile_table(ctypes.byref(dims), FAKE, FAKE, 1 << 40, None) == 4
    assert L.pa_bwd_delta(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 4
    assert L.pa_bwd_dq(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 4
    assert L.pa_bwd_dkv(ctypes.byref(dims), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40,
                        None) == 4
    # bf16 with ragged N runs on whole tiles (N rounded up to 256 here) in
    # place: one byte below that workspace is refused before any launch
    base = L.pa_workspace_bytes(ctypes.byref(d(N=256)))
    assert fwd(L, dims, ws_bytes=base - 1) == 6
    assert fwd(L, dims, q=None) == 1


def test_strided_refusals(L):
    dims = d()
    good = strides(2 * 256 * 128 * 4, 128, 4 * 128, 256 * 2 * 128, 128, 2 * 128)  # (B, N, H, D) memory
    big = L.pa_workspace_bytes_strided(ctypes.byref(dims))

    def f(st, ws_bytes=big, seg=FAKE, q=FAKE, io=0):
        return L.pa_fwd_strided(ctypes.byref(dims), None if st is None else ctypes.byref(st), io, q, FAKE, FAKE,
                                seg, FAKE, FAKE, FAKE, ws_bytes, None)
    assert f(None) == 1
    assert f(strides(1 << 20, 128, 64, 1 << 20, 128, 256)) == 4  # q_n < D
    assert f(strides(1 << 20, 128, 132, 1 << 20, 128, 256)) == 5  # not a multiple of 8 bf16
    assert f(strides(1 << 20, 128, 130, 1 << 20, 128, 256), io=1) == 5  # not a multiple of 4 fp32
    assert f(good, io=2) == 9
    assert f(good, io=-1) == 9
    # bf16 with whole tiles runs in place whatever the strides: the plain
    # workspace is what it needs (one byte less is refused before any launch)
    plain = L.pa_workspace_bytes(ctypes.byref(dims))
    assert f(good, ws_bytes=plain - 1) == 6
    assert f(good, q=None) == 1
    assert f(good, seg=FAKE + 4) == 5
    # so do contiguous strides
    cont = strides(4 * 256 * 128, 256 * 128, 128, 2 * 256 * 128, 256 * 128, 128)
    assert f(cont, ws_bytes=plain - 1) == 6
    assert L.pa_bwd_strided(ctypes.byref(dims), None, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                            FAKE, FAKE, big, None) == 1
    assert L.pa_bwd_strided(ctypes.byref(dims), ctypes.byref(good), 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                            FAKE + 8, FAKE, FAKE, FAKE, big, None) == 5
    assert L.pa_bwd_strided(ctypes.byref(dims), ctypes.byref(good), 3, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                            FAKE, FAKE, FAKE, FAKE, big, None) == 9
    # fp32 I/O always stages, so the contiguous layout then needs the staged workspace too
    cont = strides(4 * 256 * 128, 256 * 128, 128, 2 * 256 * 128, 256 * 128, 128)
    assert f(cont, ws_bytes=L.pa_workspace_bytes(ctypes.byref(dims)), io=1) == 6


def test_selftest_refusals(L):
    """The bounded-wait self-test checks its workspace before any device call."""
    assert L.pa_selftest_wait_timeout(None, 1 << 20, None) == 1
    assert L.pa_selftest_wait_timeout(FAKE + 4, 1 << 20, None) == 5
    assert L.pa_selftest_wait_timeout(FAKE, 3, None) == 6
    # the FMA-pipe exponential's self-test: shape, null and alignment first
    assert L.pa_selftest_exp2_fma(FAKE, FAKE, -1, None) == 4
    assert L.pa_selftest_exp2_fma(FAKE, FAKE, 0, None) == 0  # nothing to do, no device call
    assert L.pa_selftest_exp2_fma(None, FAKE, 8, None) == 1
    assert L.pa_selftest_exp2_fma(FAKE, None, 8, None) == 1
    assert L.pa_selftest_exp2_fma(FAKE + 2, FAKE, 8, None) == 5


def test_valid_call_without_a_gpu_is_refused_not_run(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(L, d()) in (7, 8)  # no device: arch / CUDA error, nothing launched
    assert fwd(L, d(N=200)) in (7, 8)  # ragged N passes the host checks, then the same
    assert L.pa_selftest_wait_timeout(FAKE, 1 << 20, None) in (7, 8)
    assert L.pa_selftest_exp2_fma(FAKE, FAKE, 8, None) in (7, 8)


def test_status_strings(L):
    for c in range(11):
        assert L.pa_status_string(c) != b"unknown status"
    assert pa.pa_status_string(9).startswith("io dtype")
    assert pa.pa_status_string(2).startswith("head dim")


def test_lce_refusals(L):
    """The linear cross-entropy forward checks dims, pointers and workspace on
    the host before any device call."""
    assert L.pa_lce_workspace_bytes(256, 1000, 128) > 0
    assert L.pa_lce_workspace_bytes(0, 1000, 128) == 0
    assert L.pa_lce_workspace_bytes(256, 1000, 96) == 0  # D must be a multiple of 64
    big = 1 << 30

    def f(N=256, V=1000, D=128, h=FAKE, w=FAKE, t=FAKE, ws=FAKE, ws_bytes=big):
        return L.pa_lce_fwd(N, V, D, h, w, t, FAKE, FAKE, FAKE, ws, ws_bytes, None)
    assert f(N=0) == 4
    assert f(V=0) == 4
    assert f(D=96) == 4
    assert f(D=32) == 4
    assert f(h=None) == 1
    assert f(ws=None) == 1
    assert f(w=FAKE + 8) == 5
    assert f(t=FAKE + 4) == 5
    assert f(ws_bytes=L.pa_lce_workspace_bytes(256, 1000, 128) - 1) == 6
