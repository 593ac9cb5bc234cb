"""The FMA-pipe exponential on the device (pa_selftest_exp2_fma):
2^t to the fit's relative bound against fp64 exp2 for every input the
forward can pass (t in [-126, 8]), exact powers of two at integers, exactly
+0.0 from -127 down to -inf, and the host replay of the same fp32 steps
(fit_exp2_poly.py) to within one ulp (the replay may round an FMA twice)."""
import os
import sys

import numpy as np
import pytest
import torch

import segment_masked_causal_gb300 as pa

pytestmark = pytest.mark.gpu

sys.path.insert(0, os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                "segment_masked_causal_gb300", "csrc"))
import fit_exp2_poly as fit  # noqa: E402
from test_exp2_fma_host import kernel_constants  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from segment_masked_causal_gb300 import build
    build.build()


def run(x: np.ndarray, dev) -> np.ndarray:
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)
    yd = torch.empty_like(xd)
    pa.pa_selftest_exp2_fma(xd, yd)
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def test_exp2_fma_against_fp64(cuda_dev):
    rng = np.random.default_rng(7)
    x = np.concatenate([np.linspace(-126.0, 8.0, 1 << 20), rng.uniform(-30.0, 8.0, 1 << 18),
                        rng.uniform(-1.0, 1.0, 1 << 16)]).astype(np.float32)
    y = run(x, cuda_dev)
    assert not np.isnan(y).any(), "lane mismatch inside the routine"
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(y.astype(np.float64) / ref - 1.0)
    print(f"max relative error {rel.max():.3e}")
    assert rel.max() <= 1.05e-4
    host = fit.exp2_fp32(x, kernel_constants())
    ulps = np.abs(y.view(np.int32).astype(np.int64) - host.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


def test_exp2_fma_special_inputs(cuda_dev):
    n = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(run(n, cuda_dev).astype(np.float64), np.exp2(n.astype(np.float64)))
    z = np.array([-np.inf, -1e30, -300.0, -128.0, -127.5, -127.0], dtype=np.float32)
    assert np.all(run(z, cuda_dev).view(np.uint32) == 0)
    sub = np.linspace(-127.0, -126.0, 4097, dtype=np.float32)
    ys = run(sub, cuda_dev).astype(np.float64)
    assert np.all(ys >= 0) and np.all(ys < 2.0 ** -125)
