"""Failure detection on the GPU without a fault: the bounded mbarrier waits give up, record
MX_ERR_TIMEOUT in the library's watchdog words, and the CUDA context stays usable.

The self-test kernels wait on barriers that nothing ever arrives on (no copy or MMA is issued), with
a limit of about a millisecond.  The GEMM unit runs as a cluster of two CTAs with the pair's TMEM
allocated and leaves through the GEMMs' exit path (abort flag, cluster barrier, TMEM release).
Failure detection is in scope because the E2E page's Tables 11-13 list the checks a low-precision
RL run keeps and the faults they catch."""
import time

import numpy as np
import pytest
import torch

import synthetic
from gpu_util import DEV

pytestmark = pytest.mark.gpu
LIMIT_NS = 1_000_000      # 1 ms


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_numerics_gb300 as m
    m.lib()
    return m


def tiny_mxfp8_gemm_matches_oracle(mx, orc):
    """A normal call after the expiry: MXFP8 quantize + FPROP on the tiny configuration, checked
    against the oracle (codes bit-exact, GEMM within 1e-2)."""
    d = synthetic.tiny()
    x_np, w_np = d["x"], d["w"]
    M, K = x_np.shape
    N = w_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    w = torch.from_numpy(w_np.view(np.int16)).to(DEV).view(torch.bfloat16)
    ox, ow = mx.alloc_mxfp8(M, K, DEV), mx.alloc_mxfp8(N, K, DEV)
    mx.mx_quantize_mxfp8(x, **ox)
    mx.mx_quantize_mxfp8(w, **ow)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=DEV)
    mx.mx_scaled_gemm(mx.MX_FMT_MXFP8, ox["q_row"], ox["s_row"], None, 0, ow["q_row"], ow["s_row"], None, 0, M, N, K, y)
    assert mx.mx_check_device_status() == mx.MX_OK
    qx, sx = orc.mxfp8_quantize_rowwise(x_np)
    qw, sw = orc.mxfp8_quantize_rowwise(w_np)
    assert np.array_equal(ox["q_row"].cpu().numpy(), qx)
    assert np.array_equal(ow["q_row"].cpu().numpy(), qw)
    err = orc.rel_fro_error(y.float().cpu().numpy().astype(np.float64), orc.gemm_ref_mxfp8(qx, sx, qw, sw))
    assert err <= 1e-2, err


@pytest.mark.parametrize("unit", ["gemm", "mxfp8"])
def test_wait_expires_reports_timeout_once_then_clears(mx, orc, unit):
    u = mx.MX_WATCHDOG_GEMM if unit == "gemm" else mx.MX_WATCHDOG_MXFP8
    assert mx.mx_check_device_status() == mx.MX_OK          # nothing pending before the test
    t0 = time.perf_counter()
    mx.mx_watchdog_selftest(u, LIMIT_NS)
    assert mx.mx_check_device_status() == mx.MX_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert elapsed < 1.0, f"the waits took {elapsed:.3f} s to give up (limit {LIMIT_NS} ns)"
    assert mx.mx_check_device_status() == mx.MX_OK          # the word was cleared by the read
    tiny_mxfp8_gemm_matches_oracle(mx, orc)


def test_stream_status_on_a_side_stream(mx, orc):
    side = torch.cuda.Stream()
    assert mx.mx_check_stream_status(side) == mx.MX_OK
    mx.mx_watchdog_selftest(mx.MX_WATCHDOG_GEMM, LIMIT_NS, stream=side)
    assert mx.mx_check_stream_status(side) == mx.MX_ERR_TIMEOUT
    assert mx.mx_check_stream_status(side) == mx.MX_OK
    assert mx.mx_check_device_status() == mx.MX_OK
    tiny_mxfp8_gemm_matches_oracle(mx, orc)


def test_every_unit_expires_in_one_launch_sequence(mx, orc):
    """Both words set by back-to-back expiries are reported by one check and cleared together."""
    mx.mx_watchdog_selftest(mx.MX_WATCHDOG_GEMM, LIMIT_NS)
    mx.mx_watchdog_selftest(mx.MX_WATCHDOG_MXFP8, LIMIT_NS)
    assert mx.mx_check_device_status() == mx.MX_ERR_TIMEOUT
    assert mx.mx_check_device_status() == mx.MX_OK
