"""Bounded waits: with the wait limit at zero every kernel gives up on its first
unsatisfied wait, records CONV_ERR_TIMEOUT in the device status word, drains
its copies and MMAs in flight, frees its tensor memory and returns -- no
fault, no hang.  The context stays usable: the next call at the normal limit
is correct."""
import numpy as np
import pytest
import torch

import conv_workloads as cw
from _gpu_util import as_f64, assert_close, oracle_conv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import implicit_gemm_convolution_conv3d_gb300 as p
    p.load_library()
    return p


def test_forced_wait_timeout_reports_status_and_recovers(pkg):
    x = cw.randn_bf16((2, 5, 9, 11, 64), 600, 1.0, "cuda")
    w = cw.randn_bf16((96, 3, 3, 3, 64), 601, 1.0 / np.sqrt(1728), "cuda")
    assert pkg.conv_get_device_status() == 0
    try:
        pkg.conv_set_wait_limit_ns(0)
        pkg.conv_fwd(x, w, 1, 1, 1, split_k=False)
        status = pkg.conv_get_device_status()
    finally:
        pkg.conv_set_wait_limit_ns(2_000_000_000)
    assert status == pkg.CONV_ERR_TIMEOUT
    y = pkg.conv_fwd(x, w, 1, 1, 1)
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status() == 0
    assert_close(as_f64(y), oracle_conv(x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1)), "after timeout")


def test_forced_timeout_read_in_stream_order(pkg):
    """conv_get_device_status_stream reads the word after the stream's queued
    work and synchronises that stream only: the forced timeout of a conv on
    a side stream is reported there, the word is cleared, and a later
    conv on that stream reads back CONV_OK."""
    x = cw.randn_bf16((2, 5, 9, 11, 64), 602, 1.0, "cuda")
    w = cw.randn_bf16((96, 3, 3, 3, 64), 603, 1.0 / np.sqrt(1728), "cuda")
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    assert pkg.conv_get_device_status_stream(side) == 0
    try:
        pkg.conv_set_wait_limit_ns(0)
        with torch.cuda.stream(side):
            pkg.conv_fwd(x, w, 1, 1, 1, split_k=False)
        status = pkg.conv_get_device_status_stream(side)
    finally:
        pkg.conv_set_wait_limit_ns(2_000_000_000)
    assert status == pkg.CONV_ERR_TIMEOUT
    with torch.cuda.stream(side):
        y = pkg.conv_fwd(x, w, 1, 1, 1)
    assert pkg.conv_get_device_status_stream(side) == 0
    assert_close(as_f64(y), oracle_conv(x, w, (1, 1, 1), (1, 1, 1), (1, 1, 1)), "side stream")
