"""The bounded waits' timeout path, exercised on the GPU without a fault.

q1_set_stalled_producers makes the producers of later launches issue no
copies: every wait for their data then runs out (with a 1 ms limit from
q1_set_wait_limit_ns), and no copy is in flight when the kernels give up.
The call must return, q1_device_errors must report the timeout (bit 1:
narrow kernels, bit 0: prefill kernels) and clear it, and a normal call
afterwards must be clean and correct.
"""
import time

import pytest
import torch

from oracle import q1_oracle as O
from bit_affine_quantized_g128_gb300 import synth
from tests.tolerance import check_matmul

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def q1():
    from bit_affine_quantized_g128_gb300 import q1 as mod
    mod.load_library()
    return mod


@pytest.mark.parametrize("path,M,bit", [("narrow", 4, 2), ("prefill", 300, 1)])
def test_stalled_producers_time_out_and_recover(q1, path, M, bit):
    N, K = 768, 2048
    t = synth.q1_tensor(N, K, seed=931, affine=True)
    x = synth.activations(M, K, seed=932)
    W = q1.Q1Weight.from_host(t)
    xd = x.to(DEV)
    ws = q1.qmm_workspace(M, N, K, DEV)
    assert q1.device_errors() == 0
    try:
        q1.set_wait_limit_ns(1_000_000)
        q1.set_stalled_producers(True)
        t0 = time.perf_counter()
        q1.qmm(W, xd, workspace=ws)
        flags = q1.device_errors()  # synchronizes
        elapsed = time.perf_counter() - t0
    finally:
        q1.set_stalled_producers(False)
        q1.set_wait_limit_ns(0)
    assert flags & bit, f"{path}: no timeout reported (flags {flags})"
    assert elapsed < 10.0, f"{path}: the timed-out call took {elapsed:.1f} s"
    assert q1.device_errors() == 0  # read and cleared
    y = q1.qmm(W, xd, workspace=ws)
    assert q1.device_errors() == 0
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"{path} after the timeout")


def test_wait_controls_validate_and_restore(q1):
    # the default limit comes back with 0; a normal call under it is clean
    q1.set_wait_limit_ns(0)
    q1.set_stalled_producers(False)
    t = synth.q1_tensor(256, 512, seed=933, affine=False)
    x = synth.activations(1, 512, seed=934)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmv(W, x[0].to(DEV))
    assert q1.device_errors() == 0
    check_matmul(y.reshape(1, -1), O.qmm(x, t.words, t.scales, None, 512), x,
                 O.dequantize_f32(t.words, t.scales, None, 512), "qmv under the default limit")
