"""q1_ffn_fused_noalloc: the fused FFN with its intermediate in the library's
fixed device array.  Collected last (file name), and independent of what ran
before it: two calls in a row must match q1_ffn_fused (same kernels, so bit
for bit), the largest shape that fits must run, and one past it must be
refused without touching the output.
"""
import numpy as np
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


def _ffn(q1, D, F, seed, affine=False):
    ts = [synth.q1_tensor(F, D, seed=seed, affine=affine), synth.q1_tensor(F, D, seed=seed + 1, affine=affine),
          synth.q1_tensor(D, F, seed=seed + 2, affine=affine)]
    return ts, [q1.Q1Weight.from_host(t) for t in ts]


def test_two_calls_match_workspace_path(q1):
    # call 1: M = 8, D = 1024, F = 2048, symmetric; call 2: M = 3, affine,
    # other weights and x.  Each must equal q1_ffn_fused bit for bit.
    first = None
    for (M, D, F, seed, affine) in [(8, 1024, 2048, 31, False), (3, 512, 1024, 41, True)]:
        ts, (G, U, Dn) = _ffn(q1, D, F, seed, affine)
        x = synth.activations(M, D, seed=seed + 9).to(DEV)
        y_na = q1.ffn_fused_noalloc(G, U, Dn, x)
        y_ws = q1.ffn_fused(G, U, Dn, x)
        torch.cuda.synchronize()
        assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16)), (M, D, F)
        if first is None:
            first = (ts, x.cpu(), y_na.float().cpu().double().numpy(), D, F)
    # the first (symmetric) call against the oracle as well
    ts, xo, y, D, F = first
    yo, ho = O.ffn(xo, (ts[0].words, ts[0].scales, None, D), (ts[1].words, ts[1].scales, None, D),
                   (ts[2].words, ts[2].scales, None, F))
    check_matmul(y, yo, ho, O.dequantize_f32(ts[2].words, ts[2].scales, None, F), "noalloc ffn")


def test_largest_shape_and_refusal(q1):
    cap = q1.FFN_NOALLOC_BYTES
    M, D = 8, 256
    F = cap // (2 * M)  # exactly fills the array
    ts, (G, U, Dn) = _ffn(q1, D, F, seed=51)
    x = synth.activations(M, D, seed=52).to(DEV)
    y_na = q1.ffn_fused_noalloc(G, U, Dn, x)
    y_ws = q1.ffn_fused(G, U, Dn, x)
    torch.cuda.synchronize()
    assert torch.equal(y_na.view(torch.int16), y_ws.view(torch.int16))
    # one group of rows more does not fit: refused, output untouched
    F2 = F + 128
    _, (G2, U2, D2) = _ffn(q1, D, F2, seed=61)
    y = torch.full((M, D), 7.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(q1.Q1Error) as e:
        q1.ffn_fused_noalloc(G2, U2, D2, x, out=y)
    assert e.value.status == 6  # Q1_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y.float() == 7.0).all())
