"""The matmul acceptance bar, applied element by element.

Per element: |Y - Yo| <= 2e-2 * ||x_m|| * ||Wd_n|| / sqrt(K), with the norms of
that token row and of that (fp32 dequantized) weight row; per tensor: relative
Frobenius error <= 5e-3.  Yo is the fp64 oracle.

Outputs far larger than ||x_m|| ||Wd_n|| / sqrt(K): affine weights have a
non-zero mean per group (scale/2 + bias), and when the activations share a
systematic component with those means (the FFN's h = SiLU(g) * u is one: the
affine gate and up rows see the same group sums of x) the product grows like
K instead of sqrt(K).  Rounding the exact result once to the output dtype then
already moves it by more than the per-element bar (up to 2.3x for bf16 at the
27B-class FFN shape).  For such products the bar adds half a unit in the last
place of |Yo| in the output dtype (`rounded_to`): the error a perfect result
stored in that dtype has.  The Frobenius bar is unchanged.
"""
import numpy as np
import torch

from oracle import q1_oracle as O

REL_ELEM = 2e-2
REL_FRO = 5e-3


# significand bits (with the implicit one) of the output dtypes, and the
# exponent of their smallest normal number
_SIG = {"bf16": (8, -126), "f16": (11, -14), "f32": (24, -126)}


def half_ulp(y, dtype: str) -> np.ndarray:
    """Half a unit in the last place of |y| in `dtype` ('bf16', 'f16', 'f32').

    The binade is taken from |y| * (1 + 2^-6), so that a result just below a
    power of two that rounds up into the next binade is covered; subnormal
    outputs get the half-ulp of the smallest normal binade."""
    p, emin = _SIG[dtype]
    a = np.abs(np.asarray(y, dtype=np.float64)) * (1.0 + 2.0 ** -6)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return np.ldexp(1.0, (e - p).astype(np.int64))


def check_matmul(y_gpu, y_oracle, x, wd_f32, what="", rounded_to=None):
    y = y_gpu.detach().float().cpu().double().numpy() if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu, dtype=np.float64)
    yo = np.asarray(y_oracle, dtype=np.float64)
    y = y.reshape(yo.shape)
    bound = O.tolerance_bound(x, wd_f32, REL_ELEM).reshape(yo.shape)
    if rounded_to is not None:
        bound = bound + half_ulp(yo, rounded_to)
    err = np.abs(y - yo)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    assert np.all(err <= bound), (f"{what}: element {worst} err {err[worst]:.3e} > bound "
                                  f"{bound[worst]:.3e} (y={y[worst]:.6e}, oracle={yo[worst]:.6e})")
    fro = np.linalg.norm(y - yo) / max(np.linalg.norm(yo), 1e-300)
    assert fro <= REL_FRO, f"{what}: relative Frobenius error {fro:.3e} > {REL_FRO}"
    return fro


def check_chain(y_gpu, y_oracle, h_last, wd_last, stages, what=""):
    """The matmul bar for a chain of `stages` products, on its final output.

    A product's error, fed into the next product, reaches that product's output
    at about the same size relative to ||x|| ||w_n|| / sqrt(K) (the weights are
    unrelated to the error), so the errors of the stages add: the final output
    is held to `stages` times the per-element bound of its own product (norms of
    that product's input h_last, fp64 oracle, and of its weight rows) and to
    `stages` times the relative Frobenius bound.
    """
    y = y_gpu.detach().float().cpu().double().numpy()
    yo = np.asarray(y_oracle, dtype=np.float64).reshape(y.shape)
    bound = stages * O.tolerance_bound(h_last, wd_last, REL_ELEM).reshape(y.shape)
    err = np.abs(y - yo)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    assert np.all(err <= bound), (f"{what}: element {worst} err {err[worst]:.3e} > bound "
                                  f"{bound[worst]:.3e} (y={y[worst]:.6e}, oracle={yo[worst]:.6e})")
    fro = np.linalg.norm(y - yo) / max(np.linalg.norm(yo), 1e-300)
    assert fro <= stages * REL_FRO, f"{what}: relative Frobenius error {fro:.3e} > {stages * REL_FRO}"
    return fro
