"""The matmul acceptance bar, applied element by element.

Per element: |Y - Yo| <= 2e-2 * ||x_m|| * ||Wd_n|| / sqrt(K), with the norms of
that token row and of that (fp32 dequantized) weight row; per tensor: relative
Frobenius error <= 5e-3.  Yo is the fp64 oracle.
"""
import numpy as np
import torch

from oracle import q1_oracle as O

REL_ELEM = 2e-2
REL_FRO = 5e-3


def check_matmul(y_gpu, y_oracle, x, wd_f32, what=""):
    y = y_gpu.detach().float().cpu().double().numpy() if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu, dtype=np.float64)
    yo = np.asarray(y_oracle, dtype=np.float64)
    y = y.reshape(yo.shape)
    bound = O.tolerance_bound(x, wd_f32, REL_ELEM).reshape(yo.shape)
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
