"""Seeded synthetic inputs for the Q1 (1-bit affine, group size 128) linear layer.

This module is shared by the CPU oracle side and the CUDA side of the tests and
the benchmark.  It only draws random numbers with the distributions that the
pages' workloads describe; it holds none of the method's arithmetic (no
unpacking, no dequantization, no matmul).

Distributions (the synthetic stand-in for the Bonsai-27B checkpoint that the
"Support Bonsai-27B affine Q1" page measures on, which is not available here):

* packed weight words: uniform random uint32, i.e. every weight bit is an
  independent Bernoulli(0.5) draw.  Element (n, k) is bit k % 32 of word
  [n][k // 32] (the MLX affine bits=1 layout described on the rMLX issue page,
  "The good news - packing is standard").
* scales: fp16(|N(0, 0.02)| + 1e-4), one per row and group of 128.
* affine biases: fp16(N(0, 0.01)), drawn independently of the scales.
* activations: bf16(N(0, 1)).
* token ids: uniform in [0, V).

Every function takes an explicit integer seed and uses numpy's PCG64 stream, so
the same call returns the same values in every process on the same numpy.
"""
from __future__ import annotations

import numpy as np
import torch

GROUP = 128          # weights per scale/bias group along K
BITS_PER_WORD = 32   # weights per packed uint32 word


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def weight_words(N: int, K: int, seed: int) -> np.ndarray:
    """uint32 [N, K/32]: uniform random packed weight words."""
    if K % BITS_PER_WORD:
        raise ValueError("K must be a multiple of 32")
    return _rng(seed).integers(0, 2**32, size=(N, K // BITS_PER_WORD), dtype=np.uint32)


def scales(N: int, K: int, seed: int, group: int = GROUP) -> np.ndarray:
    """fp16 [N, K/group]: |N(0, 0.02)| + 1e-4, rounded to fp16."""
    g = _rng(seed).standard_normal((N, K // group), dtype=np.float32)
    return (np.abs(g * np.float32(0.02)) + np.float32(1e-4)).astype(np.float16)


def biases(N: int, K: int, seed: int, group: int = GROUP) -> np.ndarray:
    """fp16 [N, K/group]: N(0, 0.01), rounded to fp16 (affine metadata)."""
    g = _rng(seed).standard_normal((N, K // group), dtype=np.float32)
    return (g * np.float32(0.01)).astype(np.float16)


def activations(M: int, K: int, seed: int) -> torch.Tensor:
    """bf16 [M, K] CPU tensor: N(0, 1) rounded to bf16."""
    g = _rng(seed).standard_normal((M, K), dtype=np.float32)
    return torch.from_numpy(g).to(torch.bfloat16)


def token_ids(T: int, V: int, seed: int) -> np.ndarray:
    """int32 [T]: uniform token ids in [0, V)."""
    return _rng(seed).integers(0, V, size=(T,), dtype=np.int32)


def bits(N: int, K: int, seed: int) -> np.ndarray:
    """uint8 [N, K] of 0/1 values, Bernoulli(0.5) (input of the pack step)."""
    return _rng(seed).integers(0, 2, size=(N, K), dtype=np.uint8)


class Q1Tensor:
    """Host-side bundle of one synthetic Q1 weight: words, scales, biases.

    ``biases`` is None for symmetric metadata (bias derived as -scale/2 by the
    consumer; it is never stored).
    """

    def __init__(self, words: np.ndarray, scales_: np.ndarray,
                 biases_: np.ndarray | None, K: int):
        self.words = words
        self.scales = scales_
        self.biases = biases_
        self.N = words.shape[0]
        self.K = K

    @property
    def symmetric(self) -> bool:
        return self.biases is None


def q1_tensor(N: int, K: int, seed: int, affine: bool, group: int = GROUP) -> Q1Tensor:
    """A full synthetic Q1 weight (metadata per `group` weights along K).
    Sub-streams: seed (words), seed+7919 (scales), seed+15485863 (biases)."""
    w = weight_words(N, K, seed)
    s = scales(N, K, seed + 7919, group)
    b = biases(N, K, seed + 15485863, group) if affine else None
    return Q1Tensor(w, s, b, K)


def device_weight_words(N: int, K: int, seed: int, device) -> torch.Tensor:
    """int32 view of uniform random words generated directly on a device.

    Used where a benchmark needs gigabytes of weights (more than the host can
    draw quickly); the bits are as uniform as the host stream, but the values
    differ from :func:`weight_words` for the same seed.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randint(-2**31, 2**31, (N, K // BITS_PER_WORD), dtype=torch.int32,
                         device=device, generator=g)


def device_scales(N: int, K: int, seed: int, device) -> torch.Tensor:
    """fp16 scales |N(0,0.02)|+1e-4 generated on a device (benchmark bulk)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    r = torch.randn((N, K // GROUP), dtype=torch.float32, device=device, generator=g)
    return (r.abs() * 0.02 + 1e-4).to(torch.float16)


def device_biases(N: int, K: int, seed: int, device) -> torch.Tensor:
    """fp16 biases N(0,0.01) generated on a device (benchmark bulk)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    r = torch.randn((N, K // GROUP), dtype=torch.float32, device=device, generator=g)
    return (r * 0.01).to(torch.float16)
