"""CPU oracle for the 1-bit affine group-quantized (g128) linear layer.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke entry point and
the benchmark's CPU-baseline leg may import this module.  The product path (the
CUDA library and its Python binding) never calls it, and this module never
imports the product: the two share no code.  The only shared module is the
seeded input generator (bit_affine_quantized_g128_gb300/synth.py), which holds
none of the method's arithmetic.

It is a plain, slow, obviously correct restatement of what the method computes,
written from the definitions on the pages:

* "Support Bonsai-27B affine Q1" (higgs PR #212), section "What": every affine
  1-bit weight is w = scale * q + bias with q in {0, 1}; symmetric tensors have
  bias = -scale / 2, derived from the scale instead of stored.  Section
  "Limitations / non-goals": forwards wider than the narrow threshold
  dequantize to the input dtype and run a dense matmul.
* "1-bit affine weight support" (rMLX issue #207), section "The good news -
  packing is standard": 32 weights per uint32, fp16 scales and biases per group
  of 128, bit 0 maps to the negative value and bit 1 to the positive one.
* "Bonsai masked gemv" (cactus PR #775): the packed layout is the linear
  LSB-first layout (weight k of a 32-weight run sits at bit k).

Precision: dequantized values are formed in fp32 (one rounding for s + b), and
every dot product is accumulated in fp64.  A library matmul in fp64 serves as
the dot-product step.  Where a result is rounded to bf16/fp16 (dequantize,
gather), torch's CPU round-to-nearest-even conversion does it.

Every function here is pinned by tests/test_oracle_pins.py against facts that
do not come from this module (hand-built words, closed forms, exact rational
brute force, invariants).
"""
from __future__ import annotations

import numpy as np
import torch

GROUP_SIZE = 128
WORD_BITS = 32

_TORCH_DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


# ---------------------------------------------------------------------------
# Packing (rMLX issue, "packing is standard"; cactus PR, "linear LSB layout")
# ---------------------------------------------------------------------------
def unpack(words: np.ndarray, K: int) -> np.ndarray:
    """Packed uint32 [N, K/32] -> bits uint8 [N, K].

    q(n, k) = (words[n][k // 32] >> (k % 32)) & 1: the lowest bit of a word is
    the first of its 32 weights.
    """
    words = np.asarray(words, dtype=np.uint32)
    N = words.shape[0]
    out = np.empty((N, K), dtype=np.uint8)
    for j in range(WORD_BITS):
        # weights k = 32*c + j for every word c
        out[:, j::WORD_BITS] = ((words >> np.uint32(j)) & np.uint32(1)).astype(np.uint8)
    return out


def pack(bits: np.ndarray) -> np.ndarray:
    """bits uint8 [N, K] (values 0/1) -> packed uint32 [N, K/32], LSB first."""
    bits = np.asarray(bits)
    N, K = bits.shape
    if K % WORD_BITS:
        raise ValueError("K must be a multiple of 32")
    words = np.zeros((N, K // WORD_BITS), dtype=np.uint32)
    for j in range(WORD_BITS):
        words |= (bits[:, j::WORD_BITS].astype(np.uint32) & np.uint32(1)) << np.uint32(j)
    return words


# ---------------------------------------------------------------------------
# Metadata ("Support Bonsai-27B affine Q1", section "What": bias = -scale/2)
# ---------------------------------------------------------------------------
def meta32(m) -> np.ndarray:
    """Metadata values widened to fp32, exactly.

    fp16 arrays (the rMLX checkpoint's F16 scales+biases) and bf16 tensors
    (the Bonsai image checkpoint's BF16 scales/biases) both widen without
    rounding; an fp32 array is taken as already widened (e.g. bf16 values
    held in fp32).  Any other dtype is rounded to fp16 first.
    """
    if isinstance(m, torch.Tensor):
        return m.detach().to(torch.float32).numpy()
    m = np.asarray(m)
    if m.dtype == np.float32:
        return m
    return m.astype(np.float16).astype(np.float32)


def _take_rows(m, rows):
    """Rows of a metadata array or tensor (fp16 array or bf16 tensor)."""
    if isinstance(m, torch.Tensor):
        return m[torch.as_tensor(rows)] if not isinstance(rows, slice) else m[rows]
    return np.asarray(m)[rows]


def group_size_of(K: int, s) -> int:
    """Weights per scale along K, from the metadata's shape [N, K / group]:
    128 for every checkpoint on the pages; MLX's affine format also has 32 and
    64 ("1-bit affine weight support", rMLX issue #207: mlx#3161's
    "group_size=32 occupancy" edge case)."""
    G = np.asarray(s.shape)[1]
    if G < 1 or K % G or (K // G) not in (32, 64, 128):
        raise ValueError(f"metadata of {G} groups does not fit K = {K}")
    return K // G


def resolve_metadata(scales, biases):
    """Scales/biases [N, G] (fp16 or bf16, see meta32) -> (s, b) in fp32.

    Affine: b = fp32(bias).  Symmetric (biases is None): b = -0.5 * s in fp32,
    which is exact (halving an fp16 or bf16 value in fp32 never rounds).
    """
    s = meta32(scales)
    if biases is None:
        b = np.float32(-0.5) * s
    else:
        b = meta32(biases)
    return s, b


def is_symmetric(scales: np.ndarray, biases: np.ndarray) -> bool:
    """True iff every stored bias equals -scale/2 exactly (compared in fp32).

    The page's loader compacts "exact symmetric" biases only; one group that
    differs keeps the general affine path.  +0 and -0 compare equal; a NaN
    never equals anything, so a NaN scale or bias reads as affine.
    """
    s, b = resolve_metadata(scales, biases)
    derived = np.float32(-0.5) * s
    return bool(np.all(b == derived))


# ---------------------------------------------------------------------------
# Dequantization (w = scale * q + bias, q in {0, 1})
# ---------------------------------------------------------------------------
def dequantize_f32(words: np.ndarray, scales: np.ndarray, biases: np.ndarray | None,
                   K: int) -> np.ndarray:
    """Dense fp32 weights [N, K].

    q = 0 gives the bias itself (bit for bit); q = 1 gives fl32(s + b), one
    fp32 rounding.  Symmetric metadata therefore gives exactly -s/2 and +s/2.
    """
    q = unpack(words, K)
    s, b = resolve_metadata(scales, biases)
    gs = group_size_of(K, s)
    s_k = np.repeat(s, gs, axis=1)                  # [N, K]
    b_k = np.repeat(b, gs, axis=1)
    one = (s_k + b_k).astype(np.float32)            # fl32(s + b)
    return np.where(q == 1, one, b_k).astype(np.float32)


def round_to(values_f32: np.ndarray, dtype: str) -> torch.Tensor:
    """fp32 array -> CPU tensor of `dtype` ('bf16', 'f16', 'f32'), one RNE."""
    t = torch.from_numpy(np.array(values_f32, dtype=np.float32, copy=True))
    return t.to(_TORCH_DTYPES[dtype])


def dequantize(words, scales, biases, K: int, dtype: str = "bf16") -> torch.Tensor:
    """Dense weights [N, K] in `dtype`: the fp32 dequantized value, rounded once."""
    return round_to(dequantize_f32(words, scales, biases, K), dtype)


# ---------------------------------------------------------------------------
# Matmul (decode QMV, narrow and wide QMM all compute the same product)
# ---------------------------------------------------------------------------
def _x64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def qmm(x, words, scales, biases, K: int, rows=None) -> np.ndarray:
    """Y[m][n] = sum_k x[m][k] * Wd[n][k], accumulated in fp64.

    x: [M, K] (bf16 tensor or array; widened exactly to fp64).
    rows: optional index array of output features n to compute (the others are
    not evaluated); the result then has shape [M, len(rows)].
    """
    if rows is not None:
        rows = np.asarray(rows)
        words = np.asarray(words)[rows]
        scales = _take_rows(scales, rows)
        biases = None if biases is None else _take_rows(biases, rows)
    wd = dequantize_f32(words, scales, biases, K).astype(np.float64)
    x64 = _x64(x)
    if x64.ndim == 1:
        x64 = x64[None, :]
    return x64 @ wd.T


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(g) = g / (1 + exp(-g)) in fp64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def ffn(x, gate, up, down, rows=None) -> np.ndarray:
    """Dense FFN block: y = Down . (SiLU(Gate . x) * (Up . x)).

    gate/up/down are (words, scales, biases, K) tuples.  g, u and h are kept in
    fp64 with no intermediate rounding.  rows selects output features of the
    down projection (all when None).  Returns (y [M, D'], h [M, F]).
    """
    g = qmm(x, *gate)
    u = qmm(x, *up)
    h = silu(g) * u
    y = qmm(h, *down, rows=rows)
    return y, h


def decode_chain(x, layers) -> torch.Tensor:
    """Synthetic decode chain: the Q1 linears of a decode step, layer after layer
    ("Support Bonsai-27B affine Q1", section "Measured impact": the decode time
    of a model whose linears are all Q1; no attention, norms or residuals).

    Per layer, with h_0 = x: a = attn . h_l, then
    h_{l+1} = Down . (SiLU(Gate . a) * (Up . a)).  The chain passes bf16
    activations from one call to the next (every call takes and returns bf16
    activations), so a and h_{l+1} are each rounded once to bf16; inside a
    product and inside the FFN nothing is rounded (fp64, as in qmm and ffn).

    layers: sequence of (attn, gate, up, down), each a (words, scales, biases,
    K) tuple.  x: [M, D].  Returns h_L as a bf16 tensor [M, D].
    """
    h = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.asarray(x))
    h = h.to(torch.bfloat16)
    for attn, gate, up, down in layers:
        a = round_to(qmm(h, *attn), "bf16")
        y, _ = ffn(a, gate, up, down)
        h = round_to(y, "bf16")
    return h


# ---------------------------------------------------------------------------
# Embedding gather ("Support Bonsai-27B affine Q1": Q1 embeddings, tied head)
# ---------------------------------------------------------------------------
def embed_gather(ids, words, scales, biases, K: int, dtype: str = "bf16"):
    """out[t] = dequantized row ids[t], rounded to `dtype`.

    An id outside [0, V) gives a zero row and is counted.  Returns
    (out tensor [T, K], number of out-of-range ids).
    """
    ids = np.asarray(ids, dtype=np.int64)
    V = np.asarray(words).shape[0]
    T = ids.shape[0]
    out = np.zeros((T, K), dtype=np.float32)
    bad = 0
    for t in range(T):
        r = int(ids[t])
        if r < 0 or r >= V:
            bad += 1
            continue
        b_row = None if biases is None else _take_rows(biases, slice(r, r + 1))
        out[t] = dequantize_f32(np.asarray(words)[r:r + 1], _take_rows(scales, slice(r, r + 1)),
                                b_row, K)[0]
    return round_to(out, dtype), bad


# ---------------------------------------------------------------------------
# Exact repack from dense ("Bonsai masked gemv", cactus PR #775: tensors whose
# 128-groups hold exactly two values repack with zero quantization error;
# anything else is refused)
# ---------------------------------------------------------------------------
# Order in which fp16 scales around RN16(hi - lo) are tried, in fp16 steps.
SCALE_STEPS = (0, -1, 1, -2, 2)


def _bits32(v) -> int:
    return int(np.array(v, dtype=np.float32).view(np.uint32))


def _f16_step(h: np.float16, k: int) -> np.float16:
    toward = np.float16(np.inf) if k > 0 else np.float16(-np.inf)
    for _ in range(abs(k)):
        h = np.nextafter(h, toward)
    return h


def pack_group(vals, symmetric: bool):
    """Repack one group of 128 fp32 values exactly, or refuse (None).

    Values are compared by bit pattern, so +0 and -0 are distinct values and
    any NaN or infinity refuses the group.  With two values lo < hi (-0 < +0),
    weight bits are 1 where the value is hi.  Returns (bits [128] uint8,
    scale fp16, bias fp16 or None), the metadata chosen as follows:

    * symmetric: scale = RN16(-2 lo) (one value v: scale = RN16(2v) with all
      bits 1 if v's sign bit is clear, else RN16(-2v) with all bits 0), kept
      only if the derived bias -0.5 * scale is lo and fl32(scale + bias) is hi,
      bit for bit;
    * affine: bias = RN16(lo), which must give lo back exactly; scale = the
      first of RN16(fl32(hi - lo)) and its fp16 neighbours in SCALE_STEPS
      order with fl32(scale + bias) == hi bit for bit (one value: bias = v,
      scale = +0, all bits 0).
    """
    v = np.asarray(vals, dtype=np.float32).reshape(-1)
    if not np.all(np.isfinite(v)):
        return None
    pats = v.view(np.uint32)
    distinct = list(dict.fromkeys(int(p) for p in pats))
    if len(distinct) > 2:
        return None
    f = [np.array(p, dtype=np.uint32).view(np.float32)[()] for p in distinct]
    if len(distinct) == 1:
        x = f[0]
        if symmetric:
            neg = (distinct[0] >> 31) == 1
            sc = np.float16(np.float32(-2.0) * x if neg else np.float32(2.0) * x)
            b = np.float32(-0.5) * np.float32(sc)
            val = b if neg else np.float32(np.float32(sc) + b)
            if _bits32(val) != distinct[0]:
                return None
            bits = np.full(v.shape, 0 if neg else 1, dtype=np.uint8)
            return bits, sc, None
        bias = np.float16(x)
        if _bits32(np.float32(bias)) != distinct[0]:
            return None
        return np.zeros(v.shape, dtype=np.uint8), np.float16(0.0), bias
    a, c = f
    if a < c or (a == c and (distinct[0] >> 31) == 1):
        lo, hi, hi_pat = a, c, distinct[1]
    else:
        lo, hi, hi_pat = c, a, distinct[0]
    bits = (pats == hi_pat).astype(np.uint8)
    if symmetric:
        sc = np.float16(np.float32(-2.0) * lo)
        b = np.float32(-0.5) * np.float32(sc)
        one = np.float32(np.float32(sc) + b)
        if _bits32(b) != _bits32(lo) or _bits32(one) != hi_pat:
            return None
        return bits, sc, None
    bias = np.float16(lo)
    if _bits32(np.float32(bias)) != _bits32(lo):
        return None
    c0 = np.float16(np.float32(hi - lo))
    for k in SCALE_STEPS:
        sc = _f16_step(c0, k)
        if not np.isfinite(sc):
            continue
        if _bits32(np.float32(np.float32(sc) + np.float32(bias))) == hi_pat:
            return bits, sc, bias
    return None


def pack_from_dense(dense, symmetric: bool):
    """Repack a dense [N, K] tensor (bf16, f16 or f32) group by group.

    Returns (words [N, K/32] uint32, scales [N, G] fp16, biases [N, G] fp16 or
    None when symmetric, number of refused groups).  A refused group gets zero
    words, scale and bias.  bf16 and f16 values widen to fp32 exactly, so
    comparing fp32 bit patterns compares the input's bit patterns.
    """
    if isinstance(dense, torch.Tensor):
        d32 = dense.detach().to(torch.float32).numpy()
    else:
        d32 = np.asarray(dense, dtype=np.float32)
    N, K = d32.shape
    G = K // GROUP_SIZE
    bits = np.zeros((N, K), dtype=np.uint8)
    scales = np.zeros((N, G), dtype=np.float16)
    biases = None if symmetric else np.zeros((N, G), dtype=np.float16)
    bad = 0
    for n in range(N):
        for g in range(G):
            r = pack_group(d32[n, g * GROUP_SIZE:(g + 1) * GROUP_SIZE], symmetric)
            if r is None:
                bad += 1
                continue
            bits[n, g * GROUP_SIZE:(g + 1) * GROUP_SIZE] = r[0]
            scales[n, g] = r[1]
            if not symmetric:
                biases[n, g] = r[2]
    return pack(bits), scales, biases, bad


# ---------------------------------------------------------------------------
# Storage accounting (bytes per weight of the packed format)
# ---------------------------------------------------------------------------
def storage_bytes(N: int, K: int, symmetric: bool) -> dict:
    """Bytes held by one packed weight: bits, fp16 scales, fp16 biases."""
    G = K // GROUP_SIZE
    packed = N * K // 8
    s = N * G * 2
    b = 0 if symmetric else N * G * 2
    return {"packed": packed, "scales": s, "biases": b, "total": packed + s + b}


def tolerance_bound(x, wd_f32: np.ndarray, rel: float = 2e-2) -> np.ndarray:
    """Per-element matmul error bound rel * ||x_m|| * ||Wd_n|| / sqrt(K) [M, N]."""
    x64 = _x64(x)
    if x64.ndim == 1:
        x64 = x64[None, :]
    K = x64.shape[1]
    xn = np.linalg.norm(x64, axis=1)
    wn = np.linalg.norm(np.asarray(wd_f32, dtype=np.float64), axis=1)
    return rel * np.outer(xn, wn) / np.sqrt(K)
