"""Thin Python binding of libq1 (include/q1.h) over ctypes.

Argument marshalling only: every step of every call runs in the library's CUDA
kernels.  torch tensors supply device memory and the current CUDA stream.
There is no fallback: if the library is missing or the device is not a
Blackwell GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libq1.so")

Q1_BF16, Q1_F16, Q1_F32 = 0, 1, 2
_DT = {torch.bfloat16: Q1_BF16, torch.float16: Q1_F16, torch.float32: Q1_F32}

# every symbol include/q1.h declares
EXPORTED = [
    "q1_pack", "q1_unpack", "q1_dequantize", "q1_qmv", "q1_qmm_workspace_size",
    "q1_qmm_narrow", "q1_qmm", "q1_set_qmm_max_rows", "q1_get_qmm_max_rows", "q1_set_prefill_plan",
    "q1_embed_gather", "q1_ffn_workspace_size", "q1_ffn_fused", "q1_check_symmetric",
    "q1_device_errors", "q1_status_string", "q1_ffn_fused_noalloc",
    "q1_set_wait_limit_ns", "q1_set_stalled_producers",
    "q1_decode_chain_workspace_size", "q1_decode_chain", "q1_pack_from_dense",
]


class Q1Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class _CWeight(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("biases", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("group_size", ctypes.c_int32),
                ("meta_dtype", ctypes.c_int32)]


# q1_meta_dtype of the scales/biases tensors
_META = {torch.float16: 0, torch.bfloat16: 1}


class _CLayer(ctypes.Structure):
    _fields_ = [("attn", _CWeight), ("gate", _CWeight), ("up", _CWeight), ("down", _CWeight)]


_lib = None

# K of the narrow kernel (q1_qmv / q1_qmm_narrow); q1_qmm runs larger K on the prefill path
NARROW_MAX_K = 40960
# bytes of the library's fixed array that holds h for q1_ffn_fused_noalloc
FFN_NOALLOC_BYTES = 512 * 1024


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libq1.so (after torch, so that both share one CUDA runtime)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libq1.so not built ({path}); run __graft_entry__.build() or "
                           "python -m bit_affine_quantized_g128_gb300.build")
    lib = ctypes.CDLL(path)
    P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
    W = ctypes.POINTER(_CWeight)
    sig = {
        "q1_pack": ([P, I64, I64, P, P], I32),
        "q1_unpack": ([P, I64, I64, P, P], I32),
        "q1_dequantize": ([W, I32, P, P], I32),
        "q1_qmv": ([W, P, I32, P, P], I32),
        "q1_qmm_narrow": ([W, P, I64, I32, P, P], I32),
        "q1_qmm_workspace_size": ([I64, I64, I64], SZ),
        "q1_qmm": ([W, P, I64, I32, P, P, SZ, P], I32),
        "q1_set_qmm_max_rows": ([ctypes.c_int], None),
        "q1_get_qmm_max_rows": ([], ctypes.c_int),
        "q1_set_prefill_plan": ([ctypes.c_int, ctypes.c_int], None),
        "q1_set_wait_limit_ns": ([ctypes.c_uint64], I32),
        "q1_set_stalled_producers": ([ctypes.c_int], I32),
        "q1_embed_gather": ([W, P, I64, I32, P, P, P], I32),
        "q1_ffn_workspace_size": ([I64, I64, I64], SZ),
        "q1_ffn_fused": ([W, W, W, P, I64, I32, P, P, SZ, P], I32),
        "q1_ffn_fused_noalloc": ([W, W, W, P, I64, I32, P, P], I32),
        "q1_check_symmetric": ([W, P, P], I32),
        "q1_decode_chain_workspace_size": ([I64, I64, I64], SZ),
        "q1_pack_from_dense": ([P, I32, I64, I64, P, P, P, P, P], I32),
        "q1_decode_chain": ([ctypes.POINTER(_CLayer), I32, P, I64, I32, P, P, SZ, P], I32),
        "q1_device_errors": ([ctypes.POINTER(ctypes.c_uint), P], I32),
        "q1_status_string": ([I32], ctypes.c_char_p),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def lib() -> ctypes.CDLL:
    return load_library()


def _check(fn: str, status: int):
    if status != 0:
        raise Q1Error(fn, status, lib().q1_status_string(status).decode())


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


# The library takes raw device pointers and cannot tell a host pointer, a
# tensor on another GPU or a short output buffer from a good one: the kernels
# would fault or write past the end.  It also launches on the CUDA device that
# is current for the calling thread, with that device's current stream, so a
# tensor on any other device would be handed to kernels of the wrong GPU.
# These checks turn such calls into a ValueError before anything is launched.
def _is_cuda(t: torch.Tensor) -> bool:
    return t.is_cuda


def _current_device() -> torch.device:
    return torch.device("cuda", torch.cuda.current_device())


def _cuda(t, name: str, device=None, current: bool = True) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not _is_cuda(t):
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if current:
        cur = _current_device()
        if t.device != cur:
            raise ValueError(f"{name} is on {t.device} but the current CUDA device is {cur}: the library "
                             f"launches on the current device (select it with torch.cuda.device)")
    return t


def _out(out: Optional[torch.Tensor], shape, dtype, device, name: str = "out") -> torch.Tensor:
    """`out` checked against what the call writes (or a new tensor of that shape)."""
    if out is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _cuda(out, name, device)
    n = 1
    for d in shape:
        n *= int(d)
    if out.dtype != dtype or not out.is_contiguous() or out.numel() != n:
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of {n} elements "
                         f"(got {out.dtype}, {tuple(out.shape)}, contiguous={out.is_contiguous()})")
    return out


def _x_dtype(x: torch.Tensor, name: str = "x") -> int:
    if x.dtype not in _DT:
        raise ValueError(f"{name} must be bfloat16, float16 or float32 (got {x.dtype})")
    return _DT[x.dtype]


class Q1Weight:
    """A packed Q1 weight on the GPU: words uint32 [N, K/32] (held as int32),
    scales [N, K/group_size] and biases of the same shape or None
    (symmetric), the metadata either fp16 or bf16 (both tensors the same
    dtype); all on one CUDA device."""

    def __init__(self, words: torch.Tensor, scales: torch.Tensor,
                 biases: Optional[torch.Tensor], K: int):
        _cuda(words, "Q1Weight words", current=False)
        _cuda(scales, "Q1Weight scales", words.device, current=False)
        if biases is not None:
            _cuda(biases, "Q1Weight biases", words.device, current=False)
        if words.dtype not in (torch.int32, torch.uint32):
            raise ValueError(f"Q1Weight words must be int32 or uint32 (the packed words), got {words.dtype}")
        self.words = words.contiguous()
        self.scales = scales.contiguous()
        self.biases = None if biases is None else biases.contiguous()
        if self.scales.dtype not in _META or (self.biases is not None and self.biases.dtype != self.scales.dtype):
            raise ValueError("Q1Weight: scales and biases must both be float16 or both bfloat16")
        self.N = int(words.shape[0])
        self.K = int(K)
        # weights per scale along K, from the metadata's shape [N, K / group_size]
        self.group_size = self.K // max(int(self.scales.shape[-1]), 1)
        self._c = _CWeight(self.words.data_ptr(), self.scales.data_ptr(),
                           _ptr(self.biases), self.N, self.K, self.group_size, _META[self.scales.dtype])

    @property
    def symmetric(self) -> bool:
        return self.biases is None

    @staticmethod
    def from_host(t, device="cuda") -> "Q1Weight":
        """From a host bundle with numpy words/scales/biases (synth.Q1Tensor)."""
        w = torch.from_numpy(t.words.view("<i4").copy()).to(device)
        s = torch.from_numpy(t.scales.copy()).to(device)
        b = None if t.biases is None else torch.from_numpy(t.biases.copy()).to(device)
        return Q1Weight(w, s, b, t.K)

    def cref(self):
        return ctypes.byref(self._c)


def _flat(x: torch.Tensor, K: int) -> torch.Tensor:
    if x.shape[-1] != K:
        raise ValueError(f"last dim {x.shape[-1]} != K {K}")
    return x.reshape(-1, K).contiguous()


def pack(bits: torch.Tensor) -> torch.Tensor:
    """bits uint8 [N, K] -> words int32 [N, K/32] (LSB first)."""
    _cuda(bits, "bits")
    if bits.dtype != torch.uint8 or bits.dim() != 2:
        raise ValueError(f"bits must be a 2-D uint8 tensor (got {bits.dtype}, {tuple(bits.shape)})")
    bits = bits.contiguous()
    N, K = bits.shape
    w = torch.empty((N, K // 32), dtype=torch.int32, device=bits.device)
    _check("q1_pack", lib().q1_pack(bits.data_ptr(), N, K, w.data_ptr(), _stream()))
    return w


def unpack(words: torch.Tensor, K: int) -> torch.Tensor:
    """words int32 [N, K/32] -> bits uint8 [N, K]."""
    _cuda(words, "words")
    if words.dim() != 2 or words.shape[1] * 32 != K:
        raise ValueError(f"words must be [N, K/32] for K = {K} (got {tuple(words.shape)})")
    words = words.contiguous()
    N = words.shape[0]
    out = torch.empty((N, K), dtype=torch.uint8, device=words.device)
    _check("q1_unpack", lib().q1_unpack(words.data_ptr(), N, K, out.data_ptr(), _stream()))
    return out


def dequantize(W: Q1Weight, dtype=torch.bfloat16) -> torch.Tensor:
    _cuda(W.words, "weight")
    if dtype not in _DT:
        raise ValueError(f"dtype must be bfloat16, float16 or float32 (got {dtype})")
    out = torch.empty((W.N, W.K), dtype=dtype, device=W.words.device)
    _check("q1_dequantize", lib().q1_dequantize(W.cref(), _DT[dtype], out.data_ptr(), _stream()))
    return out


def qmv(W: Q1Weight, x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """x [K] -> y [N] (M = 1 decode)."""
    _cuda(x, "x", W.words.device)
    xdt = _x_dtype(x)
    x = x.reshape(W.K).contiguous()
    y = _out(out, (W.N,), x.dtype, x.device)
    _check("q1_qmv", lib().q1_qmv(W.cref(), x.data_ptr(), xdt, y.data_ptr(), _stream()))
    return y


def qmm_workspace(M: int, N: int, K: int, device) -> torch.Tensor:
    """A byte buffer of the size q1_qmm needs for M x N x K (at least 256 B)."""
    n = lib().q1_qmm_workspace_size(M, N, K)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def qmm_narrow(W: Q1Weight, x: torch.Tensor, out=None) -> torch.Tensor:
    """x [..., K] with prod(leading dims) <= 8 -> y [..., N]; weights stay packed."""
    _cuda(x, "x", W.words.device)
    xdt = _x_dtype(x)
    lead = x.shape[:-1]
    x2 = _flat(x, W.K)
    M = x2.shape[0]
    y = _out(out, (M, W.N), x.dtype, x.device)
    _check("q1_qmm_narrow", lib().q1_qmm_narrow(W.cref(), x2.data_ptr(), M, xdt,
                                                y.data_ptr(), _stream()))
    return y.reshape(*lead, W.N)


def qmm(W: Q1Weight, x: torch.Tensor, workspace: Optional[torch.Tensor] = None,
        out=None) -> torch.Tensor:
    """x [..., K] -> y [..., N]; narrow path up to the row threshold, tcgen05
    beyond (which needs a workspace; one is allocated when none is given)."""
    _cuda(x, "x", W.words.device)
    xdt = _x_dtype(x)
    lead = x.shape[:-1]
    x2 = _flat(x, W.K)
    M = x2.shape[0]
    y = _out(out, (M, W.N), x.dtype, x.device)
    ws = workspace
    rows = get_qmm_max_rows()
    narrow = W.K <= NARROW_MAX_K and (M <= rows or (rows == 8 and M <= 16))
    if ws is None and not narrow:
        ws = qmm_workspace(M, W.N, W.K, x.device)
    if ws is not None:
        _cuda(ws, "workspace", x.device)
    wp, wn = (ws.data_ptr(), ws.numel() * ws.element_size()) if ws is not None else (None, 0)
    _check("q1_qmm", lib().q1_qmm(W.cref(), x2.data_ptr(), M, xdt, y.data_ptr(), wp, wn,
                                  _stream()))
    return y.reshape(*lead, W.N)


def set_qmm_max_rows(rows: int):
    lib().q1_set_qmm_max_rows(int(rows))


def set_prefill_plan(token_tile: int = 0, split: int = 0):
    """Fixed prefill tiling: token_tile tokens x 256 weight rows per tile;
    split 1 = whole tiles per CTA pair, 2..4 = pairs of a cluster per tile,
    0 = equal runs of work per pair (tiles shared through the workspace);
    (0, 0) restores the automatic choice."""
    lib().q1_set_prefill_plan(int(token_tile), int(split))


def get_qmm_max_rows() -> int:
    return int(lib().q1_get_qmm_max_rows())


def embed_gather(E: Q1Weight, ids: torch.Tensor, dtype=torch.bfloat16):
    """ids int32 [T] (device) -> (rows [T, K], out-of-range count int32 [1] on device)."""
    _cuda(ids, "ids", E.words.device)
    if dtype not in _DT:
        raise ValueError(f"dtype must be bfloat16, float16 or float32 (got {dtype})")
    ids = ids.to(torch.int32).contiguous()
    T = ids.numel()
    out = torch.empty((T, E.K), dtype=dtype, device=E.words.device)
    bad = torch.zeros((1,), dtype=torch.int32, device=E.words.device)
    _check("q1_embed_gather", lib().q1_embed_gather(E.cref(), ids.data_ptr(), T, _DT[dtype],
                                                    out.data_ptr(), bad.data_ptr(), _stream()))
    return out, bad


def _ffn_devices(gate: Q1Weight, up: Q1Weight, down: Q1Weight, x: torch.Tensor):
    """x and all three matrices on one device, the current one."""
    _cuda(x, "x", gate.words.device)
    _cuda(up.words, "up", gate.words.device)
    _cuda(down.words, "down", gate.words.device)


def ffn_workspace(M: int, D: int, F: int, device) -> torch.Tensor:
    """A byte buffer of the size q1_ffn_fused needs (at least 256 B)."""
    n = lib().q1_ffn_workspace_size(M, D, F)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def ffn_fused(gate: Q1Weight, up: Q1Weight, down: Q1Weight, x: torch.Tensor,
              workspace=None, out=None) -> torch.Tensor:
    """y = down . (SiLU(gate . x) * (up . x)); x [..., D] -> y [..., D]."""
    _ffn_devices(gate, up, down, x)
    xdt = _x_dtype(x)
    lead = x.shape[:-1]
    x2 = _flat(x, gate.K)
    M = x2.shape[0]
    y = _out(out, (M, down.N), x.dtype, x.device)
    ws = workspace if workspace is not None else ffn_workspace(M, gate.K, gate.N, x.device)
    _cuda(ws, "workspace", x.device)
    _check("q1_ffn_fused", lib().q1_ffn_fused(gate.cref(), up.cref(), down.cref(), x2.data_ptr(), M,
                                              xdt, y.data_ptr(), ws.data_ptr(),
                                              ws.numel() * ws.element_size(), _stream()))
    return y.reshape(*lead, down.N)


def ffn_fused_noalloc(gate: Q1Weight, up: Q1Weight, down: Q1Weight, x: torch.Tensor,
                      out=None) -> torch.Tensor:
    """q1_ffn_fused with h in the library's fixed device array (no workspace,
    no allocation in the call; `out` may be preallocated too)."""
    _ffn_devices(gate, up, down, x)
    xdt = _x_dtype(x)
    lead = x.shape[:-1]
    x2 = _flat(x, gate.K)
    M = x2.shape[0]
    y = _out(out, (M, down.N), x.dtype, x.device)
    _check("q1_ffn_fused_noalloc", lib().q1_ffn_fused_noalloc(gate.cref(), up.cref(), down.cref(),
                                                              x2.data_ptr(), M, xdt,
                                                              y.data_ptr(), _stream()))
    return y.reshape(*lead, down.N)


def ffn_h(ws: torch.Tensor, M: int, F: int) -> torch.Tensor:
    """The bf16 intermediate h [M, F] that the last q1_ffn_fused left in `ws`."""
    return ws[: M * F * 2].view(torch.bfloat16).reshape(M, F)


def pack_from_dense(dense: torch.Tensor, symmetric: bool, bad: Optional[torch.Tensor] = None,
                    out: Optional[Q1Weight] = None):
    """q1_pack_from_dense: the exact Q1 form of a dense [N, K] bf16/f16/f32
    tensor.  Returns (Q1Weight, bad), bad a device int32 [1] that counts the
    refused groups (added to `bad` when given).  `out` (a Q1Weight of the same
    shape, with biases unless symmetric) receives the result in place."""
    _cuda(dense, "dense")
    ddt = _x_dtype(dense, "dense")
    if dense.dim() != 2:
        raise ValueError(f"dense must be 2-D [N, K] (got {tuple(dense.shape)})")
    d = dense.contiguous()
    N, K = int(d.shape[0]), int(d.shape[1])
    dev = d.device
    if out is None:
        w = torch.empty((N, K // 32), dtype=torch.int32, device=dev)
        s = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
        b = None if symmetric else torch.empty((N, K // 128), dtype=torch.float16, device=dev)
        out = Q1Weight(w, s, b, K)
    elif out.N != N or out.K != K or (out.biases is None) != symmetric:
        raise ValueError("pack_from_dense: `out` does not match the dense shape or mode")
    if bad is None:
        bad = torch.zeros((1,), dtype=torch.int32, device=dev)
    elif bad.dtype != torch.int32 or bad.numel() < 1:
        raise ValueError("bad must be an int32 tensor of at least one element")
    _cuda(bad, "bad", dev)
    _cuda(out.words, "out words", dev)
    _check("q1_pack_from_dense", lib().q1_pack_from_dense(d.data_ptr(), ddt, N, K, out.words.data_ptr(),
                                                          out.scales.data_ptr(), _ptr(out.biases),
                                                          bad.data_ptr(), _stream()))
    return out, bad


def decode_chain_workspace(M: int, D: int, F_max: int, device) -> torch.Tensor:
    """A byte buffer of the size q1_decode_chain needs (at least 256 B)."""
    n = lib().q1_decode_chain_workspace_size(M, D, F_max)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def decode_chain(layers, x: torch.Tensor, workspace=None, out=None) -> torch.Tensor:
    """q1_decode_chain: layers is a sequence of (attn, gate, up, down) Q1Weights;
    per layer a = attn . h, then h = down . (SiLU(gate . a) * (up . a))."""
    layers = list(layers)
    if not layers:
        raise ValueError("decode_chain needs at least one layer")
    _cuda(x, "x", layers[0][0].words.device)
    xdt = _x_dtype(x)
    for li, lw in enumerate(layers):
        for name, W in zip(("attn", "gate", "up", "down"), lw):
            _cuda(W.words, f"layer {li} {name}", x.device)
    lead = x.shape[:-1]
    D = layers[0][0].N
    x2 = _flat(x, D)
    M = x2.shape[0]
    arr = (_CLayer * len(layers))(*[_CLayer(a._c, g._c, u._c, d._c) for (a, g, u, d) in layers])
    y = _out(out, (M, D), x.dtype, x.device)
    if workspace is None:
        workspace = decode_chain_workspace(M, D, max(g.N for (_, g, _, _) in layers), x.device)
    _cuda(workspace, "workspace", x.device)
    _check("q1_decode_chain", lib().q1_decode_chain(arr, len(layers), x2.data_ptr(), M, xdt,
                                                    y.data_ptr(), workspace.data_ptr(),
                                                    workspace.numel() * workspace.element_size(),
                                                    _stream()))
    return y.reshape(*lead, D)


def check_symmetric(W: Q1Weight) -> torch.Tensor:
    """Device int32 [1]: 1 iff every stored bias is exactly -scale/2."""
    _cuda(W.words, "weight")
    r = torch.empty((1,), dtype=torch.int32, device=W.words.device)
    _check("q1_check_symmetric", lib().q1_check_symmetric(W.cref(), r.data_ptr(), _stream()))
    return r


def set_wait_limit_ns(ns: int = 0):
    """Limit of the kernels' bounded waits in ns (0 restores 2 s); for tests."""
    _check("q1_set_wait_limit_ns", lib().q1_set_wait_limit_ns(int(ns)))


def set_stalled_producers(stall: bool):
    """Producers of later launches issue no copies, so that every wait for
    their data runs out (results undefined); for tests of the timeout path."""
    _check("q1_set_stalled_producers", lib().q1_set_stalled_producers(1 if stall else 0))


def device_errors() -> int:
    """Synchronizes the current stream; returns and clears the device error flags."""
    v = ctypes.c_uint(0)
    st = lib().q1_device_errors(ctypes.byref(v), _stream())
    if st not in (0, 8):
        _check("q1_device_errors", st)
    return int(v.value)
