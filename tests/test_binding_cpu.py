"""Host-only checks of the Python binding's argument validation.

The library takes raw device pointers, so a host tensor, a tensor on another
device or a short output buffer would make a kernel fault or write out of
bounds.  The binding must refuse such calls with a ValueError before it loads
the library or launches anything; these tests run without a GPU.
"""
import pytest
import torch

from bit_affine_quantized_g128_gb300 import q1


@pytest.fixture
def no_library(monkeypatch):
    """Any use of the library fails the test: validation must come first."""
    def _forbidden(*a, **k):
        raise AssertionError("the library was reached with invalid arguments")
    monkeypatch.setattr(q1, "lib", _forbidden)
    monkeypatch.setattr(q1, "load_library", _forbidden)


def _fake_weight(N=16, K=256):
    """A Q1Weight whose tensors live on the host (built around the constructor,
    which would refuse them), to drive the per-call checks."""
    W = object.__new__(q1.Q1Weight)
    W.words = torch.zeros((N, K // 32), dtype=torch.int32)
    W.scales = torch.ones((N, K // 128), dtype=torch.float16)
    W.biases = None
    W.N, W.K, W.group_size = N, K, 128
    return W


def test_weight_refuses_host_tensors(no_library):
    w = torch.zeros((16, 8), dtype=torch.int32)
    s = torch.ones((16, 2), dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        q1.Q1Weight(w, s, None, 256)


@pytest.mark.parametrize("call", [
    lambda W, x: q1.qmv(W, x[0]),
    lambda W, x: q1.qmm_narrow(W, x),
    lambda W, x: q1.qmm(W, x),
    lambda W, x: q1.ffn_fused(W, W, W, x),
    lambda W, x: q1.ffn_fused_noalloc(W, W, W, x),
    lambda W, x: q1.decode_chain([(W, W, W, W)], x),
])
def test_products_refuse_host_activations(no_library, call):
    W = _fake_weight()
    x = torch.zeros((2, W.K), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        call(W, x)


def test_elementwise_calls_refuse_host_tensors(no_library):
    with pytest.raises(ValueError, match="CUDA"):
        q1.pack(torch.zeros((4, 64), dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        q1.unpack(torch.zeros((4, 2), dtype=torch.int32), 64)
    with pytest.raises(ValueError, match="CUDA"):
        q1.pack_from_dense(torch.zeros((4, 128), dtype=torch.float32), symmetric=True)
    with pytest.raises(ValueError, match="CUDA"):
        q1.embed_gather(_fake_weight(), torch.zeros((3,), dtype=torch.int32))
    with pytest.raises(ValueError, match="at least one layer"):
        q1.decode_chain([], torch.zeros((1, 256), dtype=torch.bfloat16))


def test_output_buffer_must_match_what_the_call_writes(monkeypatch):
    # the device check is covered above; here only the shape/dtype/layout rules
    monkeypatch.setattr(q1, "_cuda", lambda t, name, device=None: t)
    good = torch.empty((4, 8), dtype=torch.bfloat16)
    assert q1._out(good, (4, 8), torch.bfloat16, None) is good
    # any shape with the right element count is accepted (a flat view of y)
    flat = torch.empty((32,), dtype=torch.bfloat16)
    assert q1._out(flat, (4, 8), torch.bfloat16, None) is flat
    with pytest.raises(ValueError):
        q1._out(torch.empty((4, 7), dtype=torch.bfloat16), (4, 8), torch.bfloat16, None)
    with pytest.raises(ValueError):
        q1._out(torch.empty((4, 8), dtype=torch.float16), (4, 8), torch.bfloat16, None)
    with pytest.raises(ValueError):
        q1._out(torch.empty((8, 4), dtype=torch.bfloat16).t(), (4, 8), torch.bfloat16, None)


def test_activation_dtype_and_shape_rules(no_library, monkeypatch):
    monkeypatch.setattr(q1, "_cuda", lambda t, name, device=None: t)
    W = _fake_weight()
    with pytest.raises(ValueError, match="bfloat16, float16 or float32"):
        q1.qmm_narrow(W, torch.zeros((2, W.K), dtype=torch.int32))
    with pytest.raises(ValueError, match="last dim"):
        q1.qmm_narrow(W, torch.zeros((2, W.K + 1), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match=r"\[N, K/32\]"):
        q1.unpack(torch.zeros((4, 3), dtype=torch.int32), 64)
    with pytest.raises(ValueError, match="uint8"):
        q1.pack(torch.zeros((4, 64), dtype=torch.int32))


def _pretend_cuda(monkeypatch, current):
    """Every tensor passes the is-CUDA test and `current` is the thread's CUDA
    device; tensors keep their real device, so a CPU tensor reads as a tensor
    on a device other than `current`."""
    monkeypatch.setattr(q1, "_is_cuda", lambda t: True)
    monkeypatch.setattr(q1, "_current_device", lambda: current)


@pytest.mark.parametrize("call", [
    lambda W, x: q1.qmv(W, x[0]),
    lambda W, x: q1.qmm_narrow(W, x),
    lambda W, x: q1.qmm(W, x),
    lambda W, x: q1.ffn_fused(W, W, W, x),
    lambda W, x: q1.ffn_fused_noalloc(W, W, W, x),
    lambda W, x: q1.decode_chain([(W, W, W, W)], x),
    lambda W, x: q1.dequantize(W),
    lambda W, x: q1.check_symmetric(W),
    lambda W, x: q1.embed_gather(W, torch.zeros((3,), dtype=torch.int32)),
])
def test_calls_refuse_tensors_off_the_current_device(no_library, monkeypatch, call):
    # the library launches on the current device: weights and activations on
    # another GPU must be refused before anything reaches it
    _pretend_cuda(monkeypatch, torch.device("cuda", 0))
    W = _fake_weight()
    x = torch.zeros((2, W.K), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="current CUDA device"):
        call(W, x)


@pytest.mark.parametrize("which", ["up", "down"])
@pytest.mark.parametrize("noalloc", [False, True])
def test_ffn_refuses_a_matrix_on_another_device(no_library, monkeypatch, which, noalloc):
    _pretend_cuda(monkeypatch, torch.device("cpu"))
    G, U, D = _fake_weight(), _fake_weight(), _fake_weight()
    # one matrix on another device (the meta device stands in for another GPU)
    odd = U if which == "up" else D
    odd.words = torch.zeros(odd.words.shape, dtype=torch.int32, device="meta")
    x = torch.zeros((2, G.K), dtype=torch.bfloat16)
    fn = q1.ffn_fused_noalloc if noalloc else q1.ffn_fused
    with pytest.raises(ValueError, match=f"{which} is on meta"):
        fn(G, U, D, x)


@pytest.mark.parametrize("which", ["attn", "gate", "up", "down"])
def test_decode_chain_refuses_a_layer_matrix_on_another_device(no_library, monkeypatch, which):
    _pretend_cuda(monkeypatch, torch.device("cpu"))
    layer = {n: _fake_weight() for n in ("attn", "gate", "up", "down")}
    layer[which].words = torch.zeros(layer[which].words.shape, dtype=torch.int32, device="meta")
    x = torch.zeros((1, 256), dtype=torch.bfloat16)
    ok = tuple(_fake_weight() for _ in range(4))
    with pytest.raises(ValueError, match=f"layer 1 {which} is on meta"):
        q1.decode_chain([ok, tuple(layer[n] for n in ("attn", "gate", "up", "down"))], x)
