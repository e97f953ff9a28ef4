"""Parity at the full workload sizes (27B-class shapes), in the launch
configurations the benchmark times: the GPU computes every output, the oracle
recomputes a seeded sample of output rows one by one (all tokens of those
rows), and pack/dequantize/gather stay bit-exact.
"""
import numpy as np
import pytest
import torch

from oracle import q1_oracle as O
from bit_affine_quantized_g128_gb300 import synth
from tests.tolerance import check_matmul

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda"
D_MODEL, D_FF, VOCAB = 5120, 17408, 152064


@pytest.fixture(scope="module")
def q1():
    from bit_affine_quantized_g128_gb300 import q1 as mod
    mod.load_library()
    return mod


def _rows(N, n, seed):
    r = np.random.default_rng(seed).choice(N, size=n, replace=False)
    return np.sort(np.concatenate([r, [0, N - 1]]))


def _check_rows(y, t, x, rows, what):
    yo = O.qmm(x, t.words, t.scales, t.biases, t.K, rows=rows)
    wd = O.dequantize_f32(t.words[rows], t.scales[rows], None if t.biases is None else t.biases[rows], t.K)
    check_matmul(y[:, rows], yo, x, wd, what)


@pytest.mark.parametrize("N,K,affine", [(D_FF, D_MODEL, False), (D_MODEL, D_FF, True),
                                        (D_MODEL, D_MODEL, False)])
def test_decode_qmv_full_shapes(q1, N, K, affine):
    t = synth.q1_tensor(N, K, seed=1001 + affine, affine=affine)
    x = synth.activations(1, K, seed=1006)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmv(W, x.to(DEV)).float().cpu().double().numpy()[None, :]
    _check_rows(y, t, x, _rows(N, 256, N + K), f"qmv {N}x{K}")


@pytest.mark.parametrize("M", [2, 5, 8])
@pytest.mark.parametrize("N,K,affine", [(D_FF, D_MODEL, True), (D_MODEL, D_FF, False)])
def test_narrow_full_shapes(q1, M, N, K, affine):
    t = synth.q1_tensor(N, K, seed=1002 + affine, affine=affine)
    x = synth.activations(M, K, seed=1007 + M)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV)).float().cpu().double().numpy()
    _check_rows(y, t, x, _rows(N, 128, M), f"narrow M={M} {N}x{K}")


@pytest.mark.parametrize("M", [9, 128, 1000, 2048])
@pytest.mark.parametrize("N,K,affine", [(D_FF, D_MODEL, False), (D_MODEL, D_FF, True)])
def test_prefill_full_shapes(q1, M, N, K, affine):
    t = synth.q1_tensor(N, K, seed=1004 + affine, affine=affine)
    x = synth.activations(M, K, seed=1008)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV)).float().cpu().double().numpy()
    _check_rows(y, t, x, _rows(N, 48, M), f"prefill M={M} {N}x{K}")


@pytest.mark.parametrize("M", [1000, 1024, 2048])
@pytest.mark.parametrize("affine", [False, True])
def test_prefill_attention_shape(q1, M, affine):
    # the 5120 x 5120 projection at prefill sizes, in the plan each call picks
    # (a ragged last token tile at M = 1000)
    N = K = D_MODEL
    t = synth.q1_tensor(N, K, seed=1011 + affine, affine=affine)
    x = synth.activations(M, K, seed=1012)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV)).float().cpu().double().numpy()
    _check_rows(y, t, x, _rows(N, 48, M + 7), f"prefill M={M} {N}x{K}")


@pytest.mark.parametrize("M", [8192, 16384])
def test_prefill_many_token_tiles(q1, M):
    # 32 to 64 token tiles per weight-row tile: long runs of tiles per pair,
    # in the plan each call picks; sampled rows, every token
    N, K = 768, 1024
    t = synth.q1_tensor(N, K, seed=1015, affine=True)
    x = synth.activations(M, K, seed=1016)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV)).float().cpu().double().numpy()
    _check_rows(y, t, x, _rows(N, 32, M), f"prefill M={M} {N}x{K}")


def test_prefill_attention_shape_stream_fp32_out(q1):
    # the stream schedule forced, fp32 activations and outputs (its shared
    # tiles' outputs are written by the share that completes them)
    N = K = D_MODEL
    M = 1000
    t = synth.q1_tensor(N, K, seed=1013, affine=True)
    x = synth.activations(M, K, seed=1014)
    W = q1.Q1Weight.from_host(t)
    q1.set_prefill_plan(256, 0)
    try:
        ws = q1.qmm_workspace(M, N, K, DEV)
        y = q1.qmm(W, x.float().to(DEV), workspace=ws)
    finally:
        q1.set_prefill_plan(0, 0)
    assert y.dtype == torch.float32
    _check_rows(y.cpu().double().numpy(), t, x, _rows(N, 48, 17), "prefill stream fp32 M=1000")


def test_dequantize_full_shape_bit_exact(q1):
    t = synth.q1_tensor(D_FF, D_MODEL, seed=1001, affine=True)
    W = q1.Q1Weight.from_host(t)
    got = q1.dequantize(W, torch.bfloat16).cpu().view(torch.int16).numpy()
    want = O.dequantize(t.words, t.scales, t.biases, D_MODEL, "bf16").view(torch.int16).numpy()
    np.testing.assert_array_equal(got, want)
    # pack / unpack round trip at this size
    bits = q1.unpack(W.words, D_MODEL)
    assert torch.equal(q1.pack(bits), W.words)


def test_pack_from_dense_full_shape(q1):
    """A 27B-class projection dequantized by the library, then repacked: fp32
    dense gives back the very words and scales; bf16 dense (the halves of the
    scales rounded to bf16) stays exactly representable and round-trips."""
    t = synth.q1_tensor(D_FF, D_MODEL, seed=1011, affine=False)
    W = q1.Q1Weight.from_host(t)
    d32 = q1.dequantize(W, torch.float32)
    W2, bad = q1.pack_from_dense(d32, symmetric=True)
    assert int(bad.item()) == 0
    assert torch.equal(W2.words, W.words) and torch.equal(W2.scales.view(torch.int16), W.scales.view(torch.int16))
    d16 = q1.dequantize(W, torch.bfloat16)
    W3, bad3 = q1.pack_from_dense(d16, symmetric=True)
    assert int(bad3.item()) == 0 and torch.equal(W3.words, W.words)
    assert torch.equal(q1.dequantize(W3, torch.bfloat16).view(torch.int16), d16.view(torch.int16))
    rows = _rows(D_FF, 6, 1012)
    wo, so, _, bado = O.pack_from_dense(d16[torch.from_numpy(rows).to(DEV)].cpu(), symmetric=True)
    assert bado == 0
    np.testing.assert_array_equal(W3.words[torch.from_numpy(rows).to(DEV)].cpu().numpy().view(np.uint32), wo)
    np.testing.assert_array_equal(W3.scales[torch.from_numpy(rows).to(DEV)].cpu().numpy().view(np.uint16),
                                  so.view(np.uint16))
    # affine in fp32: the same words, and the repacked tensor dequantizes to the same bits
    ta = synth.q1_tensor(D_MODEL, D_FF, seed=1013, affine=True)
    Wa = q1.Q1Weight.from_host(ta)
    da = q1.dequantize(Wa, torch.float32)
    Wb, bada = q1.pack_from_dense(da, symmetric=False)
    assert int(bada.item()) == 0 and torch.equal(Wb.words, Wa.words)
    assert torch.equal(q1.dequantize(Wb, torch.float32).view(torch.int32), da.view(torch.int32))


def test_embedding_gather_and_tied_head_full_vocab(q1):
    t = synth.q1_tensor(VOCAB, D_MODEL, seed=1003, affine=False)
    E = q1.Q1Weight.from_host(t)
    ids = synth.token_ids(64, VOCAB, seed=1003)
    out, bad = q1.embed_gather(E, torch.from_numpy(ids).to(DEV), torch.bfloat16)
    want, nbad = O.embed_gather(ids, t.words, t.scales, None, D_MODEL, "bf16")
    assert int(bad.item()) == nbad == 0
    np.testing.assert_array_equal(out.cpu().view(torch.int16).numpy(), want.view(torch.int16).numpy())
    # tied head: logits = h . E^T over the whole vocabulary, M = 1
    h = synth.activations(1, D_MODEL, seed=1009)
    logits = q1.qmv(E, h.to(DEV)).float().cpu().double().numpy()[None, :]
    _check_rows(logits, t, h, _rows(VOCAB, 256, 7), "tied head")


@pytest.mark.parametrize("M", [1, 4, 8])
def test_ffn_full_shape(q1, M):
    gate = synth.q1_tensor(D_FF, D_MODEL, seed=2001, affine=False)
    up = synth.q1_tensor(D_FF, D_MODEL, seed=2002, affine=False)
    down = synth.q1_tensor(D_MODEL, D_FF, seed=2003, affine=False)
    x = synth.activations(M, D_MODEL, seed=2004)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    ws = q1.ffn_workspace(M, D_MODEL, D_FF, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws).float().cpu().double().numpy()
    rows = _rows(D_MODEL, 128, M)
    yo, ho = O.ffn(x, (gate.words, gate.scales, None, D_MODEL), (up.words, up.scales, None, D_MODEL),
                   (down.words, down.scales, None, D_FF), rows=rows)
    h = q1.ffn_h(ws, M, D_FF).float().cpu().double().numpy()
    assert np.linalg.norm(h - ho) / np.linalg.norm(ho) < 5e-3
    check_matmul(y[:, rows], yo, ho, O.dequantize_f32(down.words[rows], down.scales[rows], None, D_FF),
                 f"ffn M={M}")


def test_ffn_full_shape_all_affine(q1):
    # the 27B-class FFN with stored biases on all three matrices, M = 4; the
    # down product's output includes its own bf16 rounding in the bar
    # (tests/tolerance.py: outputs dominated by group means times sums of h)
    M = 4
    gate = synth.q1_tensor(D_FF, D_MODEL, seed=2011, affine=True)
    up = synth.q1_tensor(D_FF, D_MODEL, seed=2012, affine=True)
    down = synth.q1_tensor(D_MODEL, D_FF, seed=2013, affine=True)
    x = synth.activations(M, D_MODEL, seed=2014)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    ws = q1.ffn_workspace(M, D_MODEL, D_FF, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws).float().cpu().double().numpy()
    rows = _rows(D_MODEL, 128, 2015)
    yo, ho = O.ffn(x, (gate.words, gate.scales, gate.biases, D_MODEL), (up.words, up.scales, up.biases, D_MODEL),
                   (down.words, down.scales, down.biases, D_FF), rows=rows)
    h = q1.ffn_h(ws, M, D_FF).float().cpu().double().numpy()
    assert np.linalg.norm(h - ho) / np.linalg.norm(ho) < 5e-3
    check_matmul(y[:, rows], yo, ho, O.dequantize_f32(down.words[rows], down.scales[rows], down.biases[rows], D_FF),
                 "affine ffn full shape", rounded_to="bf16")


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("M", [1, 8])
@pytest.mark.parametrize("N,K,affine", [(D_FF, D_MODEL, False), (D_MODEL, D_FF, True)])
def test_small_group_narrow_full_shapes(q1, group, M, N, K, affine):
    # the 27B-class shapes with metadata per 32 or 64 weights, on the narrow
    # kernel (the K-split down shape included)
    t = synth.q1_tensor(N, K, seed=1021 + group + affine, affine=affine, group=group)
    x = synth.activations(M, K, seed=1022 + M)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm_narrow(W, x.to(DEV)).float().cpu().double().numpy()
    _check_rows(y, t, x, _rows(N, 96, group + M), f"group {group} narrow M={M} {N}x{K}")
