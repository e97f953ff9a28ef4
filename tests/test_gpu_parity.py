"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: pack, unpack, dequantize (bf16/f16/f32), embedding gather.
Matmuls: the per-element and Frobenius bars of tests/tolerance.py.
Inputs are the seeded synthetic workloads (bit_affine_quantized_g128_gb300/synth.py).
"""
import numpy as np
import pytest
import torch

from oracle import q1_oracle as O
from bit_affine_quantized_g128_gb300 import synth
from tests.tolerance import check_chain, check_matmul

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def q1():
    from bit_affine_quantized_g128_gb300 import q1 as mod
    mod.load_library()
    return mod


def _u16(t):
    return t.view(torch.int16).cpu().numpy().astype(np.uint16)


# ------------------------------------------------------------------ pack / unpack
@pytest.mark.parametrize("N,K", [(1, 32), (7, 96), (33, 1024), (1024, 1024)])
def test_pack_unpack_bit_exact(q1, N, K):
    bits = synth.bits(N, K, seed=1000 + N)
    w = q1.pack(torch.from_numpy(bits).to(DEV))
    want = O.pack(bits)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), want)
    words = synth.weight_words(N, K, seed=2000 + N)
    b = q1.unpack(torch.from_numpy(words.view(np.int32)).to(DEV), K)
    np.testing.assert_array_equal(b.cpu().numpy(), O.unpack(words, K))
    # round trip on the device
    np.testing.assert_array_equal(q1.pack(b).cpu().numpy().view(np.uint32), words)


def test_pack_ignores_high_bits_of_bytes(q1):
    bits = synth.bits(4, 64, seed=3)
    noisy = bits | (np.random.default_rng(4).integers(0, 128, bits.shape, dtype=np.uint8) << 1)
    w = q1.pack(torch.from_numpy(noisy).to(DEV))
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), O.pack(bits))


# ------------------------------------------------------------------ dequantize
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("dtype,name", [(torch.bfloat16, "bf16"), (torch.float16, "f16"),
                                        (torch.float32, "f32")])
@pytest.mark.parametrize("N,K", [(1024, 1024), (37, 384)])
def test_dequantize_bit_exact(q1, affine, dtype, name, N, K):
    t = synth.q1_tensor(N, K, seed=1000 + affine, affine=affine)
    W = q1.Q1Weight.from_host(t)
    got = q1.dequantize(W, dtype).cpu()
    want = O.dequantize(t.words, t.scales, t.biases, K, name)
    if dtype == torch.float32:
        np.testing.assert_array_equal(got.view(torch.int32).numpy(), want.view(torch.int32).numpy())
    else:
        np.testing.assert_array_equal(_u16(got), _u16(want))


def test_dequantize_edge_values(q1):
    # tiny, zero and negative-zero metadata (the golden dequant fixture's cases)
    K = 128
    s = np.array([[0x0001], [0x3C01], [0x3555], [0x3555], [0x0000]], dtype=np.uint16).view(np.float16)
    b = np.array([[0x8000], [0x0001], [0x0000], [0x8000], [0x8000]], dtype=np.uint16).view(np.float16)
    words = np.tile(np.array([0x0000FFFF, 0xFFFF0000, 0x12345678, 0x80000001], dtype=np.uint32), (5, 1))
    for bias in (None, b):
        t = synth.Q1Tensor(words, s, bias, K)
        W = q1.Q1Weight.from_host(t)
        for dt, name in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
            np.testing.assert_array_equal(_u16(q1.dequantize(W, dt).cpu()),
                                          _u16(O.dequantize(words, s, bias, K, name)))
        np.testing.assert_array_equal(q1.dequantize(W, torch.float32).cpu().view(torch.int32).numpy(),
                                      O.dequantize(words, s, bias, K, "f32").view(torch.int32).numpy())


# ------------------------------------------------------------------ narrow matmul
def _case(N, K, M, affine, seed):
    t = synth.q1_tensor(N, K, seed=seed, affine=affine)
    x = synth.activations(M, K, seed=seed + 5)
    return t, x


@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("M", list(range(1, 9)))
def test_qmm_narrow_tiny(q1, affine, M):
    # 1024 x 1024 (the tiny oracle check), every window size 1..8
    t, x = _case(1024, 1024, M, affine, seed=1000 + affine)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm_narrow(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, 1024), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, 1024), f"narrow M={M}")


@pytest.mark.parametrize("N,K", [(1, 128), (17, 384), (130, 2176), (1000, 640), (333, 17408 // 4)])
@pytest.mark.parametrize("affine", [False, True])
def test_qmm_narrow_ragged(q1, N, K, affine):
    for M in (1, 3, 8):
        t, x = _case(N, K, M, affine, seed=N + K + M)
        W = q1.Q1Weight.from_host(t)
        y = q1.qmm_narrow(W, x.to(DEV))
        check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                     O.dequantize_f32(t.words, t.scales, t.biases, K), f"narrow N={N} K={K} M={M}")


def test_qmv_and_leading_dims(q1):
    K = N = 1024
    t, x = _case(N, K, 8, True, seed=1001)
    W = q1.Q1Weight.from_host(t)
    yo = O.qmm(x, t.words, t.scales, t.biases, K)
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    y1 = q1.qmv(W, x[0].to(DEV))
    check_matmul(y1[None], yo[:1], x[:1], wd, "qmv")
    # [2, 4, K] leading dimensions flatten to M = 8
    y3 = q1.qmm(W, x.reshape(2, 4, K).to(DEV))
    assert y3.shape == (2, 4, N)
    check_matmul(y3.reshape(8, N), yo, x, wd, "[2,4,K]")


@pytest.mark.parametrize("N,K", [(333, 4096), (1000, 5120)])
@pytest.mark.parametrize("affine", [False, True])
def test_qmm_narrow_many_spans(q1, N, K, affine):
    # K of 8 and 10 spans of 512 k: every consumer warp owns a span and, with
    # 10 spans, one group of the last two; ragged row tiles
    for M in (1, 3, 8):
        t, x = _case(N, K, M, affine, seed=N + K + 7 * M)
        W = q1.Q1Weight.from_host(t)
        y = q1.qmm_narrow(W, x.to(DEV))
        check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                     O.dequantize_f32(t.words, t.scales, t.biases, K), f"narrow N={N} K={K} M={M}")


@pytest.mark.parametrize("affine", [False, True])
def test_k_beyond_narrow_kernel(q1, affine):
    # K above the narrow kernel's 40960: the narrow calls refuse the shape,
    # q1_qmm runs the prefill path even for M <= the row threshold
    N, K = 48, 40960 + 512
    t, x = _case(N, K, 3, affine, seed=23)
    W = q1.Q1Weight.from_host(t)
    with pytest.raises(q1.Q1Error):
        q1.qmv(W, x[0].to(DEV))
    with pytest.raises(q1.Q1Error):
        q1.qmm_narrow(W, x.to(DEV))
    y = q1.qmm(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), "qmm K=41472")


@pytest.mark.parametrize("affine", [False, True])
def test_narrow_mixed_magnitudes(q1, affine):
    # rows far above and below 1, and groups with a single large outlier: the
    # activations enter the MMAs scaled by 1/d_p (up to 2^7), in bf16 range
    M, N, K = 8, 512, 2048
    t, x = _case(N, K, M, affine, seed=17)
    x = x.float()
    x[1] *= 1e6
    x[2] *= 1e-6
    x[3, 5] *= 1e4
    x[4, 130:140] = 0.0
    x[5, 256:384] = 0.0  # an all-zero group
    x = x.to(torch.bfloat16)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm_narrow(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), "narrow mixed magnitudes")


def test_narrow_deterministic(q1):
    t, x = _case(2048, 5120, 4, False, seed=7)
    W = q1.Q1Weight.from_host(t)
    xd = x.to(DEV)
    a = q1.qmm_narrow(W, xd)
    b = q1.qmm_narrow(W, xd)
    assert torch.equal(a, b)


def test_symmetric_complement_negates_on_gpu(q1):
    K, N = 1024, 256
    t, x = _case(N, K, 2, False, seed=11)
    W = q1.Q1Weight.from_host(t)
    Wc = q1.Q1Weight.from_host(synth.Q1Tensor(~t.words, t.scales, None, K))
    y = q1.qmm_narrow(W, x.to(DEV)).float()
    yc = q1.qmm_narrow(Wc, x.to(DEV)).float()
    # negation holds in exact arithmetic; allow the bar's rounding on both
    wd = O.dequantize_f32(t.words, t.scales, None, K)
    check_matmul(-yc, O.qmm(x, t.words, t.scales, None, K), x, wd, "complement")
    assert torch.allclose(y, -yc, rtol=0, atol=float(np.abs(wd).max()) * 2)


# ------------------------------------------------------------------ dispatch / wide
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("M,N,K", [(9, 512, 1024), (128, 256, 1024), (130, 300, 640),
                                   (256, 1024, 1024), (200, 256, 128)])
def test_qmm_wide(q1, affine, M, N, K):
    t, x = _case(N, K, M, affine, seed=M + N + K + affine)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"wide M={M} N={N} K={K}")


def test_wide_equals_dense_fp16_weight_product(q1):
    # the prefill path multiplies exactly the fp16 weights q1_dequantize returns
    M, N, K = 256, 512, 2048
    t, x = _case(N, K, M, True, seed=99)
    W = q1.Q1Weight.from_host(t)
    xd = x.to(DEV)
    y = q1.qmm(W, xd).float()
    wd16 = q1.dequantize(W, torch.float16).double()
    ref = xd.double() @ wd16.T
    mag = xd.double().abs() @ wd16.abs().T
    # the bf16 output rounding (half-ulp 2^-8) and fp32 accumulation separate the two
    assert torch.all((y.double() - ref).abs() <= 2.0 ** -8 * ref.abs() + 1e-6 * mag)


@pytest.mark.parametrize("affine", [False, True])
def test_wide_one_hot_selects_exact_weights(q1, affine):
    # x = identity rows: Y[m][n] = Wd[n][m] exactly (one product, no sums)
    M, N, K = 128, 300, 128
    t = synth.q1_tensor(N, K, seed=7 + affine, affine=affine)
    W = q1.Q1Weight.from_host(t)
    x = torch.eye(M, K, dtype=torch.bfloat16)
    y = q1.qmm(W, x.to(DEV)).cpu()
    want = O.dequantize(t.words, t.scales, t.biases, K, "f16").to(torch.bfloat16).T
    np.testing.assert_array_equal(_u16(y), _u16(want[:M].contiguous()))


def test_wide_large_and_tiny_activations(q1):
    # rows far outside the fp16 range (and far below it) go through the
    # per-row power-of-two scale of the prefill path
    M, N, K = 200, 256, 1024
    t, x = _case(N, K, M, False, seed=3)
    scale = torch.ones(M, 1)
    scale[::3] = 1e6
    scale[1::3] = 1e-6
    x = (x.float() * scale).to(torch.bfloat16)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, None, K), x,
                 O.dequantize_f32(t.words, t.scales, None, K), "wide scaled rows")


@pytest.fixture
def prefill_plan(q1):
    yield q1.set_prefill_plan
    q1.set_prefill_plan(0, 0)


# every token-tile width class and schedule of the pair kernel, forced:
# persistent tiles (split 1) with the staged TMA-store epilogue (N % 8 == 0)
# and the direct one (N % 8 != 0, fp32 outputs), split-K clusters of 2..4
# pairs summing partial tiles through distributed shared memory, and equal
# runs of work per pair (split 0) whose shared tiles are summed through the
# workspace (here a tile is shared by up to a dozen pairs)
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("NT,S", [(16, 1), (48, 1), (128, 1), (208, 1), (256, 1), (128, 2), (64, 3), (256, 4),
                                  (256, 0), (128, 0), (48, 0)])
def test_prefill_forced_plans(q1, prefill_plan, NT, S, affine):
    M, N, K = 300, 768, 2048
    t, x = _case(N, K, M, affine, seed=NT + 7 * S + affine)
    W = q1.Q1Weight.from_host(t)
    prefill_plan(NT, S)
    y = q1.qmm(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"prefill plan NT={NT} S={S}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("NT,S", [(208, 1), (96, 2), (160, 0)])
def test_prefill_forced_plans_ragged(q1, prefill_plan, dtype, NT, S):
    M, N, K = 250, 600, 1280
    t = synth.q1_tensor(N, K, seed=801 + NT, affine=True)
    x = _acts(M, K, 802 + S, dtype)
    W = q1.Q1Weight.from_host(t)
    prefill_plan(NT, S)
    y = q1.qmm(W, x.to(DEV))
    assert y.dtype == dtype
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"prefill ragged NT={NT} S={S} {dtype}")


@pytest.mark.parametrize("NT,S", [(256, 1), (256, 0), (128, 1)])
def test_prefill_forced_plans_fp16_out(q1, prefill_plan, NT, S):
    # fp16 activations and outputs through the staged epilogue: full rounds of
    # 64 columns, a last token tile of 88 tokens (M = 600), N % 8 == 0
    M, N, K = 600, 768, 1280
    t = synth.q1_tensor(N, K, seed=806 + NT + S, affine=True)
    x = _acts(M, K, 807, torch.float16)
    W = q1.Q1Weight.from_host(t)
    prefill_plan(NT, S)
    y = q1.qmm(W, x.to(DEV))
    assert y.dtype == torch.float16
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"prefill fp16 NT={NT} S={S}")


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("NT,S", [(144, 1), (80, 3), (224, 0)])
def test_prefill_forced_plans_small_groups(q1, prefill_plan, group, NT, S):
    M, N, K = 200, 512, 1536
    t = synth.q1_tensor(N, K, seed=811 + group, affine=True, group=group)
    x = synth.activations(M, K, seed=812)
    W = q1.Q1Weight.from_host(t)
    prefill_plan(NT, S)
    y = q1.qmm(W, x.to(DEV))
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"prefill g{group} NT={NT} S={S}")


def test_prefill_stream_repeated_calls_same_result(q1, prefill_plan):
    # the share counts return to zero after each tile, and the shares are
    # summed in k order: repeated calls give identical bits
    M, N, K = 700, 1024, 4096
    t, x = _case(N, K, M, True, seed=821)
    W = q1.Q1Weight.from_host(t)
    prefill_plan(256, 0)
    xd = x.to(DEV)
    ws = q1.qmm_workspace(M, N, K, DEV)
    y0 = q1.qmm(W, xd, workspace=ws)
    for _ in range(3):
        assert torch.equal(q1.qmm(W, xd, workspace=ws), y0)
    check_matmul(y0, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), "prefill stream repeated")


def test_wide_workspace_required(q1):
    t, x = _case(256, 1024, 64, False, seed=1)
    W = q1.Q1Weight.from_host(t)
    with pytest.raises(q1.Q1Error):
        q1.lib()  # library loaded
        y = torch.empty(64, 256, dtype=torch.bfloat16, device=DEV)
        st = q1.lib().q1_qmm(W.cref(), x.to(DEV).data_ptr(), 64, 0, y.data_ptr(), None, 0,
                             torch.cuda.current_stream().cuda_stream)
        q1._check("q1_qmm", st)


def test_threshold_dispatch(q1):
    K, N = 1024, 512
    t, x = _case(N, K, 9, False, seed=5)
    W = q1.Q1Weight.from_host(t)
    yo = O.qmm(x, t.words, t.scales, None, K)
    wd = O.dequantize_f32(t.words, t.scales, None, K)
    old = q1.get_qmm_max_rows()
    try:
        for rows in (0, 4, 8):
            q1.set_qmm_max_rows(rows)
            for M in (1, 4, 5, 8, 9):
                y = q1.qmm(W, x[:M].to(DEV))
                check_matmul(y, yo[:M], x[:M], wd, f"threshold={rows} M={M}")
    finally:
        q1.set_qmm_max_rows(old)
    with pytest.raises(q1.Q1Error):
        q1.qmm_narrow(W, x.to(DEV))  # M = 9 is not narrow


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M", [9, 13, 16, 17])
def test_qmm_nine_to_sixteen_rows(q1, dtype, M):
    # at the default threshold, 9..16 rows run as two narrow launches (8 and
    # M - 8 rows; the second one's x and y start 8 rows in), 17 rows on the
    # prefill path; N = 601 leaves the second chunk's y at an odd row offset
    N, K = 601, 1280
    t = synth.q1_tensor(N, K, seed=901 + M, affine=True)
    x = _acts(M, K, 902 + M, dtype)
    W = q1.Q1Weight.from_host(t)
    assert q1.get_qmm_max_rows() == 8
    y = q1.qmm(W, x.to(DEV))
    assert y.dtype == dtype
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"qmm M={M} {dtype}")
    if M <= 16:
        # the same bits as the narrow kernel on each chunk
        y0 = q1.qmm_narrow(W, x[:8].to(DEV))
        y1 = q1.qmm_narrow(W, x[8:].to(DEV))
        assert torch.equal(y, torch.cat([y0, y1]))


# ------------------------------------------------------------------ gather / head
@pytest.mark.parametrize("affine", [False, True])
def test_embed_gather_bit_exact(q1, affine):
    V, K = 3000, 640
    t = synth.q1_tensor(V, K, seed=1003 + affine, affine=affine)
    E = q1.Q1Weight.from_host(t)
    ids = synth.token_ids(64, V, seed=1003)
    ids[5], ids[9] = -1, V  # out of range -> zero rows, counted
    for dt, name in ((torch.bfloat16, "bf16"), (torch.float32, "f32"), (torch.float16, "f16")):
        out, bad = q1.embed_gather(E, torch.from_numpy(ids).to(DEV), dt)
        want, nbad = O.embed_gather(ids, t.words, t.scales, t.biases, K, name)
        assert int(bad.item()) == nbad == 2
        g, w_ = out.cpu(), want
        if dt == torch.float32:
            np.testing.assert_array_equal(g.view(torch.int32).numpy(), w_.view(torch.int32).numpy())
        else:
            np.testing.assert_array_equal(_u16(g), _u16(w_))


def test_embed_gather_empty(q1):
    t = synth.q1_tensor(10, 128, seed=1, affine=False)
    E = q1.Q1Weight.from_host(t)
    out, bad = q1.embed_gather(E, torch.zeros(0, dtype=torch.int32, device=DEV))
    assert out.shape == (0, 128) and int(bad.item()) == 0


# ------------------------------------------------------------------ fused FFN
@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("D,F", [(512, 1408), (4096, 1024)])
def test_ffn_fused(q1, M, D, F):
    gate = synth.q1_tensor(F, D, seed=301, affine=False)
    up = synth.q1_tensor(F, D, seed=302, affine=(M == 4))  # mixed metadata once
    down = synth.q1_tensor(D, F, seed=303, affine=False)
    x = synth.activations(M, D, seed=304)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    ws = q1.ffn_workspace(M, D, F, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws)
    yo, ho = O.ffn(x, (gate.words, gate.scales, None, D), (up.words, up.scales, up.biases, D),
                   (down.words, down.scales, None, F))
    # h against the oracle's fp64 h (bf16-rounded on the GPU)
    h = q1.ffn_h(ws, M, F).float().cpu().double().numpy()
    assert np.linalg.norm(h - ho) / np.linalg.norm(ho) < 5e-3
    check_matmul(y, yo, ho, O.dequantize_f32(down.words, down.scales, None, F), f"ffn M={M}")


_NAME = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_ffn_fused_all_affine(q1, M, dtype):
    # gate, up and down all with stored biases: the down product's output is
    # dominated by the group means times sums of h, so the bar includes the
    # output's own rounding (tests/tolerance.py)
    D, F = 512, 1408
    gate = synth.q1_tensor(F, D, seed=311, affine=True)
    up = synth.q1_tensor(F, D, seed=312, affine=True)
    down = synth.q1_tensor(D, F, seed=313, affine=True)
    x = _acts(M, D, 314 + M, dtype) if dtype != torch.bfloat16 else synth.activations(M, D, seed=314 + M)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    ws = q1.ffn_workspace(M, D, F, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws)
    assert y.dtype == dtype
    tup = lambda t, K: (t.words, t.scales, t.biases, K)
    # the narrow kernels' tensor-core operands are bf16: fp16 and fp32
    # activations are rounded to bf16 once as they are loaded (include/q1.h).
    # Through all-affine gate/up/down that input rounding reaches y amplified
    # by the group means (7.8e-3 relative Frobenius error measured at M = 1,
    # fp16), so the oracle takes the activations as the kernel consumes them
    x_in = x if dtype == torch.bfloat16 else x.to(torch.bfloat16)
    yo, ho = O.ffn(x_in, tup(gate, D), tup(up, D), tup(down, F))
    h = q1.ffn_h(ws, M, F).float().cpu().double().numpy()
    assert np.linalg.norm(h - ho) / np.linalg.norm(ho) < 5e-3
    check_matmul(y, yo, ho, O.dequantize_f32(down.words, down.scales, down.biases, F),
                 f"affine ffn M={M} {dtype}", rounded_to=_NAME[dtype])


# ------------------------------------------------------------------ bf16 metadata
def _bf16_meta(t):
    """The same bits with the drawn metadata rounded to bf16 (torch tensors)."""
    s = torch.from_numpy(t.scales.astype(np.float32)).to(torch.bfloat16)
    b = None if t.biases is None else torch.from_numpy(t.biases.astype(np.float32)).to(torch.bfloat16)
    return t.words, s, b


def _dev_bf16(t):
    w, s, b = _bf16_meta(t)
    return q1_weight_from(w, s, b, t.K)


def q1_weight_from(words, s, b, K):
    from bit_affine_quantized_g128_gb300 import q1 as mod
    return mod.Q1Weight(torch.from_numpy(words.view("<i4").copy()).to(DEV), s.to(DEV),
                        None if b is None else b.to(DEV), K)


@pytest.mark.parametrize("affine", [False, True])
def test_bf16_metadata_dequantize_and_gather_bit_exact(q1, affine):
    N, K = 300, 640
    t = synth.q1_tensor(N, K, seed=601 + affine, affine=affine)
    w, s, b = _bf16_meta(t)
    # one scale beyond fp16's range: fine for dequantize and gather (fp32 math)
    s[7, 2] = 65536.0
    W = q1_weight_from(w, s, b, K)
    for dt, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16"), (torch.float16, "f16")):
        got = q1.dequantize(W, dt).cpu()
        want = O.dequantize(w, s, b, K, name)
        it = torch.int32 if dt == torch.float32 else torch.int16
        assert torch.equal(got.view(it), want.view(it)), name
    ids = synth.token_ids(40, N, seed=603)
    ids[3] = 7
    out, bad = q1.embed_gather(W, torch.from_numpy(ids).to(DEV), torch.float32)
    want, nbad = O.embed_gather(ids, w, s, b, K, "f32")
    assert int(bad.item()) == nbad == 0
    assert torch.equal(out.cpu().view(torch.int32), want.view(torch.int32))


@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("M", [1, 3, 8, 200])
def test_bf16_metadata_matmul(q1, affine, M):
    N, K = 777, 1536
    t, x = _case(N, K, M, affine, seed=611 + M + affine)
    w, s, b = _bf16_meta(t)
    W = q1_weight_from(w, s, b, K)
    y = q1.qmm(W, x.to(DEV))  # narrow for M <= 8, prefill for M = 200
    check_matmul(y, O.qmm(x, w, s, b, K), x, O.dequantize_f32(w, s, b, K), f"bf16 meta M={M}")


def test_bf16_metadata_ffn_mixed_with_fp16(q1):
    # gate bf16, up fp16, down bf16: the gate/up launch reads each matrix's own type
    M, D, F = 4, 512, 1408
    gate = synth.q1_tensor(F, D, seed=621, affine=False)
    up = synth.q1_tensor(F, D, seed=622, affine=False)
    down = synth.q1_tensor(D, F, seed=623, affine=False)
    x = synth.activations(M, D, seed=624)
    gw, gs, _ = _bf16_meta(gate)
    dw, ds, _ = _bf16_meta(down)
    G, U, Dn = q1_weight_from(gw, gs, None, D), q1.Q1Weight.from_host(up), q1_weight_from(dw, ds, None, F)
    ws = q1.ffn_workspace(M, D, F, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws)
    yo, ho = O.ffn(x, (gw, gs, None, D), (up.words, up.scales, None, D), (dw, ds, None, F))
    check_matmul(y, yo, ho, O.dequantize_f32(dw, ds, None, F), "ffn bf16/fp16 metadata")


def test_bf16_metadata_check_symmetric(q1):
    t = synth.q1_tensor(64, 256, seed=631, affine=False)
    s = torch.from_numpy(t.scales.astype(np.float32)).to(torch.bfloat16)
    b = (s.float() * -0.5).to(torch.bfloat16)  # exact: halving a bf16 value
    W = q1_weight_from(t.words, s, b, 256)
    assert int(q1.check_symmetric(W).item()) == 1 == int(O.is_symmetric(s, b))
    b2 = b.clone()
    b2[5, 1] = 0.25
    W2 = q1_weight_from(t.words, s, b2, 256)
    assert int(q1.check_symmetric(W2).item()) == 0 == int(O.is_symmetric(s, b2))


def test_meta_dtype_is_validated(q1):
    t = synth.q1_tensor(16, 128, seed=641, affine=False)
    W = q1.Q1Weight.from_host(t)
    W._c.meta_dtype = 2
    x = torch.zeros((1, 128), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((1, 16), dtype=torch.bfloat16, device=DEV)
    st = q1.lib().q1_qmv(W.cref(), x.data_ptr(), 0, y.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 4  # Q1_ERR_DTYPE


# ------------------------------------------------------------------ fp16 / fp32 activations
def _acts(M, K, seed, dtype):
    """N(0, 1) activations drawn in fp32 (so that fp32 inputs carry more than
    bf16's 8 bits), rounded to fp16 for the fp16 case."""
    x = torch.from_numpy(np.random.default_rng(seed).standard_normal((M, K)).astype(np.float32))
    return x.to(dtype)


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("M", [1, 5, 8, 200])
def test_fp16_fp32_activations(q1, dtype, affine, M):
    N, K = 600, 1280
    t = synth.q1_tensor(N, K, seed=651 + affine, affine=affine)
    x = _acts(M, K, 652 + M, dtype)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV))  # narrow for M <= 8, prefill for M = 200
    assert y.dtype == dtype and y.shape == (M, N)
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"{dtype} M={M}")
    if M == 1:
        yv = q1.qmv(W, x[0].to(DEV))
        assert torch.equal(yv.reshape(1, N), y)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("M", [9, 300])
def test_prefill_ragged_rows_every_output_dtype(q1, dtype, M):
    # N % 8 != 0: the epilogues' element-wise tails (split-K clusters for M = 9,
    # whole tiles for M = 300) in every output dtype
    N, K = 601, 768
    t = synth.q1_tensor(N, K, seed=691, affine=True)
    x = _acts(M, K, 692 + M, dtype)
    W = q1.Q1Weight.from_host(t)
    y = q1.qmm(W, x.to(DEV))
    assert y.dtype == dtype
    check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x,
                 O.dequantize_f32(t.words, t.scales, t.biases, K), f"prefill N={N} M={M} {dtype}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.float32])
def test_ffn_fp16_fp32_activations(q1, dtype):
    M, D, F = 3, 512, 1408
    gate = synth.q1_tensor(F, D, seed=661, affine=False)
    up = synth.q1_tensor(F, D, seed=662, affine=False)
    down = synth.q1_tensor(D, F, seed=663, affine=False)
    x = _acts(M, D, 664, dtype)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    y = q1.ffn_fused(G, U, Dn, x.to(DEV))
    assert y.dtype == dtype
    yo, ho = O.ffn(x, (gate.words, gate.scales, None, D), (up.words, up.scales, None, D),
                   (down.words, down.scales, None, F))
    check_matmul(y, yo, ho, O.dequantize_f32(down.words, down.scales, None, F), f"ffn {dtype}")


# ------------------------------------------------------------------ group sizes 32 and 64
@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("affine", [False, True])
def test_small_groups(q1, group, affine):
    N, K = 300, 640
    t = synth.q1_tensor(N, K, seed=671 + group + affine, affine=affine, group=group)
    W = q1.Q1Weight.from_host(t)
    assert W.group_size == group
    for dt, name in ((torch.float32, "f32"), (torch.bfloat16, "bf16"), (torch.float16, "f16")):
        it = torch.int32 if dt == torch.float32 else torch.int16
        got = q1.dequantize(W, dt).cpu()
        assert torch.equal(got.view(it), O.dequantize(t.words, t.scales, t.biases, K, name).view(it)), name
    ids = synth.token_ids(24, N, seed=672)
    out, bad = q1.embed_gather(W, torch.from_numpy(ids).to(DEV), torch.bfloat16)
    want, _ = O.embed_gather(ids, t.words, t.scales, t.biases, K, "bf16")
    assert int(bad.item()) == 0 and torch.equal(out.cpu().view(torch.int16), want.view(torch.int16))
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    for M in (1, 8, 200):  # narrow (the per-word mapping) and prefill
        x = synth.activations(M, K, seed=673 + M)
        y = q1.qmm(W, x.to(DEV))
        check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x, wd, f"group {group} M={M}")


@pytest.mark.parametrize("group", [32, 64])
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("N,K", [(1024, 1024), (333, 640), (130, 5120), (48, 17408 // 4)])
def test_small_groups_narrow(q1, group, affine, N, K):
    # the narrow kernel's groups-of-32/64 path at every window size 1..8:
    # ragged row tiles, K of 5 to 34 spans (extra groups past the K-warps),
    # metadata rows whose group count is not a multiple of 8 (K = 640 at
    # group 64: 10 groups, loaded by the producer's lanes instead of TMA)
    t = synth.q1_tensor(N, K, seed=681 + group + affine + N, affine=affine, group=group)
    W = q1.Q1Weight.from_host(t)
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    for M in (1, 2, 3, 5, 8):
        x = synth.activations(M, K, seed=682 + M)
        y = q1.qmm_narrow(W, x.to(DEV))
        check_matmul(y, O.qmm(x, t.words, t.scales, t.biases, K), x, wd, f"group {group} narrow N={N} K={K} M={M}")
    y1 = q1.qmv(W, x[0].to(DEV))
    check_matmul(y1[None], O.qmm(x[:1], t.words, t.scales, t.biases, K), x[:1], wd, f"group {group} qmv")


@pytest.mark.parametrize("group", [32, 64])
def test_small_groups_fp16_fp32_and_bf16_metadata(q1, group):
    N, K = 600, 1280
    t = synth.q1_tensor(N, K, seed=691 + group, affine=True, group=group)
    W = q1.Q1Weight.from_host(t)
    wd = O.dequantize_f32(t.words, t.scales, t.biases, K)
    for dtype in (torch.float16, torch.float32):
        x = _acts(4, K, 692, dtype)
        y = q1.qmm_narrow(W, x.to(DEV))
        assert y.dtype == dtype
        # affine weights: the oracle takes the bf16 operands the kernel multiplies
        xb = x.to(torch.bfloat16)
        check_matmul(y, O.qmm(xb, t.words, t.scales, t.biases, K), xb, wd, f"group {group} {dtype}",
                     rounded_to=_NAME[dtype])
    w, s, b = _bf16_meta(t)
    Wb = q1_weight_from(w, s, b, K)
    x = synth.activations(3, K, seed=693)
    y = q1.qmm_narrow(Wb, x.to(DEV))
    check_matmul(y, O.qmm(x, w, s, b, K), x, O.dequantize_f32(w, s, b, K), f"group {group} bf16 metadata")


def test_small_groups_ffn_and_chain(q1):
    # gate/up with groups of 64, down with groups of 32; and a two-layer chain
    # mixing the three group sizes
    M, D, F = 4, 512, 1408
    gate = synth.q1_tensor(F, D, seed=701, affine=False, group=64)
    up = synth.q1_tensor(F, D, seed=702, affine=True, group=64)
    down = synth.q1_tensor(D, F, seed=703, affine=False, group=32)
    x = synth.activations(M, D, seed=704)
    G, U, Dn = (q1.Q1Weight.from_host(w) for w in (gate, up, down))
    ws = q1.ffn_workspace(M, D, F, DEV)
    y = q1.ffn_fused(G, U, Dn, x.to(DEV), workspace=ws)
    yo, ho = O.ffn(x, (gate.words, gate.scales, None, D), (up.words, up.scales, up.biases, D),
                   (down.words, down.scales, None, F))
    h = q1.ffn_h(ws, M, F).float().cpu().double().numpy()
    assert np.linalg.norm(h - ho) / np.linalg.norm(ho) < 5e-3
    check_matmul(y, yo, ho, O.dequantize_f32(down.words, down.scales, None, F), "ffn groups 64/32")
    # gate and up with different group sizes are refused
    U32 = q1.Q1Weight.from_host(synth.q1_tensor(F, D, seed=705, affine=False, group=32))
    with pytest.raises(q1.Q1Error) as e:
        q1.ffn_fused(G, U32, Dn, x.to(DEV))
    assert e.value.status == 5
    # chain: layer 0 with groups of 32 (attn) and 64 (gate/up), layer 1 of 128
    D2, F2 = 256, 512
    layers = []
    for l, (ga, gg, gd) in enumerate(((32, 64, 32), (128, 128, 64))):
        base = 710 + 10 * l
        layers.append((_scaled(synth.q1_tensor(D2, D2, seed=base, affine=False, group=ga), 7.0),
                       _scaled(synth.q1_tensor(F2, D2, seed=base + 1, affine=False, group=gg), 7.0),
                       _scaled(synth.q1_tensor(F2, D2, seed=base + 2, affine=False, group=gg), 7.0),
                       _scaled(synth.q1_tensor(D2, F2, seed=base + 3, affine=False, group=gd), 7.0)))
    dev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in layers]
    xc = synth.activations(2, D2, seed=729).to(DEV)
    yc = q1.decode_chain(dev, xc)
    hc = xc
    for A, Gg, Uu, Dd in dev:
        hc = q1.ffn_fused(Gg, Uu, Dd, q1.qmm_narrow(A, hc))
    torch.cuda.synchronize()
    assert torch.equal(yc, hc)


def test_small_groups_check_symmetric(q1):
    t = synth.q1_tensor(64, 256, seed=681, affine=False, group=32)
    s = t.scales
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    W = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b, 256))
    assert W.group_size == 32
    assert int(q1.check_symmetric(W).item()) == 1 == int(O.is_symmetric(s, b))
    b2 = b.copy()
    b2[63, 7] = np.float16(0.25)  # the last group of the last row
    W2 = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b2, 256))
    assert int(q1.check_symmetric(W2).item()) == 0 == int(O.is_symmetric(s, b2))


# ------------------------------------------------------------------ exact repack from dense
_TORCH = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
_INT = {"bf16": torch.int16, "f16": torch.int16, "f32": torch.int32}


def _planted_dense(t, dtype):
    """The dequantized tensor in `dtype` with edge-case groups planted (values
    exact in every dtype): +-0 pairs, single values, a third value, NaN and
    infinity."""
    d = O.round_to(O.dequantize_f32(t.words, t.scales, t.biases, t.K), dtype).clone()
    sign = torch.from_numpy(np.random.default_rng(5).integers(0, 2, 128).astype(bool))
    d[0, 0:128] = torch.where(sign, torch.tensor(0.0), torch.tensor(-0.0)).to(d.dtype)
    d[1, 128:256] = 0.5
    d[2, 256:384] = -0.5
    d[3, 5] = float("nan")
    d[4, 130] = float("inf")
    d[5, 7] = 3.0
    d[6, 0:128] = 0.0
    d[7, 128:256] = -0.0
    d[8, 256:384] = torch.where(sign, torch.tensor(0.75), torch.tensor(0.25)).to(d.dtype)
    return d


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("affine", [False, True])
def test_pack_from_dense_bit_exact(q1, dtype, affine):
    N, K = 37, 640
    t = synth.q1_tensor(N, K, seed=501 + affine, affine=affine)
    dense = _planted_dense(t, dtype)
    W, bad = q1.pack_from_dense(dense.to(DEV), symmetric=not affine)
    wo, so, bo, bado = O.pack_from_dense(dense, symmetric=not affine)
    assert int(bad.item()) == bado and bado >= 3
    np.testing.assert_array_equal(W.words.cpu().numpy().view(np.uint32), wo)
    np.testing.assert_array_equal(W.scales.cpu().numpy().view(np.uint16), so.view(np.uint16))
    if affine:
        np.testing.assert_array_equal(W.biases.cpu().numpy().view(np.uint16), bo.view(np.uint16))
    # every kept group dequantizes to exactly its input bits (the library's own dequantize)
    back = q1.dequantize(W, _TORCH[dtype]).cpu().view(_INT[dtype]).reshape(N, K // 128, 128)
    want = dense.view(_INT[dtype]).reshape(N, K // 128, 128)
    kept = torch.tensor([[O.pack_group(dense[n, g * 128:(g + 1) * 128].float().numpy(), not affine) is not None
                          for g in range(K // 128)] for n in range(N)])
    assert int((~kept).sum()) == bado
    assert torch.equal(back[kept], want[kept])


# ------------------------------------------------------------------ decode chain
def _scaled(t, factor):
    """The same bits with the metadata multiplied by `factor` (fp16): products
    of these shapes then keep activations of order one through the chain."""
    s = (t.scales.astype(np.float32) * factor).astype(np.float16)
    b = None if t.biases is None else (t.biases.astype(np.float32) * factor).astype(np.float16)
    return synth.Q1Tensor(t.words, s, b, t.K)


def _chain_host(D, Fs, seed, affine=(), factor=7.0):
    layers = []
    for l, F in enumerate(Fs):
        base = seed + 10 * l
        layers.append((
            _scaled(synth.q1_tensor(D, D, seed=base, affine=("attn", l) in affine), factor),
            _scaled(synth.q1_tensor(F, D, seed=base + 1, affine=("gate", l) in affine), factor),
            _scaled(synth.q1_tensor(F, D, seed=base + 2, affine=("up", l) in affine), factor),
            _scaled(synth.q1_tensor(D, F, seed=base + 3, affine=("down", l) in affine), factor)))
    return layers


@pytest.mark.parametrize("M", [1, 3, 8])
def test_decode_chain_equals_the_calls_made_one_by_one(q1, M):
    D, Fs = 256, [384, 256, 512]
    host = _chain_host(D, Fs, seed=400, affine={("attn", 1), ("up", 2), ("down", 0)})
    dev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in host]
    x = synth.activations(M, D, seed=409).to(DEV)
    y = q1.decode_chain(dev, x)
    h = x
    for A, G, U, Dn in dev:
        a = q1.qmm_narrow(A, h)
        h = q1.ffn_fused(G, U, Dn, a)
    torch.cuda.synchronize()
    assert torch.equal(y, h), "the chain differs from the same calls made one by one"
    assert float(y.float().abs().max()) > 0


@pytest.mark.parametrize("M", [1, 4])
def test_decode_chain_oracle(q1, M):
    D, Fs = 256, [512, 384]
    host = _chain_host(D, Fs, seed=430)
    dev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in host]
    x = synth.activations(M, D, seed=439)
    y = q1.decode_chain(dev, x.to(DEV))
    tup = lambda t: (t.words, t.scales, t.biases, t.K)
    layers = [tuple(tup(w) for w in L) for L in host]
    yo = O.decode_chain(x, layers)
    # the last product's input: the oracle's FFN intermediate of the last layer
    h_prev = O.decode_chain(x, layers[:-1]) if len(layers) > 1 else x
    attn, gate, up, down = layers[-1]
    a = O.round_to(O.qmm(h_prev, *attn), "bf16")
    _, h_last = O.ffn(a, gate, up, down)
    wd = O.dequantize_f32(down[0], down[1], down[2], down[3])
    check_chain(y, yo.double().numpy(), h_last, wd, stages=3 * len(layers), what=f"chain M={M}")


@pytest.mark.parametrize("M", [1, 4])
def test_decode_chain_affine_layers_stage_by_stage(q1, M):
    # every matrix of both layers affine.  The chain equals the same calls
    # made one by one, bit for bit; each of those calls is then held to the
    # single-product bar against the oracle computed from the GPU's own bf16
    # input to it (the attention product and the whole FFN block)
    D, Fs = 256, [512, 384]
    every = {(n, l) for n in ("attn", "gate", "up", "down") for l in range(len(Fs))}
    # metadata x2: with stored biases the group means make the activations
    # grow from layer to layer, and x7 (the symmetric tests' factor) would
    # overflow bf16 by the second layer
    host = _chain_host(D, Fs, seed=470, affine=every, factor=2.0)
    dev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in host]
    x = synth.activations(M, D, seed=479)
    y = q1.decode_chain(dev, x.to(DEV))
    tup = lambda t: (t.words, t.scales, t.biases, t.K)
    h = x.to(DEV)
    for l, ((A, G, U, Dn), (ta, tg, tu, td)) in enumerate(zip(dev, host)):
        a = q1.qmm_narrow(A, h)
        h_in = h.cpu()
        check_matmul(a, O.qmm(h_in, *tup(ta)), h_in, O.dequantize_f32(ta.words, ta.scales, ta.biases, D),
                     f"chain layer {l} attn M={M}", rounded_to="bf16")
        ws = q1.ffn_workspace(M, D, Fs[l], DEV)
        h = q1.ffn_fused(G, U, Dn, a, workspace=ws)
        a_in = a.cpu()
        yo, ho = O.ffn(a_in, tup(tg), tup(tu), tup(td))
        hg = q1.ffn_h(ws, M, Fs[l]).float().cpu().double().numpy()
        assert np.linalg.norm(hg - ho) / np.linalg.norm(ho) < 5e-3, f"layer {l} h"
        check_matmul(h, yo, ho, O.dequantize_f32(td.words, td.scales, td.biases, Fs[l]),
                     f"chain layer {l} ffn M={M}", rounded_to="bf16")
    torch.cuda.synchronize()
    assert torch.equal(y, h), "the chain differs from the same calls made one by one"
    assert float(y.float().abs().max()) > 0


def test_decode_chain_rejects_bad_arguments(q1):
    D = 256
    host = _chain_host(D, [256], seed=450)
    dev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in host]
    x = synth.activations(2, D, seed=459).to(DEV)
    y = torch.empty_like(x)
    lib = q1.lib()
    arr = (q1._CLayer * 1)(q1._CLayer(*(w._c for w in dev[0])))
    ws = q1.decode_chain_workspace(2, D, 256, DEV)
    st = torch.cuda.current_stream().cuda_stream
    call = lambda layers, n, M, nbytes: lib.q1_decode_chain(layers, n, x.data_ptr(), M, 0, y.data_ptr(),
                                                            ws.data_ptr(), nbytes, st)
    assert call(arr, 0, 2, ws.numel()) == 2          # no layers
    assert call(arr, 1, 9, ws.numel()) == 2          # M > 8
    assert call(arr, 1, 2, 256) == 6                 # workspace too small
    bad = _chain_host(D, [256], seed=460)
    bad[0] = (synth.q1_tensor(128, D, seed=461, affine=False),) + bad[0][1:]  # attn not [D][D]
    bdev = [tuple(q1.Q1Weight.from_host(w) for w in L) for L in bad]
    barr = (q1._CLayer * 1)(q1._CLayer(*(w._c for w in bdev[0])))
    assert call(barr, 1, 2, ws.numel()) == 2
    torch.cuda.synchronize()


# ------------------------------------------------------------------ symmetric check
def test_check_symmetric(q1):
    t = synth.q1_tensor(64, 256, seed=9, affine=False)
    s = np.maximum(t.scales, np.float16(2.0 ** -13))
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    W = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b, 256))
    assert int(q1.check_symmetric(W).item()) == 1 == int(O.is_symmetric(s, b))
    b2 = b.copy()
    b2[63, 1] = np.float16(0.25)
    W2 = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b2, 256))
    assert int(q1.check_symmetric(W2).item()) == 0 == int(O.is_symmetric(s, b2))


def test_check_symmetric_tail_and_unaligned_metadata(q1):
    # 3 x 3 groups: one 8-group vector and a scalar tail; then the same
    # metadata 2 bytes past a 16-byte boundary (the element-wise path)
    N, K = 3, 384
    t = synth.q1_tensor(N, K, seed=701, affine=False)
    s = np.maximum(t.scales, np.float16(2.0 ** -13))
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    for bad in (None, (2, 2), (0, 1)):  # (2, 2) is the tail element
        b2 = b.copy()
        if bad:
            b2[bad] = np.float16(0.5)
        W = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b2, K))
        want = int(O.is_symmetric(s, b2))
        assert int(q1.check_symmetric(W).item()) == want == (0 if bad else 1)
        sd = torch.from_numpy(np.concatenate([[np.float16(1)], s.reshape(-1)])).to(DEV)[1:].reshape(N, 3)
        bd = torch.from_numpy(np.concatenate([[np.float16(1)], b2.reshape(-1)])).to(DEV)[1:].reshape(N, 3)
        Wu = q1.Q1Weight(W.words, sd, bd, K)
        assert Wu.scales.data_ptr() % 16 != 0
        assert int(q1.check_symmetric(Wu).item()) == want


def _f16(bits):
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


@pytest.mark.parametrize("unaligned", [False, True])
@pytest.mark.parametrize("case", ["pm_zero", "nan_scale", "nan_bias", "tiny_scale", "neg_zero_scale"])
def test_check_symmetric_edge_cases(q1, case, unaligned):
    # the cases the oracle's is_symmetric is pinned on, run through the
    # kernel's 16-byte vector path (aligned metadata, 8 groups per load) and
    # its element-wise path (metadata 2 bytes past a 16-byte boundary)
    N, K = 5, 1024  # 8 groups per row
    t = synth.q1_tensor(N, K, seed=711, affine=False)
    s = np.maximum(t.scales, np.float16(2.0 ** -13))
    b = (-(s.astype(np.float32) / 2)).astype(np.float16)
    r, g = 3, 6
    if case == "pm_zero":        # scale +0 with bias +0 (derived -0): equal
        s[r, g], b[r, g] = np.float16(0.0), np.float16(0.0)
        s[r, g + 1], b[r, g + 1] = np.float16(-0.0), np.float16(-0.0)  # derived +0 vs -0
    elif case == "neg_zero_scale":  # scale -0, bias -0 stored: derived +0 == -0
        s[r, g], b[r, g] = np.float16(-0.0), np.float16(-0.0)
    elif case == "nan_scale":
        s[r, g] = np.float16(np.nan)
    elif case == "nan_bias":
        b[r, g] = np.float16(np.nan)
    elif case == "tiny_scale":   # -s/2 is not an fp16 value: no stored bias equals it
        s[r, g] = _f16(0x0001)
        b[r, g] = (-(s[r, g].astype(np.float32) / 2)).astype(np.float16)
    want = int(O.is_symmetric(s, b))
    assert want == (1 if case in ("pm_zero", "neg_zero_scale") else 0)
    if unaligned:
        sd = torch.from_numpy(np.concatenate([[np.float16(1)], s.reshape(-1)])).to(DEV)[1:].reshape(N, K // 128)
        bd = torch.from_numpy(np.concatenate([[np.float16(1)], b.reshape(-1)])).to(DEV)[1:].reshape(N, K // 128)
        W = q1.Q1Weight(torch.from_numpy(t.words.view("<i4").copy()).to(DEV), sd, bd, K)
        assert W.scales.data_ptr() % 16 != 0
    else:
        W = q1.Q1Weight.from_host(synth.Q1Tensor(t.words, s, b, K))
        assert W.scales.data_ptr() % 16 == 0 and W.biases.data_ptr() % 16 == 0
    assert int(q1.check_symmetric(W).item()) == want


def test_no_device_errors_after_suite(q1):
    assert q1.device_errors() == 0
