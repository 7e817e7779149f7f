"""GPU parity of the tcgen05 prefill dequant-GEMM (Y = X W^T, W Q4_K, X bf16,
f32 accumulate) against the oracle, through the C ABI.

Bar: |err| <= 5e-3 * sum|w_i x_i| + 1e-5 per output and cosine >= 0.9999.
Small shapes are compared in full; the prefill workload (fused gate||up
34816x5120 and down 5120x17408, P = 256/512/1024 tokens, seed 2) on sampled
rows x tokens that the oracle computes one by one.

The gate||up GEMM with the SwiGLU in its epilogue is checked three ways: its
interleaved weight rows byte for byte against the permutation written out in
numpy, its output bit for bit against the unfused GEMM followed by the SwiGLU
kernel (full gate||up shape, no K split), and small shapes against the oracle's
silu(g)*u with the GEMM bar carried through the product (below).
"""
import numpy as np
import pytest

import oracle
import synth
from _util import check_f32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fak():
    from q4_weight_quantized_block_gb300 import build
    build.build()
    import q4_weight_quantized_block_gb300 as m
    assert torch.cuda.is_available()
    return m


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gemm(fak, Wg, N, K, Xb, P):
    Y = torch.full((P, N), float("nan"), device="cuda")
    fak.fak_q4k_gemm(Wg, N, K, Xb, P, Y)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    return Y


def check_gemm(got, ref, a, what):
    check_f32(got, ref, a, what, rel=5e-3, abs_=1e-5, cos_min=0.9999)


# Shapes with few tiles run stream-K (the tiles' K work cut into one range per SM, pieces summed in
# K order by the fix-up kernel): (384, 1280, 300) and (128, 2048, 513) with ragged token tails,
# (512, 5120, 64), (640, 8192, 256) with uneven ranges, (128, 10496, 64) with 41 pieces of one tile,
# and (1000, 8192, 64) whose last row tile is partial.  The others take whole tiles; N that is not a
# multiple of 128 leaves a last partial row tile there too: (200, 512, 33) and the GDN in_proj rows
# (16480, 5120, 8).
@pytest.mark.parametrize("N,K,P", [(128, 256, 1), (128, 256, 7), (256, 512, 256), (384, 1280, 300),
                                   (128, 2048, 513), (512, 5120, 64), (640, 8192, 256), (128, 10496, 64),
                                   (200, 512, 33), (16480, 5120, 8), (1000, 8192, 64)])
def test_gemm_small_full_compare(fak, N, K, P):
    w = synth.normal(40, N + K + P, (N, K), 0.02)
    Wg, Wo = fak.fak_q4k_pack(w), oracle.q4k_pack(w)
    assert np.array_equal(Wg, Wo)
    Xb = synth.to_bf16(synth.normal(41, N + K + P, (P, K), 1.0))
    Yref, A = oracle.gemm_q4k(Wo, N, K, Xb)
    Y = gemm(fak, dev(Wg), N, K, dev(Xb.view(np.int16)), P)
    check_gemm(Y.cpu().numpy(), Yref, A, "gemm %dx%dx%d" % (N, K, P))


@pytest.mark.parametrize("N,K,P", [(256, 1024, 300), (640, 8192, 256), (128, 10496, 64)])
def test_gemm_deterministic(fak, N, K, P):
    w = synth.normal(42, 0, (N, K), 0.02)
    Wg = dev(fak.fak_q4k_pack(w))
    Xb = dev(synth.to_bf16(synth.normal(42, 1, (P, K), 1.0)).view(np.int16))
    a = gemm(fak, Wg, N, K, Xb, P).cpu().numpy()
    b = gemm(fak, Wg, N, K, Xb, P).cpu().numpy()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("N,K,P", [(34816, 5120, 512), (5120, 17408, 512), (5120, 6144, 256)])
def test_gemm_deterministic_full_shape(fak, N, K, P):
    # the prefill shapes (whole tiles; stream-K with the fix-up): repeated calls agree bit for bit,
    # so every producer / consumer hand-off of the pipeline is ordered (a reader that ran ahead of a
    # ring slot's refill would read stale quants in some calls and not in others)
    w = torch.empty(N * K, device="cuda")
    synth.normal_device(w, 44, 0, 0.02)
    Wg = torch.empty(N * K // 256 * 144, dtype=torch.uint8, device="cuda")
    fak.fak_q4k_pack_device(w, N, K, Wg)
    xf = torch.empty(P * K, device="cuda")
    synth.normal_device(xf, 44, 1, 1.0)
    Xb = xf.view(P, K).to(torch.bfloat16).view(torch.int16)
    del w, xf
    ref = gemm(fak, Wg, N, K, Xb, P)
    assert torch.isfinite(ref).all()
    for _ in range(8):
        assert torch.equal(gemm(fak, Wg, N, K, Xb, P).view(torch.int32), ref.view(torch.int32))


def test_swiglu_bf16(fak):
    P, half = 5, 1000
    Y1 = synth.normal(43, 0, (P, 2 * half), 3.0)
    X2 = torch.empty((P, half), dtype=torch.int16, device="cuda")
    fak.fak_swiglu_bf16(dev(Y1), P, half, X2)
    torch.cuda.synchronize()
    got = (X2.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y = Y1.astype(np.float64)
    ref = oracle.swiglu(y[:, :half].ravel(), y[:, half:].ravel()).reshape(P, half)
    # one bf16 rounding of an f32-computed value: within 2^-8 relative (+ tiny absolute)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)


def tile_samples(n, tile, rng, extra=8):
    """One random index in every `tile`-sized block of range(n), plus the ends and a few extra."""
    picks = [rng.integers(b, min(b + tile, n)) for b in range(0, n, tile)]
    picks += [0, n - 1] + list(rng.choice(n, extra, replace=False))
    return np.unique(np.array(picks, dtype=np.int64))


@pytest.mark.parametrize("P", [256, 512, 1024])
def test_prefill_workload_sampled(fak, P):
    # fused gate||up 34816 x 5120 (seed 2, tensor 0), down 5120 x 17408 (tensor 1), X (tensor 2);
    # sampled outputs cover one row in every 128-row tile and one token in every 256-token tile
    D, F = 5120, 17408
    w1 = synth.normal(2, 0, (2 * F, D), 0.02)
    W1g, W1o = fak.fak_q4k_pack(w1), oracle.q4k_pack(w1)
    assert np.array_equal(W1g, W1o)
    del w1
    Xb = synth.to_bf16(synth.normal(2, 2, (P, D), 1.0))
    Y1 = gemm(fak, dev(W1g), 2 * F, D, dev(Xb.view(np.int16)), P)
    rng = np.random.default_rng(P)
    rows = tile_samples(2 * F, 128, rng)
    toks = tile_samples(P, 256, rng, extra=4)
    Yr, Ar = oracle.gemm_q4k_sample(W1o, 2 * F, D, Xb, rows, toks)
    check_gemm(Y1.cpu().numpy()[np.ix_(toks, rows)], Yr, Ar, "prefill gate||up P=%d" % P)
    # second shape, isolated: down projection on the GPU's own SwiGLU output
    X2 = torch.empty((P, F), dtype=torch.int16, device="cuda")
    fak.fak_swiglu_bf16(Y1, P, F, X2)
    w2 = synth.normal(2, 1, (D, F), 0.02)
    W2g, W2o = fak.fak_q4k_pack(w2), oracle.q4k_pack(w2)
    del w2
    Y2 = gemm(fak, dev(W2g), D, F, X2, P)
    X2h = X2.cpu().numpy().view(np.uint16)
    rows2 = tile_samples(D, 128, rng)
    Yr2, Ar2 = oracle.gemm_q4k_sample(W2o, D, F, X2h, rows2, toks)
    check_gemm(Y2.cpu().numpy()[np.ix_(toks, rows2)], Yr2, Ar2, "prefill down P=%d" % P)
    # second shape, end to end from the oracle's own X2 = bf16(silu(g) * u) for two tokens: the GPU's
    # down GEMM fed with it meets the GEMM bar, and the GPU's whole pipeline (its own X2) stays
    # within twice the bar (two bf16 GEMMs in series) of the oracle's whole pipeline
    t2 = np.array([0, P - 1])
    Yfull, _ = oracle.gemm_q4k(W1o, 2 * F, D, Xb[t2])
    x2o = synth.to_bf16(oracle.swiglu(Yfull[:, :F].ravel(), Yfull[:, F:].ravel()).astype(np.float32)).reshape(2, F)
    Yo2, Ao2 = oracle.gemm_q4k(W2o, D, F, x2o)
    Yg2 = gemm(fak, dev(W2g), D, F, dev(x2o.view(np.int16)), 2)
    check_gemm(Yg2.cpu().numpy(), Yo2, Ao2, "prefill down from the oracle's X2, P=%d" % P)
    check_f32(Y2.cpu().numpy()[t2], Yo2, Ao2, "prefill gate||up -> SwiGLU -> down end to end, P=%d" % P,
              rel=1e-2, abs_=2e-5, cos_min=0.9999)


def interleave_rows(g, u):
    """The row order fak_q4k_gemm_swiglu reads: per 16 channels, 16 gate rows then 16 up rows."""
    F = g.shape[0]
    out = np.empty((2 * F,) + g.shape[1:], g.dtype)
    for b in range(F // 16):
        out[32 * b:32 * b + 16] = g[16 * b:16 * b + 16]
        out[32 * b + 16:32 * b + 32] = u[16 * b:16 * b + 16]
    return out


def test_interleave_gate_up_bytes(fak):
    F, K = 192, 768
    g = fak.fak_q4k_pack(synth.normal(44, 0, (F, K), 0.02))
    u = fak.fak_q4k_pack(synth.normal(44, 1, (F, K), 0.02))
    W13 = torch.zeros((2 * F, g.shape[1]), dtype=torch.uint8, device="cuda")
    fak.fak_q4k_interleave_gate_up(dev(g), dev(u), F, K, W13)
    torch.cuda.synchronize()
    assert np.array_equal(W13.cpu().numpy(), interleave_rows(g, u))


def bf16_bits_to_f64(t):
    return (t.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("P", [64, 300])
def test_gemm_swiglu_equals_unfused(fak, P):
    # full gate||up shape (seed 2 workload): 272 row tiles, so the unfused GEMM runs without a K split
    D, F = 5120, 17408
    scratch = torch.empty(2 * F * D, dtype=torch.float32, device="cuda")
    synth.normal_device(scratch, 2, 0, 0.02)
    W1 = torch.empty(2 * F * D // 256 * 144, dtype=torch.uint8, device="cuda")
    fak.fak_q4k_pack_device(scratch, 2 * F, D, W1)
    Xf = scratch[: P * D]
    synth.normal_device(Xf, 2, 2, 1.0)
    X = Xf.view(P, D).to(torch.bfloat16)
    del scratch, Xf
    row = D // 256 * 144
    W13 = torch.empty_like(W1)
    fak.fak_q4k_interleave_gate_up(W1[: F * row], W1[F * row:], F, D, W13)
    Y1 = gemm(fak, W1, 2 * F, D, X, P)
    ref = torch.empty((P, F), dtype=torch.int16, device="cuda")
    fak.fak_swiglu_bf16(Y1, P, F, ref)
    X2 = torch.full((P, F), -1, dtype=torch.int16, device="cuda")
    fak.fak_q4k_gemm_swiglu(W13, F, D, X, P, X2)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    a, b = X2.cpu().numpy(), ref.cpu().numpy()
    assert np.array_equal(a, b), "fused SwiGLU differs from the unfused path in %d of %d" % ((a != b).sum(), a.size)


def silu(g):
    return g / (1.0 + np.exp(-g))


@pytest.mark.parametrize("F,K,P", [(64, 512, 7), (192, 1280, 300), (128, 2048, 513)])
def test_gemm_swiglu_small_vs_oracle(fak, F, K, P):
    # Bar: the GEMM bar per product, d = 5e-3 * sum|w x| + 1e-5 for g and for u, carried through
    # silu(g) * u (|silu'| <= 1.1) plus one bf16 rounding (2^-8 relative) of the result.
    wg = synth.normal(45, F + K, (F, K), 0.02)
    wu = synth.normal(46, F + K, (F, K), 0.02)
    Wg, Wu = oracle.q4k_pack(wg), oracle.q4k_pack(wu)
    Xb = synth.to_bf16(synth.normal(47, F + K + P, (P, K), 1.0))
    W13 = torch.zeros((2 * F, Wg.shape[1]), dtype=torch.uint8, device="cuda")
    fak.fak_q4k_interleave_gate_up(dev(Wg), dev(Wu), F, K, W13)
    X2 = torch.full((P, F), -1, dtype=torch.int16, device="cuda")
    fak.fak_q4k_gemm_swiglu(W13, F, K, dev(Xb.view(np.int16)), P, X2)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    got = bf16_bits_to_f64(X2)
    G, Ag = oracle.gemm_q4k(Wg, F, K, Xb)
    U, Au = oracle.gemm_q4k(Wu, F, K, Xb)
    G, U = G.astype(np.float64), U.astype(np.float64)
    ref = silu(G) * U
    dg, du = 5e-3 * Ag + 1e-5, 5e-3 * Au + 1e-5
    err_in = 1.1 * np.abs(U) * dg + (np.abs(silu(G)) + 1.1 * dg) * du
    bound = err_in + 2.0 ** -8 * (np.abs(ref) + err_in) + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), "swiglu gemm %dx%dx%d: %d of %d outside the bar" % (F, K, P, bad.sum(), bad.size)
    cos = float((got * ref).sum() / np.sqrt((got * got).sum() * (ref * ref).sum()))
    assert cos >= 0.9999, cos


def test_gemm_and_batch_under_graph_capture(fak):
    # while a stream is being captured their scratch comes from cudaMallocAsync (a graph memory
    # node), otherwise from the library's pool: replays equal the eager results bit for bit
    N, K, P, M = 640, 8192, 256, 8  # the GEMM takes a K split here, so it has a workspace
    Wg = dev(fak.fak_q4k_pack(synth.normal(48, 0, (N, K), 0.02)))
    Xb = dev(synth.to_bf16(synth.normal(48, 1, (P, K), 1.0)).view(np.int16))
    Xf = dev(synth.normal(48, 2, (M, K), 1.0))
    Y_e, Yb_e = torch.empty((P, N), device="cuda"), torch.empty((M, N), device="cuda")
    fak.fak_q4k_gemm(Wg, N, K, Xb, P, Y_e)
    fak.fak_q4k_gemv_batch(Wg, N, K, Xf, M, Yb_e)
    torch.cuda.synchronize()
    Y_g, Yb_g = torch.full((P, N), float("nan"), device="cuda"), torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fak.fak_q4k_gemm(Wg, N, K, Xb, P, Y_g)
            fak.fak_q4k_gemv_batch(Wg, N, K, Xf, M, Yb_g)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    assert np.array_equal(Y_g.cpu().numpy().view(np.uint32), Y_e.cpu().numpy().view(np.uint32))
    assert np.array_equal(Yb_g.cpu().numpy().view(np.uint32), Yb_e.cpu().numpy().view(np.uint32))
