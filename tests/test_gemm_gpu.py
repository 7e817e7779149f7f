"""GPU parity of the tcgen05 prefill dequant-GEMM (Y = X W^T, W Q4_K, X bf16,
f32 accumulate) against the oracle, through the C ABI.

Bar: |err| <= 5e-3 * sum|w_i x_i| + 1e-5 per output and cosine >= 0.9999.
Small shapes are compared in full; the prefill workload (fused gate||up
34816x5120 and down 5120x17408, P = 256/512/1024 tokens, seed 2) on sampled
rows x tokens that the oracle computes one by one.
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


# (640, 8192, 256) and (128, 10496, 64) have few tiles: K is split across CTAs (4 splits of 8
# super-blocks; 11 + 11 + 11 + 8) and the partial tiles are summed in split order
@pytest.mark.parametrize("N,K,P", [(128, 256, 1), (128, 256, 7), (256, 512, 256), (384, 1280, 300),
                                   (128, 2048, 513), (512, 5120, 64), (640, 8192, 256), (128, 10496, 64)])
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


@pytest.mark.parametrize("P", [256, 512, 1024])
def test_prefill_workload_sampled(fak, P):
    # fused gate||up 34816 x 5120 (seed 2, tensor 0), down 5120 x 17408 (tensor 1), X (tensor 2)
    D, F = 5120, 17408
    w1 = synth.normal(2, 0, (2 * F, D), 0.02)
    W1g, W1o = fak.fak_q4k_pack(w1), oracle.q4k_pack(w1)
    assert np.array_equal(W1g, W1o)
    del w1
    Xb = synth.to_bf16(synth.normal(2, 2, (P, D), 1.0))
    Y1 = gemm(fak, dev(W1g), 2 * F, D, dev(Xb.view(np.int16)), P)
    rng = np.random.default_rng(P)
    rows = np.sort(rng.choice(2 * F, 48, replace=False))
    rows[0], rows[-1] = 0, 2 * F - 1
    toks = np.unique(np.concatenate([[0, P - 1], rng.choice(P, 6, replace=False)]))
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
    rows2 = np.sort(rng.choice(D, 48, replace=False))
    Yr2, Ar2 = oracle.gemm_q4k_sample(W2o, D, F, X2h, rows2, toks)
    check_gemm(Y2.cpu().numpy()[np.ix_(toks, rows2)], Yr2, Ar2, "prefill down P=%d" % P)
