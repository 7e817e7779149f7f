"""GPU checks of the int8-activation variant (the pages' int8-SDOT decode GEMV path,
"Qwen3.6-27B on Apple M3 Pro", reconciliation table): every 32-element sub-block of x
becomes d * X with d = max|x| / 127 and X = rint(x * (127 / max|x|)).

1. The GEMV equals the oracle's GEMV of those quantized activations within the f32 bar
   (1e-5 * sum|w x~| + 1e-6, cosine >= 0.999999): the oracle quantizes x itself
   (oracle.quantize_act_i8, pinned by hand cases and its half-step bound) and dots the
   dequantized weights with d * X in f64, so the integer dot itself is checked exactly.
2. Against the unquantized x the variant is held to a cosine bound only, as on the
   pages (N(0,1) activations: cosine >= 0.9999).
3. The decode step with int8 activations: one launch equals one launch per matmul bit
   for bit, and its logits stay within cosine 0.999 of the exact decode's (4-layer
   full-width stack).
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


def cosine(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float((a * b).sum() / np.sqrt((a * a).sum() * (b * b).sum()))


def gemv_i8x(fak, Wg, N, K, x):
    y = torch.full((N,), float("nan"), device="cuda")
    fak.fak_q4k_gemv_i8x(dev(Wg), N, K, dev(x.astype(np.float32)), y)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("N,K", [(300, 1024), (5120, 5120), (1000, 17408), (129, 1280)])
def test_gemv_i8x_is_the_gemv_of_quantized_x(fak, N, K):
    W = oracle.q4k_pack(synth.normal(50, N + K, (N, K), 0.02))
    x = synth.normal(51, N + K, (K,), 1.0)
    y = gemv_i8x(fak, W, N, K, x)
    yq, aq = oracle.gemv_q4k_act_i8(W, N, K, x)
    check_f32(y, yq, aq, "i8x gemv %dx%d vs quantized x" % (N, K))
    ye, _ = oracle.gemv_q4k(W, N, K, x)
    assert cosine(y, ye) >= 0.9999, cosine(y, ye)


def test_gemv_i8x_awkward_activations(fak):
    N, K = 256, 2048
    W = oracle.q4k_pack(synth.normal(52, 0, (N, K), 0.02))
    rng = np.random.default_rng(52)
    for x in (np.zeros(K), rng.normal(0, 1, K) * np.repeat(10.0 ** rng.integers(-6, 6, K // 32), 32),
              np.where(rng.uniform(size=K) < 0.9, 0.0, rng.normal(0, 50, K)), rng.standard_t(1.5, K),
              np.full(K, -2.5), rng.normal(0, 1e-30, K)):
        x = x.astype(np.float32)
        y = gemv_i8x(fak, W, N, K, x)
        yq, aq = oracle.gemv_q4k_act_i8(W, N, K, x)
        check_f32(y, yq, aq, "i8x awkward activations")


def test_decode_i8x_one_launch_equals_per_matmul_and_tracks_exact(fak):
    import bench
    layers, lm, emb, _ = bench.build_decode_model(fak, torch, 4, 16384, seed=3)
    args = (bench.D, bench.F, 16384, bench.GI, bench.QG, bench.KV, bench.NM, layers, lm, emb)
    exact = fak.DecodeContext(*args, mode=fak.FAK_DECODE_ONE_LAUNCH)
    one = fak.DecodeContext(*args, mode=fak.FAK_DECODE_ONE_LAUNCH_I8X)
    per = fak.DecodeContext(*args, mode=fak.FAK_DECODE_PER_MATMUL_I8X)
    assert one.launches_per_step() == 1 and per.launches_per_step() > 1
    tin = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(3)]
    logs = [torch.empty(16384, device="cuda") for _ in range(3)]
    for t in (0, 11, 16383):
        tin.fill_(t)
        for ctx, o, lg in zip((exact, one, per), outs, logs):
            ctx.step(tin, o, lg)
            assert ctx.status() == 0
        le, lo, lp = (l.cpu().numpy() for l in logs)
        assert np.all(np.isfinite(lo))
        assert np.array_equal(lo.view(np.uint32), lp.view(np.uint32)), "one launch != per matmul (int8) at %d" % t
        assert int(outs[1].item()) == int(np.argmax(lo))
        assert cosine(lo, le) >= 0.999, (t, cosine(lo, le))
    for c in (exact, one, per):
        c.close()
