"""GPU parity of the batched Q4_K GEMV (W read once for up to 64 input rows).

Bar: |err| <= 1e-5 * sum|w_i x_i| + 1e-6 per output and cosine >= 0.999999
(the f32-accumulate bar), against the oracle's f64 dot products.  Covers every
input-row bucket edge (1, 2, 8, 9, 16, 17, 32, 33, 64), ragged row tiles,
split-K (few row tiles), one-super-block rows, awkward activations (zero rows,
huge and tiny magnitudes, per-super-block scale jumps), degenerate super-blocks
(all-zero, constant negative), determinism, the gate projection of the MLP
workload at M = 1, 8, 64 sampled by rows, and bit-for-bit repeats of the full gate
shape at M = 2, 8, 16, 64.
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


def run_batch(fak, Wg, N, K, X):
    M = X.shape[0]
    Y = torch.full((M, N), float("nan"), device="cuda")
    fak.fak_q4k_gemv_batch(dev(Wg), N, K, dev(X), M, Y)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    return Y.cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16, 17, 31, 32, 33, 48, 63, 64])
def test_batch_bucket_edges(fak, M):
    N, K = 300, 1024  # three row tiles (last ragged), four super-blocks split across CTAs
    w = synth.normal(40, M, (N, K), 0.02)
    Wg = fak.fak_q4k_pack(w)
    Wo = oracle.q4k_pack(w)
    assert np.array_equal(Wg, Wo)
    X = synth.normal(41, M, (M, K), 1.0)
    Yref, A = oracle.gemv_batch_q4k(Wo, N, K, X)
    check_f32(run_batch(fak, Wg, N, K, X), Yref, A, "batch M=%d" % M)


@pytest.mark.parametrize("N,K,M", [(1, 256, 2), (128, 256, 64), (129, 256, 5), (1000, 5120, 12), (640, 17408, 40),
                                   (4096, 2048, 64), (50, 18432, 7)])
def test_batch_shapes(fak, N, K, M):
    w = synth.normal(42, N + K + M, (N, K), 0.02)
    Wo = oracle.q4k_pack(w)
    X = synth.normal(43, N + K + M, (M, K), 1.0)
    Yref, A = oracle.gemv_batch_q4k(Wo, N, K, X)
    check_f32(run_batch(fak, Wo, N, K, X), Yref, A, "batch %dx%d M=%d" % (N, K, M))


def test_batch_awkward_activations(fak):
    N, K = 200, 2048
    w = synth.normal(44, 0, (N, K), 0.02)
    Wo = oracle.q4k_pack(w)
    rng = np.random.default_rng(44)
    rows = [np.zeros(K), np.ones(K), rng.normal(0, 1, K) * np.repeat(10.0 ** rng.integers(-6, 6, K // 256), 256),
            np.where(rng.uniform(size=K) < 0.95, 0.0, rng.normal(0, 100, K)), rng.standard_t(1.5, K),
            np.concatenate([rng.normal(0, 1e-30, K // 2), rng.normal(0, 1, K // 2)]), rng.normal(0, 1e20, K),
            rng.normal(0, 1e-20, K), np.full(K, -3.0), rng.normal(0, 1, K) * (rng.uniform(size=K) < 0.01)]
    X = np.stack(rows).astype(np.float32)
    Yref, A = oracle.gemv_batch_q4k(Wo, N, K, X)
    check_f32(run_batch(fak, Wo, N, K, X), Yref, A, "awkward rows")


def test_batch_degenerate_superblocks(fak):
    N, K, M = 256, 1536, 6
    w = synth.normal(45, 0, (N, K), 0.02)
    w[0:16] = 0.0  # d = dmin = 0
    w[16:32] = -0.5  # constant negative: d = 0, dmin > 0
    w[32:48, :256] = 7.0  # one constant positive super-block
    w[48:64] = w[48:64] * 1e-4  # tiny weights
    w[64:80, 256:512] = np.linspace(-3, 3, 256, dtype=np.float32)  # wide range
    Wo = oracle.q4k_pack(w)
    X = synth.normal(46, 0, (M, K), 1.0)
    Yref, A = oracle.gemv_batch_q4k(Wo, N, K, X)
    check_f32(run_batch(fak, Wo, N, K, X), Yref, A, "degenerate super-blocks")


def test_batch_rows_equal_single_gemvs_and_determinism(fak):
    N, K, M = 700, 4096, 10
    w = synth.normal(47, 0, (N, K), 0.02)
    Wo = oracle.q4k_pack(w)
    X = synth.normal(48, 0, (M, K), 1.0)
    Y1 = run_batch(fak, Wo, N, K, X)
    Y2 = run_batch(fak, Wo, N, K, X)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32)), "batched GEMV not bitwise deterministic"
    for m in (0, 4, 9):
        y, a = oracle.gemv_q4k(Wo, N, K, X[m])
        check_f32(Y1[m], y, a, "row %d vs single GEMV oracle" % m)


@pytest.fixture(scope="module")
def gate_packed():
    # the MLP workload's gate projection: seed 1, tensor 1, 17408 x 5120
    return oracle.q4k_pack(synth.normal(1, 1, (17408, 5120), 0.02))


@pytest.mark.parametrize("M", [1, 8, 64])
def test_batch_gate_workload_sampled(fak, gate_packed, M):
    # input rows: seed 1, tensor 4; outputs compared on sampled rows (all of the first and last tile)
    N, K = 17408, 5120
    Wo = gate_packed
    X = synth.normal(1, 4, (64, K), 1.0)[:M]
    Y = run_batch(fak, Wo, N, K, X)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N), rng.choice(N, 256, replace=False)]))
    rb = Wo.reshape(N, -1)[rows]
    Yref, A = oracle.gemv_batch_q4k(rb, len(rows), K, X)
    check_f32(Y[:, rows], Yref, A, "gate workload M=%d (sampled rows)" % M)


@pytest.mark.parametrize("M", [2, 8, 16, 64])
def test_batch_gate_workload_repeats_bitwise(fak, M):
    # the full gate shape, repeated: every ring hand-off of the kernel (W tiles, x parts, S records,
    # TMEM buffers) is ordered, so repeated calls agree bit for bit
    N, K = 17408, 5120
    w = torch.empty(N * K, device="cuda")
    synth.normal_device(w, 45, 0, 0.02)
    Wg = torch.empty(N * K // 256 * 144, dtype=torch.uint8, device="cuda")
    fak.fak_q4k_pack_device(w, N, K, Wg)
    del w
    X = torch.empty(M * K, device="cuda")
    synth.normal_device(X, 45, 1, 1.0)
    Ys = []
    for _ in range(6):
        Y = torch.full((M, N), float("nan"), device="cuda")
        fak.fak_q4k_gemv_batch(Wg, N, K, X, M, Y)
        Ys.append(Y)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    assert torch.isfinite(Ys[0]).all()
    for Y in Ys[1:]:
        assert torch.equal(Y.view(torch.int32), Ys[0].view(torch.int32))
