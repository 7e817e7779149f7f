"""GPU parity of the matrix-vector engine in its "rows" work split.

The engine cuts a GEMV into (4-row group, 8-block slab) units.  When one CTA's
share of the rows holds more than 200 units, every warp of the grid takes its
own contiguous range of rows instead ("rows" mode); smaller GEMVs deal a CTA's
units to its warps ("split" mode).  At K = 5120 (3 slabs per row) rows mode
starts near 40k rows, so the lm_head-sized Q4_K GEMV of the pages' decode
("Mac Qwen3.6-27B Metal Q4_K perf diagnosis", section 2: lm_head and the
per-projection GEMVs) and the large shapes of the GEMV sweep run there.

Each case checks, through the C ABI, every output row of fak_q4k_gemv and of
fak_q4k_gemv_i8x against the oracle (f32 bar: |err| <= 1e-5 * sum|w x| + 1e-6,
cosine >= 0.999999; the int8 variant against the oracle's GEMV of the int8
activations), after asserting from the work-split arithmetic that every CTA
of the launch really takes the rows branch.  The weights the GPU reads are the
oracle packer's bytes, generated on the host.

Shapes: 248320 x 5120 (the sweep's largest shape), 41041 x 5120 (ragged: warp
ranges of 22-23 rows leave partial last groups), 20000 x 17408 (68 blocks per
row: a last slab of four blocks, taken by half-warps, inside rows mode).
"""
import numpy as np
import pytest

import oracle
import synth
from _util import check_f32

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

WARPS_PER_CTA = 12      # consumer warps of one engine CTA
ROWS_PER_GROUP = 4
SLAB_BLOCKS = 8
MAX_SPLIT_UNITS = 200


@pytest.fixture(scope="module")
def fak():
    from q4_weight_quantized_block_gb300 import build
    build.build()
    import q4_weight_quantized_block_gb300 as m
    assert torch.cuda.is_available()
    return m


def warp_windows(N, K, sms):
    """The engine's work split of an N x K Q4_K GEMV on `sms` CTAs: asserts rows mode on every CTA and
    returns the row window [lo, hi) of every warp of the grid."""
    grid = min((N + ROWS_PER_GROUP - 1) // ROWS_PER_GROUP, sms)
    nslab = (K // 256 + SLAB_BLOCKS - 1) // SLAB_BLOCKS
    for c in range(grid):
        r0, r1 = N * c // grid, N * (c + 1) // grid
        units = (r1 - r0 + ROWS_PER_GROUP - 1) // ROWS_PER_GROUP * nslab
        assert units > MAX_SPLIT_UNITS, "CTA %d of %dx%d would take the split branch" % (c, N, K)
    gw = grid * WARPS_PER_CTA
    lo = [N * w // gw for w in range(gw)]
    return np.array(lo), np.array(lo[1:] + [N])


def host_weights(seed, tid, N, K, chunk_rows=16384):
    """Oracle-packed Q4_K bytes of W ~ N(0, 0.02^2) [N, K], generated on the host in row chunks."""
    out = np.empty((N, K // 256 * 144), np.uint8)
    for r0 in range(0, N, chunk_rows):
        nr = min(chunk_rows, N - r0)
        out[r0:r0 + nr] = oracle.q4k_pack(synth.normal(seed, tid, (nr, K), 0.02, start=r0 * K))
    return out


@pytest.mark.parametrize("N,K,tid", [(248320, 5120, 4), (41041, 5120, 7), (20000, 17408, 8)])
def test_gemv_rows_mode_every_row(fak, N, K, tid):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lo, hi = warp_windows(N, K, sms)
    assert np.any((hi - lo) % ROWS_PER_GROUP != 0)  # some warp windows end in a partial group
    W = host_weights(4, tid, N, K)
    x = synth.normal(4, 100 + tid, (K,), 1.0)
    Wd = torch.from_numpy(W).cuda()
    xd = torch.from_numpy(x).cuda()
    y = torch.full((N,), float("nan"), device="cuda")
    yq = torch.full((N,), float("nan"), device="cuda")
    fak.fak_q4k_gemv(Wd, N, K, xd, y)
    fak.fak_q4k_gemv_i8x(Wd, N, K, xd, yq)
    torch.cuda.synchronize()
    assert fak.fak_device_status() == 0
    yref, a = oracle.gemv_q4k(W, N, K, x)
    got = y.cpu().numpy()
    check_f32(got, yref, a, "rows-mode gemv %dx%d" % (N, K))
    # the edges of every warp window, named explicitly (a failure there points at the split)
    edges = np.unique(np.concatenate([lo, hi - 1]))
    check_f32(got[edges], yref[edges], a[edges], "rows-mode gemv %dx%d, warp window edges" % (N, K))
    yref8, a8 = oracle.gemv_q4k_act_i8(W, N, K, x)
    check_f32(yq.cpu().numpy(), yref8, a8, "rows-mode int8-activation gemv %dx%d" % (N, K))
