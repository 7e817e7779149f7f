"""The allocation-free MLP entry point (fak_mlp_decode_noalloc), for callers
that cannot allocate device memory when they call: its scratch is a static
device array inside the library.  Checked through the C ABI on two calls in a
row with different inputs, at the largest d_ff it accepts: against the oracle's
MLP (RMSNorm, gate / up GEMVs, SwiGLU, down GEMV; f32 bar), against the regular
fak_mlp_decode with a caller-allocated workspace (the same kernel, so equal bit
for bit), and that the second call changes neither the caching allocator's
counters nor the device's free memory.

Kept in a file of its own that pytest collects last."""
import gc

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


def test_noalloc_mlp_matches_oracle_and_workspace_mlp_twice(fak):
    Dm, Ff = 1024, fak.FAK_MLP_NOALLOC_MAX_FF
    mats = {}
    for name, tid, shp in (("gate", 1, (Ff, Dm)), ("up", 2, (Ff, Dm)), ("down", 3, (Dm, Ff))):
        w = synth.normal(61, tid, shp, 0.02)
        o = oracle.q4k_pack(w)
        mats[name] = (o, torch.from_numpy(o).cuda())
    ws = torch.empty(fak.fak_mlp_workspace_bytes(Ff), dtype=torch.uint8, device="cuda")
    for call, xid in enumerate((10, 11)):
        x = synth.normal(61, xid, (Dm,), 1.0)
        xd = torch.from_numpy(x).cuda()
        y_ref = torch.full((Dm,), float("nan"), device="cuda")
        y_new = torch.full((Dm,), float("nan"), device="cuda")
        fak.fak_mlp_decode(mats["gate"][1], mats["up"][1], mats["down"][1], Dm, Ff, xd, 1e-6, y_ref, ws)
        torch.cuda.synchronize()
        gc.collect()  # no collection of earlier tests' objects (and their frees) inside the measured call
        alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
        free0 = torch.cuda.mem_get_info()[0]
        fak.fak_mlp_decode_noalloc(mats["gate"][1], mats["up"][1], mats["down"][1], Dm, Ff, xd, 1e-6, y_new)
        torch.cuda.synchronize()
        if call == 1:  # the first call on the device looks up the array's address; later calls allocate nothing
            assert torch.cuda.memory_allocated() <= alloc0 and torch.cuda.memory_reserved() <= reserved0
            assert torch.cuda.mem_get_info()[0] >= free0
        assert fak.fak_device_status() == 0
        # the oracle's MLP: n = rms(x) (f64), f32 input to each GEMV, SwiGLU in f64, down GEMV
        n = oracle.rmsnorm(x.astype(np.float64)).astype(np.float32)
        g, _ = oracle.gemv_q4k(mats["gate"][0], Ff, Dm, n)
        u, _ = oracle.gemv_q4k(mats["up"][0], Ff, Dm, n)
        y_orc, a = oracle.gemv_q4k(mats["down"][0], Dm, Ff, oracle.swiglu(g, u).astype(np.float32))
        got = y_new.cpu().numpy()
        check_f32(got, y_orc, a, "no-alloc MLP call %d vs the oracle" % call)
        check_f32(got, y_ref.cpu().numpy(), a, "no-alloc MLP call %d vs fak_mlp_decode" % call)
        assert np.array_equal(got.view(np.uint32), y_ref.cpu().numpy().view(np.uint32))


def test_noalloc_mlp_rejects_oversized_d_ff(fak):
    Dm, Ff = 256, fak.FAK_MLP_NOALLOC_MAX_FF + 256
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(Dm, device="cuda")
    y = torch.zeros(Dm, device="cuda")
    with pytest.raises(fak.FakError) as ei:
        fak.fak_mlp_decode_noalloc(dummy, dummy, dummy, Dm, Ff, x, 1e-6, y)
    assert ei.value.status == 2
