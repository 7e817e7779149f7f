"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports every
symbol include/fak.h declares, validates arguments before touching the device,
and its packers are bit-exact with the oracle's packers."""
import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fak():
    from q4_weight_quantized_block_gb300 import build
    build.build()
    import q4_weight_quantized_block_gb300 as m
    return m


def test_library_exports_every_declared_symbol(fak):
    hdr = open(os.path.join(ROOT, "include", "fak.h")).read()
    names = set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(fak_\w+)\s*\(", hdr, re.M))
    assert len(names) >= 20
    for n in sorted(names):
        assert hasattr(fak.lib, n), n
    assert "sm_103a" in fak.fak_version()
    assert fak.fak_strerror(5).startswith("bounded")


def test_validation_happens_before_any_device_call(fak):
    lib = fak.lib
    ok_ptr = 1 << 20            # 16-byte aligned, never dereferenced: validation fails first
    assert lib.fak_q4k_gemv(None, 16, 256, ok_ptr, ok_ptr, None) == 1
    assert lib.fak_q4k_gemv(ok_ptr, 16, 100, ok_ptr, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv(ok_ptr, 0, 256, ok_ptr, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv(ok_ptr, 16, fak.FAK_ENGINE_MAX_K + 256, ok_ptr, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv(ok_ptr + 4, 16, 256, ok_ptr, ok_ptr, None) == 3
    assert lib.fak_q4k_gemv(ok_ptr, 16, 256, ok_ptr + 8, ok_ptr, None) == 3
    assert lib.fak_q8_0_gemv(ok_ptr, 16, 288, ok_ptr, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_i8x(ok_ptr, 16, 300, ok_ptr, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_i8x(ok_ptr + 4, 16, 256, ok_ptr, ok_ptr, None) == 3
    assert lib.fak_q4k_gemv_i8x(None, 16, 256, ok_ptr, ok_ptr, None) == 1
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 256, ok_ptr, 65, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 256, ok_ptr, 0, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 256, None, 4, ok_ptr, None) == 1
    assert lib.fak_q4k_gemv_batch(ok_ptr, 0, 256, ok_ptr, 4, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 300, ok_ptr, 4, ok_ptr, None) == 2
    assert lib.fak_q4k_gemv_batch(ok_ptr + 8, 16, 256, ok_ptr, 4, ok_ptr, None) == 3
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 256, ok_ptr + 4, 4, ok_ptr, None) == 3
    assert lib.fak_q4k_gemv_batch(ok_ptr, 16, 256, ok_ptr, 4, ok_ptr + 2, None) == 3
    assert lib.fak_mlp_decode(ok_ptr, ok_ptr, ok_ptr, 256, 512, ok_ptr, 1e-6, ok_ptr, ok_ptr, 16, None) == 2
    assert lib.fak_mlp_decode(ok_ptr, ok_ptr, None, 256, 512, ok_ptr, 1e-6, ok_ptr, ok_ptr, 4096, None) == 1
    assert lib.fak_q4k_gemm(ok_ptr, 0, 256, ok_ptr, 8, ok_ptr, None) == 2
    assert lib.fak_q4k_gemm(ok_ptr, 128, 256, ok_ptr, 0, ok_ptr, None) == 2
    assert lib.fak_q4k_gemm(ok_ptr, 128, 300, ok_ptr, 8, ok_ptr, None) == 2
    assert lib.fak_q4k_gemm(ok_ptr + 8, 128, 256, ok_ptr, 8, ok_ptr, None) == 3
    assert lib.fak_q4k_gemm(None, 128, 256, ok_ptr, 8, ok_ptr, None) == 1
    assert lib.fak_q4k_gemm_swiglu(ok_ptr, 100, 256, ok_ptr, 8, ok_ptr, None) == 2
    assert lib.fak_q4k_gemm_swiglu(ok_ptr, 128, 300, ok_ptr, 8, ok_ptr, None) == 2
    assert lib.fak_q4k_gemm_swiglu(ok_ptr, 128, 256, ok_ptr, 8, ok_ptr + 8, None) == 3
    assert lib.fak_q4k_gemm_swiglu(ok_ptr, 128, 256, ok_ptr, 8, None, None) == 1
    assert lib.fak_q4k_interleave_gate_up(ok_ptr, ok_ptr, 96, 256, ok_ptr, None) == 2
    assert lib.fak_q4k_interleave_gate_up(ok_ptr, ok_ptr, 64, 200, ok_ptr, None) == 2
    assert lib.fak_q4k_interleave_gate_up(ok_ptr, ok_ptr + 4, 64, 256, ok_ptr, None) == 3
    assert lib.fak_q4k_interleave_gate_up(ok_ptr, None, 64, 256, ok_ptr, None) == 1
    assert lib.fak_decode_create(None, None) == 1


def test_packers_reject_bad_shapes(fak):
    with pytest.raises(fak.FakError):
        fak.fak_q4k_pack(np.zeros((2, 100), np.float32))
    with pytest.raises(fak.FakError):
        fak.fak_q8_0_pack(np.zeros((2, 40), np.float32))
    assert fak.fak_mlp_workspace_bytes(17408) >= 17408 * 4 + 256


def _edge_tensor():
    rng = np.random.default_rng(12)
    rows = [
        np.zeros(512), np.full(512, 0.37), np.full(512, -0.37), rng.uniform(0.5, 2, 512), -rng.uniform(0.5, 2, 512),
        rng.normal(0, 1e-7, 512), rng.normal(0, 1e4, 512), rng.standard_t(2, 512) * 0.01,
        np.where(rng.uniform(size=512) < 0.9, 0.0, rng.normal(0, 1, 512)), np.linspace(-1, 1, 512),
        np.concatenate([np.zeros(256), np.full(256, 65000.0)]), np.concatenate([np.full(256, -1e-30), np.ones(256)]),
    ]
    return np.stack(rows).astype(np.float32)


def test_q4k_packer_bit_exact_with_oracle(fak):
    for w in [_edge_tensor(), synth.normal(0, 0, (5120, 5120), 0.02), synth.normal(1, 1, (2048, 5120), 0.02),
              synth.normal(1, 3, (512, 17408), 0.02)]:
        a, b = fak.fak_q4k_pack(w), oracle.q4k_pack(w)
        assert a.shape == b.shape
        diff = np.nonzero(a != b)
        assert diff[0].size == 0, "first mismatch at %s" % (list(zip(*diff))[:3],)


def test_q8_0_packer_bit_exact_with_oracle(fak):
    for w in [_edge_tensor(), synth.normal(3, 900000, (2048, 5120), 0.02)]:
        a, b = fak.fak_q8_0_pack(w), oracle.q8_0_pack(w)
        assert np.array_equal(a, b)


def test_prefill_create_rejects_bad_shapes_before_any_device_call(fak):
    ok_ptr = 1 << 20
    layer = {"kind": fak.FAK_LAYER_GDN, "w_in": ok_ptr, "w_out": ok_ptr, "w_gate": ok_ptr, "w_up": ok_ptr,
             "w_down": ok_ptr}
    good = dict(d_model=256, d_ff=512, vocab=300, gdn_in=640, fa_qg=512, fa_kv=256, n_mix=256)
    bad = [dict(gdn_in=642),     # in_proj rows not a multiple of 4 (the bf16 slice reads float4)
           dict(fa_qg=514),      # q+gate rows not a multiple of 4
           dict(fa_kv=255),      # q+gate, k, v concatenated: the row width must stay a multiple of 4
           dict(n_mix=300),      # out_proj input not whole super-blocks
           dict(d_ff=544),       # d_ff not a multiple of 64 (gate/up interleave)
           dict(d_model=200),    # K not whole super-blocks
           dict(d_model=8448)]   # d_model above the RMSNorm kernel's 8192
    for change in bad:
        args = dict(good, **change)
        with pytest.raises(fak.FakError) as ei:
            fak.PrefillContext(args["d_model"], args["d_ff"], args["vocab"], args["gdn_in"], args["fa_qg"],
                               args["fa_kv"], args["n_mix"], [layer], ok_ptr, ok_ptr, 64)
        assert ei.value.status == 2, change
    for n_tokens in (0, 16385):
        with pytest.raises(fak.FakError) as ei:
            fak.PrefillContext(256, 512, 300, 640, 512, 256, 256, [layer], ok_ptr, ok_ptr, n_tokens)
        assert ei.value.status == 2


def test_decode_create_rejects_unknown_modes_before_any_device_call(fak):
    ok_ptr = 1 << 20
    layer = {"kind": fak.FAK_LAYER_GDN, "w_in": ok_ptr, "w_out": ok_ptr, "w_gate": ok_ptr, "w_up": ok_ptr,
             "w_down": ok_ptr}
    assert fak.FAK_DECODE_PER_MATMUL_HOST_WAIT == 4
    for mode in (-1, 5):
        with pytest.raises(fak.FakError) as ei:
            fak.DecodeContext(256, 512, 300, 640, 512, 256, 256, [layer], ok_ptr, ok_ptr, mode=mode)
        assert ei.value.status == 1, mode
