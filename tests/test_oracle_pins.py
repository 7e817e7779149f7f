"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources of truth used here: IEEE 754 binary16 as implemented by numpy's float16
(exhaustive / randomized), the hand transcription of the Q4_K layout in
tests/golden/q4k_layout.txt, exact rational arithmetic (fractions), integer
special cases that reduce to an exact integer GEMV, closed forms for RMSNorm and
SwiGLU, and the pages' byte figure for one decode token (about 15 GB of weights
per token: "Mac Qwen3.6-27B Metal Q4_K perf diagnosis", section 4; a 15.4 GB
q4_k_m file: "Qwen3.6-27B on Apple M3 Pro", section "Can it even run it?").
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "q4k_layout.txt")


def _layout():
    hdr, nib, fld = [], [], {}
    for line in open(GOLDEN):
        t = line.split()
        if not t or t[0].startswith("#"):
            continue
        if t[0] == "hdr":
            hdr.append((int(t[1]), int(t[2]), t[3], int(t[4])))
        elif t[0] == "nib":
            nib.append((int(t[1]), t[2], int(t[3])))
        elif t[0] == "fld":
            fld[t[1]] = (int(t[2]), int(t[3]))
    return hdr, nib, fld


def _f16(h):
    return float(np.array([h], dtype=np.uint16).view(np.float16)[0])


# ------------------------------------------------------------------ binary16
def test_f16_decode_exhaustive_vs_numpy():
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = allh.view(np.float16).astype(np.float32)
    mine = np.array([oracle.f16_decode(int(h)) for h in allh], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(mine[finite], ref[finite])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(np.isinf(mine), np.isinf(ref))


def test_f16_round_up_is_smallest_upper_bound():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.uniform(0, 65504, 2000), np.exp(rng.uniform(np.log(1e-9), np.log(6e4), 6000)),
        rng.uniform(0, 2 ** -14, 1000),                       # subnormal range
        np.array([0.0, 2 ** -24, 2 ** -25, 2 ** -14, 1.0, 65504.0, 1e-30]),
    ]).astype(np.float32)
    for v in vals:
        h = oracle.f16_round_up(v)
        assert _f16(h) >= v, (v, h)
        if h > 0:
            assert _f16(h - 1) < v, (v, h)
    # exactly representable values map to themselves
    for h in list(range(0, 0x7C00, 97)) + [0x3C00, 0x0001, 0x03FF, 0x0400, 0x7BFF]:
        assert oracle.f16_round_up(_f16(h)) == h
    assert oracle.f16_round_up(70000.0) == 0x7BFF       # saturates


def test_f16_rne_vs_numpy():
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.normal(0, 1, 5000), rng.normal(0, 1e-5, 2000), rng.uniform(-65000, 65000, 2000),
        np.exp(rng.uniform(np.log(1e-8), np.log(6e4), 3000)) * rng.choice([-1, 1], 3000),
    ]).astype(np.float32)
    # ties: midpoints between adjacent binary16 values
    hs = np.arange(1, 0x7BFF, 37, dtype=np.uint16)
    lo = hs.view(np.float16).astype(np.float64)
    hi = (hs + 1).view(np.float16).astype(np.float64)
    vals = np.concatenate([vals, ((lo + hi) / 2).astype(np.float32)])
    for v in vals:
        ref = np.float32(v).astype(np.float16).view(np.uint16)
        assert oracle.f16_rne(v) == int(ref), v


def test_bf16_decode():
    for b in [0, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x8000]:
        ref = np.array([b << 16], dtype=np.uint32).view(np.float32)[0]
        assert oracle.bf16_decode(b) == ref


# ------------------------------------------------------------------ Q4_K layout
def _block(d=0x3C00, dmin=0x0000, s=None, qs=None):
    b = np.zeros(144, np.uint8)
    b[0], b[1] = d & 0xFF, d >> 8
    b[2], b[3] = dmin & 0xFF, dmin >> 8
    if s is not None:
        b[4:16] = s
    if qs is not None:
        b[16:144] = qs
    return b


def test_q4k_header_bits_match_transcription():
    hdr, _, _ = _layout()
    assert len(hdr) == 96
    for sidx, bit, field, fbit in hdr:
        s = np.zeros(12, np.uint8)
        s[sidx] = 1 << bit
        _, _, sc, m, _ = oracle.q4k_fields(_block(s=s))
        want_sc, want_m = np.zeros(8, np.uint8), np.zeros(8, np.uint8)
        j = int(field[-1])
        (want_sc if field.startswith("sc") else want_m)[j] = 1 << fbit
        assert np.array_equal(sc, want_sc) and np.array_equal(m, want_m), (sidx, bit, field, fbit)


def test_q4k_nibble_positions_match_transcription():
    _, nib, fld = _layout()
    assert fld["qs"] == (16, 128) and fld["d"] == (0, 2) and fld["dmin"] == (2, 2)
    s = np.zeros(12, np.uint8)
    s[0:4] = 1                      # sc0..3 = 1
    s[8:12] = 1                     # sc4..7 = 1 (low nibble of s[8..11])
    for byte, half, widx in nib:
        qs = np.zeros(128, np.uint8)
        qs[byte] = 0x0F if half == "lo" else 0xF0
        w = oracle.q4k_dequant_block(_block(s=s, qs=qs))
        nz = np.nonzero(w)[0]
        assert list(nz) == [widx] and w[widx] == 15.0, (byte, half, widx, nz)


def test_q4k_value_formula_on_hand_built_block():
    # d = 1, dmin = 0, every sc = 1, m = 0, q_i = i mod 16 -> w_i = i mod 16
    s = np.zeros(12, np.uint8)
    s[0:4] = 1
    s[8:12] = 1
    q = np.arange(256) % 16
    qs = np.zeros(128, np.uint8)
    for g in range(4):
        for l in range(32):
            qs[32 * g + l] = q[64 * g + l] | (q[64 * g + 32 + l] << 4)
    w = oracle.q4k_dequant_block(_block(s=s, qs=qs))
    assert np.array_equal(w, q.astype(np.float32))
    # d = 0.5, dmin = 2, sc_j = j+1, m_j = 7 - j, all q = 3:  w = 0.5*(j+1)*3 - 2*(7-j)
    sc = np.arange(1, 9)
    m = 7 - np.arange(8)
    s = np.zeros(12, np.uint8)
    for j in range(4):
        s[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    w = oracle.q4k_dequant_block(_block(d=0x3800, dmin=0x4000, s=s, qs=np.full(128, 0x33, np.uint8)))
    want = np.repeat(0.5 * sc * 3 - 2.0 * m, 32).astype(np.float32)
    assert np.array_equal(w, want)


def test_q4k_field_roundtrip_every_value_every_slot():
    # the oracle's packer writes fields the transcription reads back
    hdr, _, _ = _layout()
    for j in range(8):
        for v in range(64):
            for which in ("sc", "m"):
                s = np.zeros(12, np.uint8)
                for sidx, bit, field, fbit in hdr:
                    if field == "%s%d" % (which, j) and (v >> fbit) & 1:
                        s[sidx] |= 1 << bit
                _, _, sc, m, _ = oracle.q4k_fields(_block(s=s))
                got = sc if which == "sc" else m
                other = m if which == "sc" else sc
                assert got[j] == v and got.sum() == v and other.sum() == 0


# ------------------------------------------------------------------ quantizer
def _check_roundtrip(x):
    x = np.ascontiguousarray(x, np.float32).reshape(-1, 256)
    for row in x:
        blk = oracle.q4k_quantize_superblock(row)
        dh, mh, sc, m, q = oracle.q4k_fields(blk)
        d, dmin = _f16(dh), _f16(mh)
        w = oracle.q4k_dequant_block(blk)
        assert q.max() <= 15 and sc.max() <= 63 and m.max() <= 63
        for j in range(8):
            sub = row[32 * j: 32 * j + 32].astype(np.float64)
            lo, hi = min(0.0, sub.min()), sub.max()
            bound = 0.5 * d * sc[j] + 2.0 ** -20 * (abs(lo) + abs(hi))
            err = np.abs(sub - w[32 * j: 32 * j + 32].astype(np.float64))
            assert err.max() <= bound, (j, err.max(), bound)
            # order preserved (non-strict)
            order = np.argsort(sub, kind="stable")
            assert np.all(np.diff(q[32 * j: 32 * j + 32][order].astype(int)) >= 0)


def test_q4k_roundtrip_bound_gaussian():
    _check_roundtrip(synth.normal(9, 0, (64, 256), 0.02))


def test_q4k_roundtrip_bound_shapes_of_data():
    rng = np.random.default_rng(3)
    cases = [
        rng.uniform(-1, 1, (8, 256)), rng.uniform(0.5, 2.0, (4, 256)),      # all positive
        -rng.uniform(0.5, 2.0, (4, 256)),                                     # all negative
        rng.standard_t(2, (8, 256)) * 0.01,                                   # heavy tails
        np.full((1, 256), 0.37), np.full((1, 256), -0.37),                    # constants
        rng.normal(0, 1e-6, (4, 256)), rng.normal(0, 1e3, (4, 256)),          # tiny / large scale
        np.where(rng.uniform(size=(4, 256)) < 0.9, 0.0, rng.normal(0, 1, (4, 256))),  # sparse
    ]
    for c in cases:
        _check_roundtrip(c)


def test_q4k_zero_block():
    blk = oracle.q4k_quantize_superblock(np.zeros(256, np.float32))
    assert not blk.any()
    assert not oracle.q4k_dequant_block(blk).any()


# ------------------------------------------------------------------ Q8_0
def test_q8_0_layout_and_roundtrip():
    blk = np.zeros(34, np.uint8)
    blk[0], blk[1] = 0x00, 0x38                       # d = 0.5
    blk[2:34] = (np.arange(32) - 16).astype(np.int8).view(np.uint8)
    assert np.array_equal(oracle.q8_0_dequant_block(blk), 0.5 * (np.arange(32) - 16).astype(np.float32))
    x = synth.normal(9, 1, (16, 320), 0.02)
    W = oracle.q8_0_pack(x)
    assert W.shape == (16, 10 * 34)
    for n in range(16):
        for b in range(10):
            blk = W[n, 34 * b: 34 * b + 34]
            d = _f16(int(blk[0]) | int(blk[1]) << 8)
            q = blk[2:].view(np.int8)
            assert np.abs(q).max() <= 127
            err = np.abs(oracle.q8_0_dequant_block(blk) - x[n, 32 * b: 32 * b + 32])
            assert err.max() <= 0.5 * d * (1 + 2 ** -10)


# ------------------------------------------------------------------ GEMV / GEMM
def _exact_row(blk_bytes, K):
    """Exact rational weights of one row from the transcription, decoded bit by bit."""
    hdr, _, _ = _layout()
    out = []
    for b in range(K // 256):
        blk = blk_bytes[144 * b: 144 * b + 144]
        d = Fraction(_f16(int(blk[0]) | int(blk[1]) << 8))
        dmin = Fraction(_f16(int(blk[2]) | int(blk[3]) << 8))
        fields = {("sc%d" % j): 0 for j in range(8)}
        fields.update({("m%d" % j): 0 for j in range(8)})
        for sidx, bit, field, fbit in hdr:
            if (blk[4 + sidx] >> bit) & 1:
                fields[field] |= 1 << fbit
        w = [None] * 256
        for byte in range(128):
            g, l = divmod(byte, 32)
            for half, shift, base in (("lo", 0, 0), ("hi", 4, 32)):
                i = 64 * g + base + l
                q = (int(blk[16 + byte]) >> shift) & 15
                j = i // 32
                w[i] = d * fields["sc%d" % j] * q - dmin * fields["m%d" % j]
        out += w
    return out


def test_gemv_brute_force_exact_arithmetic():
    rng = np.random.default_rng(4)
    for N, K in [(1, 256), (2, 512), (3, 256)]:
        W = rng.integers(0, 256, (N, K // 256 * 144), dtype=np.uint8)
        for n in range(N):                              # keep d, dmin finite and moderate
            for b in range(K // 256):
                for off in (0, 2):
                    h = int(rng.integers(0x1000, 0x3C00))
                    W[n, 144 * b + off], W[n, 144 * b + off + 1] = h & 0xFF, h >> 8
        x = synth.normal(4, N, (K,), 1.0)
        y, a = oracle.gemv_q4k(W, N, K, x)
        for n in range(N):
            w = _exact_row(W[n], K)
            exact = sum(wi * Fraction(float(xi)) for wi, xi in zip(w, x))
            sabs = sum(abs(wi * Fraction(float(xi))) for wi, xi in zip(w, x))
            # oracle rounds each weight to f32 once (|rel| <= 2^-24 per product), then sums in f64
            assert abs(Fraction(y[n]) - exact) <= sabs * Fraction(1, 2 ** 23), (N, K, n)
            assert abs(a[n] - float(sabs)) <= float(sabs) * 2 ** -20


def test_gemv_integer_special_case_is_exact():
    # d = 1, dmin = 1: w = sc*q - m are integers; x integers -> an exact integer GEMV
    rng = np.random.default_rng(5)
    N, K = 7, 512
    sc = rng.integers(0, 64, (N, K // 32))
    m = rng.integers(0, 64, (N, K // 32))
    q = rng.integers(0, 16, (N, K))
    W = np.zeros((N, K // 256 * 144), np.uint8)
    for n in range(N):
        for b in range(K // 256):
            s = np.zeros(12, np.uint8)
            scb, mb = sc[n, 8 * b: 8 * b + 8], m[n, 8 * b: 8 * b + 8]
            for j in range(4):
                s[j] = scb[j] | ((scb[j + 4] >> 4) << 6)
                s[j + 4] = mb[j] | ((mb[j + 4] >> 4) << 6)
                s[j + 8] = (scb[j + 4] & 15) | ((mb[j + 4] & 15) << 4)
            qq = q[n, 256 * b: 256 * b + 256]
            qs = np.zeros(128, np.uint8)
            for g in range(4):
                qs[32 * g: 32 * g + 32] = qq[64 * g: 64 * g + 32] | (qq[64 * g + 32: 64 * g + 64] << 4)
            W[n, 144 * b: 144 * b + 144] = _block(d=0x3C00, dmin=0x3C00, s=s, qs=qs)
    wint = np.repeat(sc, 32, axis=1) * q - np.repeat(m, 32, axis=1)
    x = rng.integers(-1000, 1000, K)
    y, _ = oracle.gemv_q4k(W, N, K, x.astype(np.float32))
    assert np.array_equal(y, (wint.astype(np.int64) @ x.astype(np.int64)).astype(np.float64))


def test_gemv_batch_equals_single():
    w = synth.normal(6, 0, (96, 512), 0.02)
    W = oracle.q4k_pack(w)
    X = synth.normal(6, 1, (5, 512), 1.0)
    Y, A = oracle.gemv_batch_q4k(W, 96, 512, X)
    for i in range(5):
        y, a = oracle.gemv_q4k(W, 96, 512, X[i])
        assert np.array_equal(Y[i], y) and np.array_equal(A[i], a)


def test_gemm_equals_rows_of_gemv_and_sample():
    w = synth.normal(7, 0, (40, 512), 0.02)
    W = oracle.q4k_pack(w)
    Xb = synth.to_bf16(synth.normal(7, 2, (6, 512), 1.0))
    Y, A = oracle.gemm_q4k(W, 40, 512, Xb)
    xf = (Xb.astype(np.uint32) << 16).view(np.float32)
    for p in range(6):
        y, a = oracle.gemv_q4k(W, 40, 512, xf[p])
        assert np.array_equal(Y[p], y) and np.array_equal(A[p], a)
    rows, toks = np.array([0, 17, 39]), np.array([5, 1])
    Ys, As = oracle.gemm_q4k_sample(W, 40, 512, Xb, rows, toks)
    assert np.array_equal(Ys, Y[np.ix_(toks, rows)]) and np.array_equal(As, A[np.ix_(toks, rows)])


def test_gemv_matches_float64_matmul_of_dequantized():
    w = synth.normal(8, 0, (64, 1024), 0.02)
    W = oracle.q4k_pack(w)
    wd = oracle.q4k_dequant(W, 64, 1024).astype(np.float64)
    x = synth.normal(8, 1, (1024,), 1.0)
    y, a = oracle.gemv_q4k(W, 64, 1024, x)
    ref = wd @ x.astype(np.float64)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(wd).sum(1).max() * np.abs(x).max())
    assert np.allclose(a, np.abs(wd * x.astype(np.float64)).sum(1), rtol=1e-12)
    W8 = oracle.q8_0_pack(w)
    y8, _ = oracle.gemv_q8_0(W8, 64, 1024, x)
    wd8 = np.stack([np.concatenate([oracle.q8_0_dequant_block(W8[n, 34 * b: 34 * b + 34]) for b in range(32)])
                    for n in range(64)]).astype(np.float64)
    assert np.allclose(y8, wd8 @ x.astype(np.float64), rtol=0, atol=1e-12)


# ------------------------------------------------------------------ norms, activation, argmax
def test_rmsnorm_closed_forms():
    for c in (1e-3, 0.7, -5.0, 1e4):
        out = oracle.rmsnorm(np.full(5120, c), eps=0.0)
        assert np.allclose(out, np.sign(c), rtol=1e-15)
    x = synth.normal(10, 0, (5120,), 1.0).astype(np.float64)
    a, b = oracle.rmsnorm(x, 1e-6), oracle.rmsnorm(3.0 * x, 9e-6)
    assert np.allclose(a, b, rtol=1e-14)
    ms = np.mean(x * x)
    assert np.isclose(np.mean(a * a), ms / (ms + 1e-6), rtol=1e-14)


def test_swiglu_closed_forms():
    scipy_special = pytest.importorskip("scipy.special")
    g = np.array([0.0, 40.0, -40.0, 1.0, -2.5, 3.25])
    u = np.array([3.0, 2.0, 5.0, 1.0, 1.0, -2.0])
    out = oracle.swiglu(g, u)
    assert out[0] == 0.0
    assert np.isclose(out[1], 80.0, rtol=1e-15) and abs(out[2]) < 1e-15
    assert np.allclose(out, g * scipy_special.expit(g) * u, rtol=1e-14, atol=0)


def test_argmax_lowest_index_wins_ties():
    v = np.array([1.0, 3.0, np.nan, 3.0, -1.0], np.float32)
    assert oracle.argmax_f32(v) == 1
    assert oracle.argmax_f32(np.array([np.nan, 2.0, 2.0], np.float32)) == 1


# ------------------------------------------------------------------ decode stack
def _tiny_model(seed=11, D=256, F=512, V=300, gdn_in=512, qg=512, kv=256, n_mix=256, n_layers=4):
    layers = []
    for l in range(n_layers):
        fa = l % 4 == 3
        L = {"kind": oracle.LAYER_FA if fa else oracle.LAYER_GDN}
        tid = lambda s: 1000 * l + s
        L["w_in"] = oracle.q4k_pack(synth.normal(seed, tid(0), (qg if fa else gdn_in, D), 0.02))
        L["w_out"] = oracle.q4k_pack(synth.normal(seed, tid(1), (D, n_mix), 0.02))
        if fa:
            L["w_k"] = oracle.q4k_pack(synth.normal(seed, tid(2), (kv, D), 0.02))
            L["w_v"] = oracle.q4k_pack(synth.normal(seed, tid(3), (kv, D), 0.02))
        L["w_gate"] = oracle.q4k_pack(synth.normal(seed, tid(4), (F, D), 0.02))
        L["w_up"] = oracle.q4k_pack(synth.normal(seed, tid(5), (F, D), 0.02))
        L["w_down"] = oracle.q4k_pack(synth.normal(seed, tid(6), (D, F), 0.02))
        layers.append(L)
    lm = oracle.q8_0_pack(synth.normal(seed, 900000, (V, D), 0.02))
    emb = synth.normal(seed, 900001, (V, D), 1.0)
    m = oracle.Model(D, F, V, gdn_in, qg, kv, n_mix, layers, lm, emb)
    return m, layers, lm, emb


def test_decode_stack_equals_layers_one_by_one():
    D, F, V, n_mix, kv = 256, 512, 300, 256, 256
    m, layers, lm, emb = _tiny_model()
    tok = 7
    nxt, logits, la, h_final, kvout = m.decode_token(tok)
    f32 = lambda a: np.asarray(a, np.float64).astype(np.float32)
    h = emb[tok].astype(np.float64)
    kv_ref = []
    for L in layers:
        n = f32(oracle.rmsnorm(h))
        if L["kind"] == oracle.LAYER_FA:
            t, _ = oracle.gemv_q4k(L["w_in"], 512, D, n)
            kv_ref.append(f32(oracle.gemv_q4k(L["w_k"], kv, D, n)[0]))
            kv_ref.append(f32(oracle.gemv_q4k(L["w_v"], kv, D, n)[0]))
        else:
            t, _ = oracle.gemv_q4k(L["w_in"], 512, D, n)
        h = h + oracle.gemv_q4k(L["w_out"], D, n_mix, f32(t[:n_mix]))[0]
        n = f32(oracle.rmsnorm(h))
        g, _ = oracle.gemv_q4k(L["w_gate"], F, D, n)
        u, _ = oracle.gemv_q4k(L["w_up"], F, D, n)
        h = h + oracle.gemv_q4k(L["w_down"], D, F, f32(oracle.swiglu(g, u)))[0]
    assert np.array_equal(h, h_final)
    y, a = oracle.gemv_q8_0(lm, V, D, f32(oracle.rmsnorm(h)))
    assert np.array_equal(f32(y), logits) and np.array_equal(a, la)
    assert nxt == int(np.argmax(f32(y)))
    assert np.array_equal(np.concatenate(kv_ref), kvout)


def test_decode_weight_bytes_match_pages_figure():
    # The 27B hybrid shape: 64 layers (48 GDN + 16 FA, every 4th layer FA), hidden 5120,
    # SwiGLU 17408, vocab 248320 ("Qwen3.6-27B on Apple M3 Pro", architecture list).
    dummy = np.zeros(1, np.uint8)
    layers = [{"kind": oracle.LAYER_FA if l % 4 == 3 else oracle.LAYER_GDN, "w_in": dummy, "w_k": dummy,
               "w_v": dummy, "w_out": dummy, "w_gate": dummy, "w_up": dummy, "w_down": dummy}
              for l in range(64)]
    m = oracle.Model(5120, 17408, 248320, 16480, 12288, 1024, 6144, layers, dummy, np.zeros((1, 1), np.float32))
    b = m.weight_bytes()
    assert b == 15_048_048_640
    assert abs(b - 15e9) / 15e9 < 0.05          # "~15 GB of weights per token"
    assert b < 15.4e9                            # the whole q4_k_m file is 15.4 GB


# ------------------------------------------------------------------ int8 activations
def test_act_i8_hand_cases():
    # sub-block maxima chosen so that 127 / max is a power of two: the products x * (127 / max)
    # are exact and every rounding below, ties to even included, is decided by hand
    x = np.zeros(128, np.float32)
    x[0:9] = [127, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, -1.5, 126.25]        # max 127: scale 1, d = 1
    x[32:37] = [254, 5, 7, -3, 1]                                         # max 254: scale 1/2, d = 2
    x[64:67] = [-63.5, 1.25, 0.75]                                        # max 63.5: scale 2, d = 1/2
    # x[96:128] all zero: d = 0, X = 0
    X, d = oracle.quantize_act_i8(x)
    want = np.zeros(128, np.int8)
    want[0:9] = [127, 2, 4, -2, 0, 0, 2, -2, 126]
    want[32:37] = [127, 2, 4, -2, 0]
    want[64:67] = [-127, 2, 2]
    assert np.array_equal(X, want)
    assert d.tolist() == [1.0, 2.0, 0.5, 0.0]


def test_act_i8_bound_range_and_symmetry():
    rng = np.random.default_rng(40)
    K = 4096
    cases = [rng.normal(0, 1, K), rng.standard_t(1.5, K), rng.normal(0, 1, K) * np.repeat(
        10.0 ** rng.integers(-20, 20, K // 32), 32), np.where(rng.uniform(size=K) < 0.9, 0.0, rng.normal(0, 50, K)),
        np.full(K, -3.0)]
    for x in cases:
        x = x.astype(np.float32)
        X, d = oracle.quantize_act_i8(x)
        assert X.min() >= -127 and X.max() <= 127
        dd = np.repeat(d.astype(np.float64), 32)
        err = np.abs(x.astype(np.float64) - dd * X)
        # half a step, plus the f32 roundings of 127/max and of the product (a few ulps of max|x|)
        am = np.repeat(np.abs(x.reshape(-1, 32)).max(axis=1).astype(np.float64), 32)
        assert np.all(err <= dd / 2 + am * 2.0 ** -21)
        # the largest element of every non-zero sub-block lands on +-127
        xs = x.reshape(-1, 32)
        top = np.abs(xs).argmax(axis=1)
        nz = np.abs(xs).max(axis=1) > 0
        assert np.all(np.abs(X.reshape(-1, 32)[np.arange(xs.shape[0]), top][nz]) == 127)
        Xn, dn = oracle.quantize_act_i8(-x)
        assert np.array_equal(Xn, -X) and np.array_equal(dn, d)


def test_gemv_act_i8_exact_arithmetic():
    rng = np.random.default_rng(41)
    N, K = 3, 512
    W = oracle.q4k_pack(synth.normal(41, 0, (N, K), 0.02))
    x = rng.standard_t(2.0, K).astype(np.float32)
    X, d = oracle.quantize_act_i8(x)
    xq = [Fraction(float(d[k // 32])) * int(X[k]) for k in range(K)]
    y, a = oracle.gemv_q4k_act_i8(W, N, K, x)
    for n in range(N):
        w = _exact_row(W[n], K)
        exact = sum(wi * xi for wi, xi in zip(w, xq))
        sabs = sum(abs(wi * xi) for wi, xi in zip(w, xq))
        assert abs(Fraction(y[n]) - exact) <= sabs * Fraction(1, 2 ** 23)
        assert abs(a[n] - float(sabs)) <= float(sabs) * 2 ** -20


# ------------------------------------------------------------------ bf16 rounding, prefill forward
def test_bf16_rne_is_nearest_with_ties_to_even():
    # hand-decided cases: halfway points go to the even significand
    assert oracle.bf16_rne(1.0) == 0x3F80
    assert oracle.bf16_rne(1.0 + 2.0 ** -8) == 0x3F80            # tie between 0x3F80 (even) and 0x3F81
    assert oracle.bf16_rne(1.0 + 3 * 2.0 ** -8) == 0x3F82        # tie between 0x3F81 and 0x3F82 (even)
    assert oracle.bf16_rne(-(1.0 + 2.0 ** -8 + 2.0 ** -20)) == 0xBF81
    assert oracle.bf16_rne(0.0) == 0 and oracle.bf16_rne(-0.0) == 0x8000
    # random values: no other bfloat16 is closer, and ties pick the even pattern
    rng = np.random.default_rng(30)
    xs = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    for x in xs:
        b = oracle.bf16_rne(x)
        v = oracle.bf16_decode(b)
        err = abs(float(x) - v)
        for nb in (b - 1, b + 1):
            assert err <= abs(float(x) - oracle.bf16_decode(nb & 0xFFFF))
            if err == abs(float(x) - oracle.bf16_decode(nb & 0xFFFF)):
                assert b % 2 == 0


def test_prefill_forward_equals_layers_one_by_one():
    D, F, V, n_mix, kv = 256, 512, 300, 256, 256
    m, layers, lm, emb = _tiny_model()
    toks = np.array([7, 3, 299, 0, 42])
    nxt, logits, la, hf = m.prefill_forward(toks)
    bf = lambda a: synth.to_bf16(np.asarray(a, np.float64).astype(np.float32))
    P = toks.size
    h = emb[toks].astype(np.float64)
    for L in layers:
        n = np.stack([oracle.rmsnorm(h[p]) for p in range(P)])
        t, _ = oracle.gemm_q4k(L["w_in"], 512, D, bf(n))
        h = h + oracle.gemm_q4k(L["w_out"], D, n_mix, bf(t[:, :n_mix]))[0]
        n = np.stack([oracle.rmsnorm(h[p]) for p in range(P)])
        g, _ = oracle.gemm_q4k(L["w_gate"], F, D, bf(n))
        u, _ = oracle.gemm_q4k(L["w_up"], F, D, bf(n))
        a = oracle.swiglu(g.ravel(), u.ravel()).reshape(P, F)
        h = h + oracle.gemm_q4k(L["w_down"], D, F, bf(a))[0]
    assert np.array_equal(h, hf)
    y, ya = oracle.gemv_q8_0(lm, V, D, oracle.rmsnorm(h[-1]).astype(np.float32))
    assert np.array_equal(y.astype(np.float32), logits) and np.array_equal(ya, la)
    assert nxt == int(np.argmax(logits))
