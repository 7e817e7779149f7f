"""Pins for the oracle's mixer bodies (the Gated DeltaNet step and the gated full-attention
step of the hybrid stack: "Qwen3.6-27B on Apple M3 Pro", model architecture list).  Each
check ties the oracle to something other than itself: a library routine (numpy's
convolution, complex multiplication for the rotary embedding, scipy's logistic function),
an independent formulation of the recurrence (the closed product form of the gated delta
rule), or a special case with a closed form (a zero state, one position, identical keys,
stored associations read back).
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth
from _mixer import small_mixer_model

DK = 128


def silu(x):
    return x * expit(x)


def dims(**kw):
    base = dict(nk=2, nv=6, nq=4, nkv=2)
    base.update(kw)
    return oracle.MixerDims(**base)


def gdn_params(d, conv_w=None, a_log=None, dt_bias=None, norm_w=None):
    rng = np.random.default_rng(0)
    if conv_w is None:
        conv_w = np.tile([0.0, 0.0, 0.0, 1.0], (d.conv_dim, 1))   # the conv passes the new input through
    return oracle.MixerParams(conv_w=conv_w,
                              a_log=np.log(rng.uniform(1, 16, d.nv)) if a_log is None else a_log,
                              dt_bias=rng.normal(0, 1, d.nv) if dt_bias is None else dt_bias,
                              norm_w=np.ones(d.dv) if norm_w is None else norm_w)


def gdn_input(d, q, k, v, z, b, a):
    return np.concatenate([q.ravel(), k.ravel(), v.ravel(), z.ravel(), b.ravel(), a.ravel()])


def fresh_state(d):
    return np.zeros((d.conv_dim, d.conv - 1)), np.zeros((d.nv, d.dk, d.dv))


# ------------------------------------------------------------------ causal conv
def test_causal_conv_equals_numpy_convolution():
    rng = np.random.default_rng(1)
    n, K, T = 5, 4, 12
    w = rng.normal(0, 1, (n, K)).astype(np.float32)
    xs = rng.normal(0, 1, (T, n))
    state = np.zeros((n, K - 1))
    ys = np.array([oracle.causal_conv_step(w, state, xs[t]) for t in range(T)])
    for c in range(n):
        # causal: y[t] = sum_j w[j] x[t - (K-1) + j]  ==  full convolution with the reversed taps
        ref = np.convolve(xs[:, c], w[c, ::-1].astype(np.float64))[:T]
        assert np.allclose(ys[:, c], ref, rtol=1e-13, atol=1e-13)
    assert np.array_equal(state, xs[-(K - 1):].T)       # the state holds the last K-1 inputs, oldest first


# ------------------------------------------------------------------ Gated DeltaNet
def test_gdn_zero_state_is_beta_times_kq_times_v():
    # zero state: S = k (beta v)^T after the write, so o = S^T q = beta (k.q) v, with the key head
    # of value head h being h // (nv / nk); q and k differ per key head, so a wrong mapping shows
    d = dims()
    rng = np.random.default_rng(2)
    q, k = rng.normal(0, 1, (d.nk, DK)), rng.normal(0, 1, (d.nk, DK))
    v = rng.normal(0, 1, (d.nv, DK))
    b = rng.normal(0, 2, d.nv)
    t = gdn_input(d, q, k, v, rng.normal(0, 1, (d.nv, DK)), b, rng.normal(0, 1, d.nv))
    cs, S = fresh_state(d)
    _, raw = oracle.gdn_step(d, gdn_params(d), t, cs, S)
    qn = silu(q) / np.sqrt((silu(q) ** 2).sum(axis=1, keepdims=True) + d.eps) / np.sqrt(DK)
    kn = silu(k) / np.sqrt((silu(k) ** 2).sum(axis=1, keepdims=True) + d.eps)
    for h in range(d.nv):
        kh = h // (d.nv // d.nk)
        want = expit(b[h]) * (kn[kh] @ qn[kh]) * silu(v[h])
        assert np.allclose(raw[h * DK:(h + 1) * DK], want, rtol=1e-12, atol=1e-15), h


def test_gdn_recurrence_equals_product_form():
    # S_T = sum_t [prod_{s>t} alpha_s (I - beta_s k_s k_s^T)] beta_t k_t v_t^T, from a zero state
    d = dims(nk=1, nv=2)
    rng = np.random.default_rng(3)
    p = gdn_params(d)
    cs, S = fresh_state(d)
    T = 6
    ks, vs, qs, betas, alphas = [], [], [], [], []
    for _ in range(T):
        q, k = rng.normal(0, 1, (1, DK)), rng.normal(0, 1, (1, DK))
        v = rng.normal(0, 1, (d.nv, DK))
        b, a = rng.normal(0, 1, d.nv), rng.normal(0, 1, d.nv)
        t = gdn_input(d, q, k, v, rng.normal(0, 1, (d.nv, DK)), b, a)
        _, raw = oracle.gdn_step(d, p, t, cs, S)
        kn = silu(k[0]) / np.sqrt((silu(k[0]) ** 2).sum() + d.eps)
        qn = silu(q[0]) / np.sqrt((silu(q[0]) ** 2).sum() + d.eps) / np.sqrt(DK)
        g = -np.exp(p.arrays["a_log"].astype(np.float64)) * np.logaddexp(0, a + p.arrays["dt_bias"])
        ks.append(kn), qs.append(qn), vs.append(silu(v)), betas.append(expit(b)), alphas.append(np.exp(g))
    for h in range(d.nv):
        ST = np.zeros((DK, DK))
        for t in range(T):
            term = betas[t][h] * np.outer(ks[t], vs[t][h])
            for s in range(t + 1, T):       # A_s = alpha_s (I - beta_s k_s k_s^T) applied on the left
                term = alphas[s][h] * (term - betas[s][h] * np.outer(ks[s], ks[s] @ term))
            ST += term
        # S_0 = 0, so the first step's own decay does not show; each later step's does
        assert np.allclose(S[h], ST, rtol=1e-10, atol=1e-12)
        assert np.allclose(raw[h * DK:(h + 1) * DK], ST.T @ qs[-1], rtol=1e-10, atol=1e-12)


def _onehot_raw(i, big=20.0, small=-40.0):
    x = np.full(DK, small)
    x[i] = big
    return x


def test_gdn_delta_rule_reads_back_stored_values():
    # no decay (a_log -> -inf), beta -> 1, one-hot keys: the state is an exact associative memory
    d = dims(nk=1, nv=1)
    p = gdn_params(d, a_log=np.array([-200.0]), dt_bias=np.array([0.0]))
    cs, S = fresh_state(d)
    rng = np.random.default_rng(4)
    vals = {}
    for slot in (0, 1, 2):
        v = rng.normal(0, 1, (1, DK))
        vals[slot] = silu(v[0])
        t = gdn_input(d, _onehot_raw(7)[None], _onehot_raw(slot)[None], v, np.zeros((1, DK)), np.array([40.0]),
                      np.array([0.0]))
        oracle.gdn_step(d, p, t, cs, S)
    # overwrite slot 1, then read slots 1 and 2 while writing an unrelated slot 9
    v_new = rng.normal(0, 1, (1, DK))
    t = gdn_input(d, _onehot_raw(7)[None], _onehot_raw(1)[None], v_new, np.zeros((1, DK)), np.array([40.0]),
                  np.array([0.0]))
    oracle.gdn_step(d, p, t, cs, S)
    vals[1] = silu(v_new[0])
    for slot in (1, 2):
        t = gdn_input(d, _onehot_raw(slot)[None], _onehot_raw(9)[None], rng.normal(0, 1, (1, DK)),
                      np.zeros((1, DK)), np.array([40.0]), np.array([0.0]))
        _, raw = oracle.gdn_step(d, p, t, cs, S)
        # exact up to the norms' eps: |k|^2 = 400, so each unit key is short by eps / 800 = 1.25e-9
        assert np.allclose(raw * np.sqrt(DK), vals[slot], rtol=1e-8, atol=1e-8), slot


def test_gdn_gated_norm_closed_form():
    # a head whose raw output is a constant c: out = sign(c) * |c| / sqrt(c^2 + eps) * w * silu(z)
    d = dims(nk=1, nv=3)
    rng = np.random.default_rng(5)
    w = rng.uniform(0.5, 1.5, DK).astype(np.float32).astype(np.float64)   # the gains are f32 parameters
    p = gdn_params(d, norm_w=w)
    cs, S = fresh_state(d)
    qk = rng.normal(0, 1, (1, DK))
    v = np.repeat(rng.normal(0, 2, (d.nv, 1)), DK, axis=1)      # constant over each head
    z = rng.normal(0, 1, (d.nv, DK))
    t = gdn_input(d, qk, qk, v, z, rng.normal(0, 1, d.nv), rng.normal(0, 1, d.nv))
    out, raw = oracle.gdn_step(d, p, t, cs, S)
    for h in range(d.nv):
        c = raw[h * DK]
        assert np.allclose(raw[h * DK:(h + 1) * DK], c)
        want = c / np.sqrt(c * c + d.eps) * w * silu(z[h])
        assert np.allclose(out[h * DK:(h + 1) * DK], want, rtol=1e-12, atol=1e-15)


def test_gdn_pure_decay_without_writes():
    # beta -> 0 (b = -60): nothing is written, S only decays by exp(g) per step
    d = dims(nk=1, nv=2)
    p = gdn_params(d)
    rng = np.random.default_rng(6)
    cs, S = fresh_state(d)
    S[:] = rng.normal(0, 1, S.shape)
    S0 = S.copy()
    a = rng.normal(0, 1, d.nv)
    t = gdn_input(d, rng.normal(0, 1, (1, DK)), rng.normal(0, 1, (1, DK)), rng.normal(0, 1, (d.nv, DK)),
                  np.zeros((d.nv, DK)), np.full(d.nv, -60.0), a)
    oracle.gdn_step(d, p, t, cs, S)
    g = -np.exp(p.arrays["a_log"].astype(np.float64)) * np.logaddexp(0, a + p.arrays["dt_bias"])
    for h in range(d.nv):
        assert np.allclose(S[h], np.exp(g[h]) * S0[h], rtol=1e-12, atol=1e-20)


# ------------------------------------------------------------------ gated attention
def attn_params(d, qw=None, kw=None):
    return oracle.MixerParams(q_norm_w=np.ones(d.dh) if qw is None else qw,
                              k_norm_w=np.ones(d.dh) if kw is None else kw)


def test_attention_first_position_is_gated_value():
    d = dims(nq=4, nkv=2)
    rng = np.random.default_rng(7)
    qg = rng.normal(0, 1, d.nq * 2 * d.dh)
    k, v = rng.normal(0, 1, d.nkv * d.dh), rng.normal(0, 1, d.nkv * d.dh)
    kc, vc = np.zeros((d.nkv, 8, d.dh)), np.zeros((d.nkv, 8, d.dh))
    out = oracle.attn_step(d, attn_params(d), qg, k, v, 0, kc, vc)
    for h in range(d.nq):
        g = h // (d.nq // d.nkv)
        gate = qg[h * 2 * d.dh + d.dh:(h + 1) * 2 * d.dh]
        assert np.allclose(out[h * d.dh:(h + 1) * d.dh], v[g * d.dh:(g + 1) * d.dh] * expit(gate), rtol=1e-13)


def test_attention_identical_keys_average_the_values():
    # keys with zeros in the rotary dims are not moved by RoPE: identical keys, uniform weights
    d = dims(nq=2, nkv=1)
    rng = np.random.default_rng(8)
    kc, vc = np.zeros((1, 16, d.dh)), np.zeros((1, 16, d.dh))
    k = rng.normal(0, 1, d.dh)
    k[:d.rot] = 0.0
    vs = []
    for pos in range(5):
        v = rng.normal(0, 1, d.dh)
        vs.append(v)
        qg = rng.normal(0, 1, d.nq * 2 * d.dh)
        out = oracle.attn_step(d, attn_params(d), qg, k, v, pos, kc, vc)
    for h in range(d.nq):
        gate = qg[h * 2 * d.dh + d.dh:(h + 1) * 2 * d.dh]
        assert np.allclose(out[h * d.dh:(h + 1) * d.dh], np.mean(vs, axis=0) * expit(gate), rtol=1e-12)


def test_attention_cached_key_is_normed_and_rotated_as_complex_pairs():
    # RoPE in the rotate-half form is the complex rotation of the pairs (x_i, x_{i+rot/2}) by
    # pos * theta^(-2i/rot); the qk-norm of a +-1 vector divides by sqrt(1 + eps)
    d = dims(nq=2, nkv=1)
    rng = np.random.default_rng(9)
    gain = rng.uniform(0.5, 1.5, d.dh).astype(np.float32).astype(np.float64)   # f32 parameters
    kc, vc = np.zeros((1, 64, d.dh)), np.zeros((1, 64, d.dh))
    for pos in (0, 1, 17, 63):
        k = rng.choice([-1.0, 1.0], d.dh)
        oracle.attn_step(d, attn_params(d, kw=gain), rng.normal(0, 1, d.nq * 2 * d.dh), k, rng.normal(0, 1, d.dh),
                         pos, kc, vc)
        kn = k / np.sqrt(1.0 + d.eps) * gain
        half = d.rot // 2
        z = (kn[:half] + 1j * kn[half:d.rot]) * np.exp(1j * pos * d.theta ** (-2.0 * np.arange(half) / d.rot))
        want = np.concatenate([z.real, z.imag, kn[d.rot:]])
        assert np.allclose(kc[0, pos], want, rtol=1e-12, atol=1e-12), pos


def test_attention_weights_closed_form_with_the_sqrt_dh_scale():
    # keys with no rotary part; key 0 equals the query's pattern, key 1 is orthogonal to it.  After the
    # qk-norm (mean square 0.75) the scores are 256/16 = 16 and 0: weights e^16/(e^16+1), 1/(e^16+1)
    d = dims(nq=1, nkv=1)
    pat = np.concatenate([np.zeros(d.rot), np.ones(96), -np.ones(96)])
    flip = np.concatenate([np.zeros(d.rot), -np.ones(96), -np.ones(96)])
    rng = np.random.default_rng(11)
    v0, v1 = rng.normal(0, 1, d.dh), rng.normal(0, 1, d.dh)
    kc, vc = np.zeros((1, 4, d.dh)), np.zeros((1, 4, d.dh))
    qg = np.concatenate([pat, rng.normal(0, 1, d.dh)])
    oracle.attn_step(d, attn_params(d), qg, pat, v0, 0, kc, vc)
    out = oracle.attn_step(d, attn_params(d), qg, flip, v1, 1, kc, vc)
    r = 0.75 / (0.75 + d.eps)                        # (q.k) / (rms_q rms_k) over the 192 non-zero dims
    s0 = 192 * r / 0.75 / 16.0
    w0 = 1.0 / (1.0 + np.exp(-s0))
    want = (w0 * v0 + (1 - w0) * v1) * expit(qg[d.dh:])
    assert np.allclose(out, want, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ the decode with the mixer bodies
def test_decode_with_mixer_equals_layers_one_by_one():
    m, d, layers, params, lm, emb = small_mixer_model()
    D, F, V = 256, 512, 300
    n_mix = d.nv * d.dv
    dec = oracle.MixerDecoder(m, d, params, max_ctx=8)
    f32 = lambda a: np.asarray(a, np.float64).astype(np.float32)
    conv = {l: np.zeros((d.conv_dim, d.conv - 1)) for l in range(4) if l != 3}
    S = {l: np.zeros((d.nv, d.dk, d.dv)) for l in range(4) if l != 3}
    kc, vc = np.zeros((d.nkv, 8, d.dh)), np.zeros((d.nkv, 8, d.dh))
    tok = 5
    for pos in range(3):
        nxt, logits, la, h_final = dec.decode_token(tok)
        h = emb[tok].astype(np.float64)
        for l, L in enumerate(layers):
            n = f32(oracle.rmsnorm(h))
            if L["kind"] == oracle.LAYER_FA:
                t, _ = oracle.gemv_q4k(L["w_in"], 2 * d.nq * d.dh, D, n)
                k, _ = oracle.gemv_q4k(L["w_k"], d.nkv * d.dh, D, n)
                v, _ = oracle.gemv_q4k(L["w_v"], d.nkv * d.dh, D, n)
                mix = oracle.attn_step(d, params[l], t, k, v, pos, kc, vc)
            else:
                t, _ = oracle.gemv_q4k(L["w_in"], d.gdn_in, D, n)
                mix, _ = oracle.gdn_step(d, params[l], t, conv[l], S[l])
            h = h + oracle.gemv_q4k(L["w_out"], D, n_mix, f32(mix))[0]
            n = f32(oracle.rmsnorm(h))
            g, _ = oracle.gemv_q4k(L["w_gate"], F, D, n)
            u, _ = oracle.gemv_q4k(L["w_up"], F, D, n)
            h = h + oracle.gemv_q4k(L["w_down"], D, F, f32(oracle.swiglu(g, u)))[0]
        assert np.array_equal(h, h_final), pos
        y, a = oracle.gemv_q8_0(lm, V, D, f32(oracle.rmsnorm(h)))
        assert np.array_equal(f32(y), logits) and np.array_equal(a, la)
        assert nxt == int(np.argmax(f32(y)))
        tok = nxt
    dec.close()
