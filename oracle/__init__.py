"""The CPU oracle (ctypes binding over oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in __graft_entry__
and bench.py's CPU-baseline / reference leg may import this package.  The
product (q4_weight_quantized_block_gb300) never imports it, and the two share
no code.  Every function is the plain definition: Q4_K / Q8_0 dequantize to
f32, then an f64-accumulated dot in index order (see oracle.h).

Parity pins for each function live in tests/test_oracle_pins.py.
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

Q4K_BLOCK_BYTES = 144
Q8_0_BLOCK_BYTES = 34
LAYER_GDN, LAYER_FA = 0, 1


def build(force=False):
    """Compile oracle.c into _build/liboracle.so (gcc, no FMA contraction, OpenMP over rows)."""
    src = os.path.join(_HERE, "oracle.c")
    hdr = os.path.join(_HERE, "oracle.h")
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr))
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("w_in", ctypes.c_void_p), ("w_k", ctypes.c_void_p),
                ("w_v", ctypes.c_void_p), ("w_out", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p)]


class _MixerDims(ctypes.Structure):
    _fields_ = [("nk", ctypes.c_int64), ("nv", ctypes.c_int64), ("dk", ctypes.c_int64), ("dv", ctypes.c_int64),
                ("conv", ctypes.c_int64), ("nq", ctypes.c_int64), ("nkv", ctypes.c_int64), ("dh", ctypes.c_int64),
                ("rot", ctypes.c_int64), ("theta", ctypes.c_double), ("eps", ctypes.c_double)]


class _MixerParams(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("a_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
                ("norm_w", ctypes.c_void_p), ("q_norm_w", ctypes.c_void_p), ("k_norm_w", ctypes.c_void_p)]


class _Model(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int64), ("d_model", ctypes.c_int64), ("d_ff", ctypes.c_int64),
                ("vocab", ctypes.c_int64), ("gdn_in", ctypes.c_int64), ("fa_qg", ctypes.c_int64),
                ("fa_kv", ctypes.c_int64), ("n_mix", ctypes.c_int64), ("eps", ctypes.c_double),
                ("layers", ctypes.POINTER(_Layer)), ("lm_head", ctypes.c_void_p),
                ("embedding", ctypes.c_void_p)]


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P, I64, U16, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint16, ctypes.c_float
    sig = {
        "orc_f16_decode": ([U16], F), "orc_f16_round_up": ([F], U16), "orc_f16_rne": ([F], U16),
        "orc_bf16_decode": ([U16], F),
        "orc_q4k_quantize_superblock": ([P, P], None), "orc_q4k_pack": ([P, I64, I64, P], ctypes.c_int),
        "orc_q4k_fields": ([P, P, P, P, P, P], None), "orc_q4k_dequant_block": ([P, P], None),
        "orc_q4k_dequant_rows": ([P, I64, I64, P], None),
        "orc_q8_0_quantize_block": ([P, P], None), "orc_q8_0_pack": ([P, I64, I64, P], ctypes.c_int),
        "orc_q8_0_dequant_block": ([P, P], None),
        "orc_gemv_q4k": ([P, I64, I64, P, P, P], None), "orc_gemv_q8_0": ([P, I64, I64, P, P, P], None),
        "orc_gemv_batch_q4k": ([P, I64, I64, P, I64, P, P], None),
        "orc_gemm_q4k": ([P, I64, I64, P, I64, P, P], None),
        "orc_gemm_q4k_sample": ([P, I64, I64, P, I64, P, I64, P, I64, P, P], None),
        "orc_rmsnorm": ([P, I64, ctypes.c_double, P], None), "orc_swiglu": ([P, P, I64, P], None),
        "orc_argmax_f32": ([P, I64], I64),
        "orc_quantize_act_i8": ([P, I64, P, P], None),
        "orc_bf16_rne": ([F], U16),
        "orc_prefill_forward": ([ctypes.POINTER(_Model), P, I64, P, P, P], I64),
        "orc_causal_conv_step": ([P, P, P, I64, I64, P], None),
        "orc_gdn_step": ([ctypes.POINTER(_MixerDims), ctypes.POINTER(_MixerParams), P, P, P, P, P], None),
        "orc_attn_step": ([ctypes.POINTER(_MixerDims), ctypes.POINTER(_MixerParams), P, P, P, I64, I64, P, P, P],
                          None),
        "orc_mixer_state_create": ([ctypes.POINTER(_Model), ctypes.POINTER(_MixerDims), I64], P),
        "orc_mixer_state_destroy": ([P], None),
        "orc_decode_token_mixer": ([ctypes.POINTER(_Model), ctypes.POINTER(_MixerDims),
                                    ctypes.POINTER(_MixerParams), P, I64, P, P, P], I64),
        "orc_gemv_q4k_act_i8": ([P, I64, I64, P, P, P], None),
        "orc_decode_token": ([ctypes.POINTER(_Model), I64, P, P, P, P], I64),
        "orc_decode_weight_bytes": ([ctypes.POINTER(_Model)], I64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


# ---------------------------------------------------------------- f16 / bf16
def f16_decode(h):
    return _load().orc_f16_decode(int(h))


def f16_round_up(v):
    return _load().orc_f16_round_up(float(np.float32(v)))


def f16_rne(v):
    return _load().orc_f16_rne(float(np.float32(v)))


def bf16_decode(b):
    return _load().orc_bf16_decode(int(b))


def bf16_rne(v):
    return int(_load().orc_bf16_rne(float(np.float32(v))))


# ---------------------------------------------------------------- Q4_K / Q8_0
def q4k_pack(w):
    """f32 [N, K] -> uint8 [N, K/256*144] (covering min/max quantizer)."""
    w, pw = _c(w, np.float32)
    N, K = w.shape
    out = np.empty((N, K // 256 * Q4K_BLOCK_BYTES), dtype=np.uint8)
    if _load().orc_q4k_pack(pw, N, K, out.ctypes.data) != 0:
        raise ValueError("K must be a multiple of 256")
    return out


def q4k_quantize_superblock(x256):
    x, px = _c(x256, np.float32)
    assert x.size == 256
    out = np.empty(Q4K_BLOCK_BYTES, dtype=np.uint8)
    _load().orc_q4k_quantize_superblock(px, out.ctypes.data)
    return out


def q4k_fields(blk):
    """(d bits, dmin bits, sc[8], m[8], q[256]) of one 144-byte block."""
    b, pb = _c(blk, np.uint8)
    d = ctypes.c_uint16()
    dm = ctypes.c_uint16()
    sc = np.empty(8, np.uint8)
    m = np.empty(8, np.uint8)
    q = np.empty(256, np.uint8)
    _load().orc_q4k_fields(pb, ctypes.addressof(d), ctypes.addressof(dm), sc.ctypes.data, m.ctypes.data,
                           q.ctypes.data)
    return d.value, dm.value, sc, m, q


def q4k_dequant_block(blk):
    b, pb = _c(blk, np.uint8)
    out = np.empty(256, np.float32)
    _load().orc_q4k_dequant_block(pb, out.ctypes.data)
    return out


def q4k_dequant(W, N, K):
    W, pw = _c(W, np.uint8)
    out = np.empty((N, K), np.float32)
    _load().orc_q4k_dequant_rows(pw, N, K, out.ctypes.data)
    return out


def q8_0_pack(w):
    """f32 [N, K] -> uint8 [N, K/32*34] (absmax quantizer)."""
    w, pw = _c(w, np.float32)
    N, K = w.shape
    out = np.empty((N, K // 32 * Q8_0_BLOCK_BYTES), dtype=np.uint8)
    if _load().orc_q8_0_pack(pw, N, K, out.ctypes.data) != 0:
        raise ValueError("K must be a multiple of 32")
    return out


def q8_0_dequant_block(blk):
    b, pb = _c(blk, np.uint8)
    out = np.empty(32, np.float32)
    _load().orc_q8_0_dequant_block(pb, out.ctypes.data)
    return out


# ---------------------------------------------------------------- matmuls
def gemv_q4k(W, N, K, x):
    """(y f64 [N], a f64 [N]) with a = sum_k |w*x|."""
    W, pw = _c(W, np.uint8)
    x, px = _c(x, np.float32)
    y = np.empty(N, np.float64)
    a = np.empty(N, np.float64)
    _load().orc_gemv_q4k(pw, N, K, px, y.ctypes.data, a.ctypes.data)
    return y, a


def gemv_q8_0(W, N, K, x):
    W, pw = _c(W, np.uint8)
    x, px = _c(x, np.float32)
    y = np.empty(N, np.float64)
    a = np.empty(N, np.float64)
    _load().orc_gemv_q8_0(pw, N, K, px, y.ctypes.data, a.ctypes.data)
    return y, a


def gemv_batch_q4k(W, N, K, X):
    W, pw = _c(W, np.uint8)
    X, px = _c(X, np.float32)
    M = X.shape[0]
    Y = np.empty((M, N), np.float64)
    A = np.empty((M, N), np.float64)
    _load().orc_gemv_batch_q4k(pw, N, K, px, M, Y.ctypes.data, A.ctypes.data)
    return Y, A


def gemm_q4k(W, N, K, Xbf16):
    """Y[p, n] = sum_k What[n,k] * bf16(X[p,k]); X given as bf16 bit patterns (uint16 [P, K])."""
    W, pw = _c(W, np.uint8)
    X, px = _c(Xbf16, np.uint16)
    P = X.shape[0]
    Y = np.empty((P, N), np.float64)
    A = np.empty((P, N), np.float64)
    _load().orc_gemm_q4k(pw, N, K, px, P, Y.ctypes.data, A.ctypes.data)
    return Y, A


def gemm_q4k_sample(W, N, K, Xbf16, rows, toks):
    """Y[i, j] for token toks[i] and weight row rows[j] only."""
    W, pw = _c(W, np.uint8)
    X, px = _c(Xbf16, np.uint16)
    rows, pr = _c(rows, np.int64)
    toks, pt = _c(toks, np.int64)
    Y = np.empty((toks.size, rows.size), np.float64)
    A = np.empty((toks.size, rows.size), np.float64)
    _load().orc_gemm_q4k_sample(pw, N, K, px, X.shape[0], pr, rows.size, pt, toks.size,
                                Y.ctypes.data, A.ctypes.data)
    return Y, A


def rmsnorm(x, eps=1e-6):
    x, px = _c(x, np.float64)
    out = np.empty_like(x)
    _load().orc_rmsnorm(px, x.size, float(eps), out.ctypes.data)
    return out


def swiglu(g, u):
    g, pg = _c(g, np.float64)
    u, pu = _c(u, np.float64)
    out = np.empty_like(g)
    _load().orc_swiglu(pg, pu, g.size, out.ctypes.data)
    return out


def argmax_f32(v):
    v, pv = _c(v, np.float32)
    return int(_load().orc_argmax_f32(pv, v.size))


# ---------------------------------------------------------------- int8 activations
def quantize_act_i8(x):
    """(X int8 [n], d f32 [n/32]): per 32-element sub-block d = max|x| / 127 and
    X = clamp(rint(x * (127 / max|x|)), -127, 127), in f32 (see oracle.h)."""
    x, px = _c(x, np.float32)
    assert x.size % 32 == 0
    X = np.empty(x.size, np.int8)
    d = np.empty(x.size // 32, np.float32)
    _load().orc_quantize_act_i8(px, x.size, X.ctypes.data, d.ctypes.data)
    return X, d


def gemv_q4k_act_i8(W, N, K, x):
    """(y, a) of the GEMV of the int8 activations of x: sum_k What[n,k] * d_j * X_k in f64."""
    W, pw = _c(W, np.uint8)
    x, px = _c(x, np.float32)
    y = np.empty(N, np.float64)
    a = np.empty(N, np.float64)
    _load().orc_gemv_q4k_act_i8(pw, N, K, px, y.ctypes.data, a.ctypes.data)
    return y, a


# ---------------------------------------------------------------- decode stack
class Model:
    """A hybrid decode stack held as packed numpy byte arrays (kept alive here).

    layers: list of dicts with keys kind (LAYER_GDN / LAYER_FA) and w_in, w_k, w_v,
    w_out, w_gate, w_up, w_down (uint8 arrays; w_k / w_v only for FA layers).
    """

    def __init__(self, d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, layers, lm_head, embedding,
                 eps=1e-6):
        self._keep = [lm_head, embedding] + [v for L in layers for v in L.values() if isinstance(v, np.ndarray)]
        self._layers = (_Layer * len(layers))()
        for i, L in enumerate(layers):
            cl = self._layers[i]
            cl.kind = L["kind"]
            for key in ("w_in", "w_k", "w_v", "w_out", "w_gate", "w_up", "w_down"):
                arr = L.get(key)
                setattr(cl, key, arr.ctypes.data if arr is not None else None)
        emb = np.ascontiguousarray(embedding, dtype=np.float32)
        self._keep.append(emb)
        self.c = _Model(len(layers), d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, float(eps),
                        self._layers, lm_head.ctypes.data, emb.ctypes.data)
        self.d_model, self.vocab, self.fa_kv = d_model, vocab, fa_kv
        self.n_fa = sum(1 for L in layers if L["kind"] == LAYER_FA)

    def decode_token(self, tok):
        """(next token, logits f32, logit_abs f64, final hidden f64, kv f32)."""
        h = np.empty(self.d_model, np.float64)
        logits = np.empty(self.vocab, np.float32)
        la = np.empty(self.vocab, np.float64)
        kv = np.empty(max(1, 2 * self.n_fa * self.fa_kv), np.float32)
        nxt = _load().orc_decode_token(ctypes.byref(self.c), int(tok), h.ctypes.data, logits.ctypes.data,
                                       la.ctypes.data, kv.ctypes.data)
        return int(nxt), logits, la, h, kv[: 2 * self.n_fa * self.fa_kv]

    def weight_bytes(self):
        return int(_load().orc_decode_weight_bytes(ctypes.byref(self.c)))

    def prefill_forward(self, toks):
        """The projections-only prefill of tokens `toks` (bf16 GEMM operands): (next token, logits of the
        last token f32, logit_abs f64, final hidden states f64 [P, d_model])."""
        toks, pt = _c(toks, np.int64)
        P = toks.size
        h = np.empty((P, self.d_model), np.float64)
        logits = np.empty(self.vocab, np.float32)
        la = np.empty(self.vocab, np.float64)
        nxt = _load().orc_prefill_forward(ctypes.byref(self.c), pt, P, h.ctypes.data, logits.ctypes.data,
                                          la.ctypes.data)
        return int(nxt), logits, la, h


# ---------------------------------------------------------------- mixer bodies
class MixerDims:
    """Head counts and sizes of the two mixer bodies (defaults: the 27B shape)."""

    def __init__(self, nk=16, nv=48, dk=128, dv=128, conv=4, nq=24, nkv=4, dh=256, rot=64, theta=1e7, eps=1e-6):
        self.nk, self.nv, self.dk, self.dv, self.conv = nk, nv, dk, dv, conv
        self.nq, self.nkv, self.dh, self.rot, self.theta, self.eps = nq, nkv, dh, rot, theta, eps
        self.c = _MixerDims(nk, nv, dk, dv, conv, nq, nkv, dh, rot, float(theta), float(eps))

    @property
    def conv_dim(self):
        return 2 * self.nk * self.dk + self.nv * self.dv

    @property
    def gdn_in(self):
        return self.conv_dim + self.nv * self.dv + 2 * self.nv


class MixerParams:
    """One layer's mixer parameters (f32 numpy arrays, kept alive here)."""

    def __init__(self, conv_w=None, a_log=None, dt_bias=None, norm_w=None, q_norm_w=None, k_norm_w=None):
        self.arrays = {}
        vals = {}
        for name, arr in (("conv_w", conv_w), ("a_log", a_log), ("dt_bias", dt_bias), ("norm_w", norm_w),
                          ("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
            if arr is not None:
                arr = np.ascontiguousarray(arr, dtype=np.float32)
                self.arrays[name] = arr
                vals[name] = arr.ctypes.data
            else:
                vals[name] = None
        self.c = _MixerParams(**vals)


def causal_conv_step(w, state, x):
    """y = one step of the depthwise causal conv (w [n, K] f32, state [n, K-1] f64 updated in place)."""
    w, pw = _c(w, np.float32)
    x, px = _c(x, np.float64)
    assert state.dtype == np.float64 and state.flags.c_contiguous
    n, K = w.shape
    y = np.empty(n, np.float64)
    _load().orc_causal_conv_step(pw, state.ctypes.data, px, n, K, y.ctypes.data)
    return y


def gdn_step(dims, params, t, conv_state, S):
    """One Gated DeltaNet step on f64 arrays; conv_state [conv_dim, conv-1] and S [nv, dk, dv] are
    updated in place.  Returns (out [nv*dv], o_raw [nv*dv] before the gated norm)."""
    t, pt = _c(t, np.float64)
    assert conv_state.dtype == np.float64 and conv_state.flags.c_contiguous
    assert S.dtype == np.float64 and S.flags.c_contiguous
    out = np.empty(dims.nv * dims.dv, np.float64)
    raw = np.empty(dims.nv * dims.dv, np.float64)
    _load().orc_gdn_step(ctypes.byref(dims.c), ctypes.byref(params.c), pt, conv_state.ctypes.data, S.ctypes.data,
                         out.ctypes.data, raw.ctypes.data)
    return out, raw


def attn_step(dims, params, qg, k, v, pos, kc, vc):
    """One gated attention step at position pos; kc, vc [nkv, max_ctx, dh] f64 updated in place."""
    qg, pq = _c(qg, np.float64)
    k, pk = _c(k, np.float64)
    v, pv = _c(v, np.float64)
    assert kc.dtype == np.float64 and kc.flags.c_contiguous and vc.shape == kc.shape
    out = np.empty(dims.nq * dims.dh, np.float64)
    _load().orc_attn_step(ctypes.byref(dims.c), ctypes.byref(params.c), pq, pk, pv, int(pos), kc.shape[1],
                          kc.ctypes.data, vc.ctypes.data, out.ctypes.data)
    return out


class MixerDecoder:
    """A decode that runs the mixer bodies: a Model, its MixerDims, one MixerParams per layer, and the
    recurrent state (conv states, S, KV caches, position) owned by the oracle."""

    def __init__(self, model, dims, params, max_ctx=256):
        self.model, self.dims, self.params = model, dims, params
        self._mp = (_MixerParams * len(params))()
        for i, p in enumerate(params):
            self._mp[i] = p.c
        self._st = _load().orc_mixer_state_create(ctypes.byref(model.c), ctypes.byref(dims.c), int(max_ctx))

    def decode_token(self, tok):
        """(next token, logits f32, logit_abs f64, final hidden f64); the state advances one token."""
        m = self.model
        h = np.empty(m.d_model, np.float64)
        logits = np.empty(m.vocab, np.float32)
        la = np.empty(m.vocab, np.float64)
        nxt = _load().orc_decode_token_mixer(ctypes.byref(m.c), ctypes.byref(self.dims.c), self._mp, self._st,
                                             int(tok), h.ctypes.data, logits.ctypes.data, la.ctypes.data)
        return int(nxt), logits, la, h

    def close(self):
        if self._st:
            _load().orc_mixer_state_destroy(self._st)
            self._st = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
