"""ctypes binding over libfak.so: argument marshalling only (see include/fak.h)."""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfak.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("libfak.so not built: run q4_weight_quantized_block_gb300.build.build() "
                      "(nvcc, sm_103a); there is no fallback implementation")

lib = ctypes.CDLL(LIB_PATH)

STATUS = {0: "FAK_OK", 1: "FAK_ERR_INVALID_ARG", 2: "FAK_ERR_SHAPE", 3: "FAK_ERR_ALIGN", 4: "FAK_ERR_CUDA",
          5: "FAK_ERR_TIMEOUT", 6: "FAK_ERR_NOMEM", 7: "FAK_ERR_DEVICE", 8: "FAK_ERR_UNSUPPORTED"}
FAK_ENGINE_MAX_K = 18432
FAK_MLP_NOALLOC_MAX_FF = 18432
FAK_LAYER_GDN, FAK_LAYER_FA = 0, 1
FAK_DECODE_ONE_LAUNCH, FAK_DECODE_PER_MATMUL, FAK_DECODE_ONE_LAUNCH_I8X, FAK_DECODE_PER_MATMUL_I8X = 0, 1, 2, 3
FAK_DECODE_PER_MATMUL_HOST_WAIT = 4

P, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t


class FakError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%s)" % (where, STATUS.get(status, status), fak_strerror(status)))


class LayerDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("w_in", P), ("w_k", P), ("w_v", P), ("w_out", P), ("w_gate", P),
                ("w_up", P), ("w_down", P)]


class MixerLayer(ctypes.Structure):
    _fields_ = [("conv_w", P), ("a_log", P), ("dt_bias", P), ("norm_w", P), ("q_norm_w", P), ("k_norm_w", P)]


class MixerDesc(ctypes.Structure):
    _fields_ = [("gdn_nk", ctypes.c_int32), ("gdn_nv", ctypes.c_int32), ("gdn_dk", ctypes.c_int32),
                ("gdn_dv", ctypes.c_int32), ("fa_nq", ctypes.c_int32), ("fa_nkv", ctypes.c_int32),
                ("fa_dh", ctypes.c_int32), ("fa_rot", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("eps", ctypes.c_float), ("max_ctx", ctypes.c_int32), ("layers", ctypes.POINTER(MixerLayer))]


class DecodeDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("gdn_in", ctypes.c_int32), ("fa_qg", ctypes.c_int32),
                ("fa_kv", ctypes.c_int32), ("n_mix", ctypes.c_int32), ("eps", ctypes.c_float),
                ("mode", ctypes.c_int32), ("layers", ctypes.POINTER(LayerDesc)), ("lm_head", P),
                ("embedding", P), ("mixer", ctypes.POINTER(MixerDesc))]


_SIGS = {
    "fak_strerror": ([I32], ctypes.c_char_p),
    "fak_version": ([], ctypes.c_char_p),
    "fak_q4k_pack": ([P, I64, I64, P, SZ], I32),
    "fak_q8_0_pack": ([P, I64, I64, P, SZ], I32),
    "fak_q4k_pack_device": ([P, I64, I64, P, SZ, P], I32),
    "fak_q8_0_pack_device": ([P, I64, I64, P, SZ, P], I32),
    "fak_q4k_gemv": ([P, I64, I64, P, P, P], I32),
    "fak_q4k_gemv_i8x": ([P, I64, I64, P, P, P], I32),
    "fak_q8_0_gemv": ([P, I64, I64, P, P, P], I32),
    "fak_q4k_gemv_batch": ([P, I64, I64, P, I32, P, P], I32),
    "fak_mlp_workspace_bytes": ([I64], SZ),
    "fak_mlp_decode": ([P, P, P, I64, I64, P, ctypes.c_float, P, P, SZ, P], I32),
    "fak_mlp_decode_noalloc": ([P, P, P, I64, I64, P, ctypes.c_float, P, P], I32),
    "fak_q4k_gemm": ([P, I64, I64, P, I64, P, P], I32),
    "fak_swiglu_bf16": ([P, I64, I64, P, P], I32),
    "fak_q4k_gemm_swiglu": ([P, I64, I64, P, I64, P, P], I32),
    "fak_q4k_interleave_gate_up": ([P, P, I64, I64, P, P], I32),
    "fak_decode_create": ([ctypes.POINTER(DecodeDesc), ctypes.POINTER(P)], I32),
    "fak_decode_step": ([P, P, P, P, P], I32),
    "fak_decode_status": ([P, P], I32),
    "fak_decode_read_state": ([P, I32, P, SZ, P], I32),
    "fak_decode_reset": ([P, P], I32),
    "fak_decode_launches_per_step": ([P], I32),
    "fak_decode_set_timeout_ns": ([P, I64], I32),
    "fak_decode_debug_unreachable_wait": ([P, I32], I32),
    "fak_decode_destroy": ([P], None),
    "fak_device_status": ([P], I32),
    "fak_prefill_create": ([ctypes.POINTER(DecodeDesc), I64, ctypes.POINTER(P)], I32),
    "fak_prefill_run": ([P, P, P, P, P], I32),
    "fak_prefill_read_hidden": ([P, P, SZ, P], I32),
    "fak_prefill_kernels": ([P], I32),
    "fak_prefill_status": ([P, P], I32),
    "fak_prefill_destroy": ([P], None),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


def fak_strerror(status):
    return lib.fak_strerror(int(status)).decode()


def fak_version():
    return lib.fak_version().decode()


def _check(status, where):
    if status != 0:
        raise FakError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ host packers
def fak_q4k_pack(w):
    """Host f32 [N, K] -> uint8 [N, K/256*144] Q4_K bytes."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.empty((N, K // 256 * 144), dtype=np.uint8)
    _check(lib.fak_q4k_pack(w.ctypes.data, N, K, out.ctypes.data, out.nbytes), "fak_q4k_pack")
    return out


def fak_q8_0_pack(w):
    """Host f32 [N, K] -> uint8 [N, K/32*34] Q8_0 bytes."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    out = np.empty((N, K // 32 * 34), dtype=np.uint8)
    _check(lib.fak_q8_0_pack(w.ctypes.data, N, K, out.ctypes.data, out.nbytes), "fak_q8_0_pack")
    return out


def fak_q4k_pack_device(w, N, K, out, stream=None):
    """Device f32 [N, K] (tensor or pointer) -> device Q4_K bytes `out` (N*(K/256)*144 bytes)."""
    nbytes = N * (K // 256) * 144
    _check(lib.fak_q4k_pack_device(_ptr(w), N, K, _ptr(out), nbytes, _stream(stream)), "fak_q4k_pack_device")


def fak_q8_0_pack_device(w, N, K, out, stream=None):
    """Device f32 [N, K] -> device Q8_0 bytes `out` (N*(K/32)*34 bytes)."""
    nbytes = N * (K // 32) * 34
    _check(lib.fak_q8_0_pack_device(_ptr(w), N, K, _ptr(out), nbytes, _stream(stream)), "fak_q8_0_pack_device")


# ------------------------------------------------------------------ device calls
def fak_q4k_gemv(Wq, N, K, x, y, stream=None):
    _check(lib.fak_q4k_gemv(_ptr(Wq), N, K, _ptr(x), _ptr(y), _stream(stream)), "fak_q4k_gemv")


def fak_q4k_gemv_i8x(Wq, N, K, x, y, stream=None):
    """fak_q4k_gemv on int8 activations (one scale per 32-element sub-block of x)."""
    _check(lib.fak_q4k_gemv_i8x(_ptr(Wq), N, K, _ptr(x), _ptr(y), _stream(stream)), "fak_q4k_gemv_i8x")


def fak_q8_0_gemv(Wq, N, K, x, y, stream=None):
    _check(lib.fak_q8_0_gemv(_ptr(Wq), N, K, _ptr(x), _ptr(y), _stream(stream)), "fak_q8_0_gemv")


def fak_q4k_gemv_batch(Wq, N, K, X, M, Y, stream=None):
    _check(lib.fak_q4k_gemv_batch(_ptr(Wq), N, K, _ptr(X), M, _ptr(Y), _stream(stream)), "fak_q4k_gemv_batch")


def fak_mlp_workspace_bytes(d_ff):
    return int(lib.fak_mlp_workspace_bytes(d_ff))


def fak_mlp_decode(Wgate, Wup, Wdown, d_model, d_ff, x, eps, y, workspace, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.fak_mlp_decode(_ptr(Wgate), _ptr(Wup), _ptr(Wdown), d_model, d_ff, _ptr(x), float(eps), _ptr(y),
                              _ptr(workspace), workspace_bytes, _stream(stream)), "fak_mlp_decode")


def fak_mlp_decode_noalloc(Wgate, Wup, Wdown, d_model, d_ff, x, eps, y, stream=None):
    """fak_mlp_decode with the library's own static scratch (no allocation; calls must not overlap)."""
    _check(lib.fak_mlp_decode_noalloc(_ptr(Wgate), _ptr(Wup), _ptr(Wdown), d_model, d_ff, _ptr(x), float(eps),
                                      _ptr(y), _stream(stream)), "fak_mlp_decode_noalloc")


def fak_q4k_gemm(Wq, N, K, X, P_, Y, stream=None):
    _check(lib.fak_q4k_gemm(_ptr(Wq), N, K, _ptr(X), P_, _ptr(Y), _stream(stream)), "fak_q4k_gemm")


def fak_swiglu_bf16(Y1, P_, half, X2, stream=None):
    _check(lib.fak_swiglu_bf16(_ptr(Y1), P_, half, _ptr(X2), _stream(stream)), "fak_swiglu_bf16")


def fak_q4k_gemm_swiglu(W13, F, K, X, P_, X2, stream=None):
    _check(lib.fak_q4k_gemm_swiglu(_ptr(W13), F, K, _ptr(X), P_, _ptr(X2), _stream(stream)), "fak_q4k_gemm_swiglu")


def fak_q4k_interleave_gate_up(Wg, Wu, F, K, W13, stream=None):
    _check(lib.fak_q4k_interleave_gate_up(_ptr(Wg), _ptr(Wu), F, K, _ptr(W13), _stream(stream)),
           "fak_q4k_interleave_gate_up")


def fak_device_status(stream=None):
    return int(lib.fak_device_status(_stream(stream)))


# ------------------------------------------------------------------ decode context
class DecodeContext:
    """Owns a fak_decode context.  `layers` is a list of dicts with keys kind, w_in,
    w_k, w_v, w_out, w_gate, w_up, w_down (device tensors or pointers)."""

    def __init__(self, d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, layers, lm_head, embedding,
                 eps=1e-6, mode=FAK_DECODE_ONE_LAUNCH, mixer=None):
        """mixer: None (projections only), or a dict with the head counts gdn_nk, gdn_nv, fa_nq, fa_nkv,
        fa_rot, rope_theta, eps, max_ctx and `layers`: one dict per layer with the device tensors
        conv_w, a_log, dt_bias, norm_w (GDN layers) or q_norm_w, k_norm_w (FA layers)."""
        self._keep = (layers, lm_head, embedding, mixer)
        arr = (LayerDesc * max(1, len(layers)))()
        for i, L in enumerate(layers):
            arr[i].kind = L["kind"]
            for key in ("w_in", "w_k", "w_v", "w_out", "w_gate", "w_up", "w_down"):
                setattr(arr[i], key, _ptr(L.get(key)))
        self._arr = arr
        mptr = None
        if mixer is not None:
            ml = (MixerLayer * max(1, len(layers)))()
            for i, M in enumerate(mixer["layers"]):
                for key in ("conv_w", "a_log", "dt_bias", "norm_w", "q_norm_w", "k_norm_w"):
                    setattr(ml[i], key, _ptr(M.get(key)))
            self._ml = ml
            self._md = MixerDesc(mixer["gdn_nk"], mixer["gdn_nv"], 128, 128, mixer["fa_nq"], mixer["fa_nkv"], 256,
                                 mixer["fa_rot"], float(mixer["rope_theta"]), float(mixer["eps"]), mixer["max_ctx"],
                                 ctypes.cast(ml, ctypes.POINTER(MixerLayer)))
            mptr = ctypes.pointer(self._md)
        desc = DecodeDesc(len(layers), d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, float(eps), mode,
                          ctypes.cast(arr, ctypes.POINTER(LayerDesc)), _ptr(lm_head), _ptr(embedding), mptr)
        h = P()
        _check(lib.fak_decode_create(ctypes.byref(desc), ctypes.byref(h)), "fak_decode_create")
        self.handle = h
        self.d_model, self.vocab, self.fa_kv = d_model, vocab, fa_kv
        self.n_fa = sum(1 for L in layers if L["kind"] == FAK_LAYER_FA)

    def step(self, tok_in, tok_out, logits=None, stream=None):
        _check(lib.fak_decode_step(self.handle, _ptr(tok_in), _ptr(tok_out), _ptr(logits), _stream(stream)),
               "fak_decode_step")

    def status(self, stream=None):
        return int(lib.fak_decode_status(self.handle, _stream(stream)))

    def reset(self, stream=None):
        """Start a new sequence: clear the mixer state (conv states, S, KV cache, position)."""
        _check(lib.fak_decode_reset(self.handle, _stream(stream)), "fak_decode_reset")

    def read_state(self, which, dst, stream=None):
        """which 0: hidden state [d_model]; 1: FA k/v projections [n_fa][2][fa_kv]; 2: the last
        layer's mixer output [n_mix]."""
        count = dst.numel() if hasattr(dst, "numel") else dst.size
        _check(lib.fak_decode_read_state(self.handle, int(which), _ptr(dst), count, _stream(stream)),
               "fak_decode_read_state")

    def launches_per_step(self):
        return int(lib.fak_decode_launches_per_step(self.handle))

    def set_timeout_ns(self, ns):
        _check(lib.fak_decode_set_timeout_ns(self.handle, int(ns)), "fak_decode_set_timeout_ns")

    def debug_unreachable_wait(self, op_index):
        _check(lib.fak_decode_debug_unreachable_wait(self.handle, int(op_index)), "fak_decode_debug_unreachable_wait")

    def close(self):
        if self.handle:
            lib.fak_decode_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fak_decode_create(*args, **kw):
    return DecodeContext(*args, **kw)


# ------------------------------------------------------------------ prefill forward
class PrefillContext:
    """Owns a fak_prefill context: the projections-only prefill forward of P tokens as one CUDA graph.
    Same model arguments as DecodeContext (no mixer)."""

    def __init__(self, d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, layers, lm_head, embedding, n_tokens,
                 eps=1e-6):
        self._keep = (layers, lm_head, embedding)
        arr = (LayerDesc * max(1, len(layers)))()
        for i, L in enumerate(layers):
            arr[i].kind = L["kind"]
            for key in ("w_in", "w_k", "w_v", "w_out", "w_gate", "w_up", "w_down"):
                setattr(arr[i], key, _ptr(L.get(key)))
        self._arr = arr
        desc = DecodeDesc(len(layers), d_model, d_ff, vocab, gdn_in, fa_qg, fa_kv, n_mix, float(eps), 0,
                          ctypes.cast(arr, ctypes.POINTER(LayerDesc)), _ptr(lm_head), _ptr(embedding), None)
        h = P()
        _check(lib.fak_prefill_create(ctypes.byref(desc), int(n_tokens), ctypes.byref(h)), "fak_prefill_create")
        self.handle = h
        self.P, self.d_model, self.vocab = int(n_tokens), d_model, vocab

    def run(self, tokens, tok_out, logits=None, stream=None):
        _check(lib.fak_prefill_run(self.handle, _ptr(tokens), _ptr(tok_out), _ptr(logits), _stream(stream)),
               "fak_prefill_run")

    def read_hidden(self, dst, stream=None):
        count = dst.numel() if hasattr(dst, "numel") else dst.size
        _check(lib.fak_prefill_read_hidden(self.handle, _ptr(dst), count, _stream(stream)), "fak_prefill_read_hidden")

    def kernels(self):
        return int(lib.fak_prefill_kernels(self.handle))

    def status(self, stream=None):
        return int(lib.fak_prefill_status(self.handle, _stream(stream)))

    def close(self):
        if self.handle:
            lib.fak_prefill_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
