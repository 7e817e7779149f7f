"""Seeded synthetic inputs, shared by the oracle side and the GPU side.

Holds no step of the Q4_K method: it only draws numbers (counter-based
SplitMix64 uniforms mapped through Wichura's AS 241 normal quantile, see
synth.c) and converts f32 -> bf16 bits.  Every
element is a pure function of (seed, tensor_id, index), so any slice of a
tensor can be regenerated independently and in parallel.

Tensor ids per workload (row-major [N, K] tensors use index n*K + k):
  single GEMV 5120x5120 (seed 0):   W=0, x=1
  MLP decode (seed 1):              x=0, gate=1, up=2, down=3, batched X=4 ([64,5120])
  prefill GEMM (seed 2):            W1 (gate||up)=0, W2 (down)=1, X=2 ([1024,5120])
  27B-shape decode (seed 3):        1000*layer + slot (GDN in=0, out=1; FA qg=0, o=1,
                                    k=2, v=3; MLP gate=4, up=5, down=6),
                                    lm_head=900000, embedding=900001
  sweep (seed 4):                   W shape i -> i, x shape i -> 100+i, batched X=200
"""
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_SO_CUDA = os.path.join(_HERE, "_build", "libsynth_cuda.so")
_lib_cuda = None


def build(force=False):
    """Compile synth.c into _build/libsynth.so (gcc, OpenMP)."""
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                         ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_f32_to_bf16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64]
        lib.synth_f32_to_bf16.restype = None
        lib.synth_ndtri.argtypes = [ctypes.c_double]
        lib.synth_ndtri.restype = ctypes.c_double
        lib.synth_uniform_f64.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_void_p]
        lib.synth_uniform_f64.restype = None
        lib.synth_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.synth_key.restype = ctypes.c_uint64
        _lib = lib
    return _lib


def normal_into(out, seed, tensor_id, sigma=1.0, start=0):
    """Fill the contiguous float32 array `out` with elements start.. of tensor (seed, tensor_id)."""
    assert out.dtype == np.float32 and out.flags.c_contiguous
    _load().synth_normal_f32(seed, tensor_id, start, out.size, float(sigma), out.ctypes.data)
    return out


def normal(seed, tensor_id, shape, sigma=1.0, start=0):
    """float32 array of `shape` holding sigma * N(0,1) draws of tensor (seed, tensor_id)."""
    out = np.empty(shape, dtype=np.float32)
    return normal_into(out, seed, tensor_id, sigma, start)


def uniforms(seed, tensor_id, n, start=0):
    """The raw uniforms u_start.. behind tensor (seed, tensor_id), float64."""
    out = np.empty(n, dtype=np.float64)
    _load().synth_uniform_f64(seed, tensor_id, start, n, out.ctypes.data)
    return out


def ndtri(p):
    """The generator's normal quantile (AS 241) at one probability p in (0, 1)."""
    return _load().synth_ndtri(float(p))


def to_bf16(a):
    """bfloat16 bit patterns (uint16) of a float32 array, round to nearest even."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().synth_f32_to_bf16(a.ctypes.data, out.ctypes.data, a.size)
    return out


def build_cuda(force=False):
    """Compile synth_cuda.cu (the GPU twin of the generator) into _build/libsynth_cuda.so."""
    src = os.path.join(_HERE, "synth_cuda.cu")
    if force or not os.path.exists(_SO_CUDA) or os.path.getmtime(_SO_CUDA) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO_CUDA), exist_ok=True)
        tmp = _SO_CUDA + ".%d.tmp" % os.getpid()
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        subprocess.check_call([nvcc if os.path.exists(nvcc) else "nvcc", "-gencode",
                               "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false", "-Xcompiler", "-fPIC",
                               "-shared", src, "-o", tmp])
        os.replace(tmp, _SO_CUDA)
    return _SO_CUDA


def normal_device(out, seed, tensor_id, sigma=1.0, start=0, stream=0):
    """Fill a contiguous float32 CUDA tensor with elements start.. of tensor (seed, tensor_id),
    generated on the GPU (same formula as the host; see synth_cuda.cu for the one caveat)."""
    global _lib_cuda
    if _lib_cuda is None:
        lib = ctypes.CDLL(build_cuda())
        lib.synth_normal_f32_device.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                                ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_normal_f32_device.restype = ctypes.c_int
        _lib_cuda = lib
    assert out.is_cuda and out.is_contiguous() and str(out.dtype) == "torch.float32"
    rc = _lib_cuda.synth_normal_f32_device(seed, tensor_id, start, out.numel(), float(sigma), out.data_ptr(), stream)
    if rc != 0:
        raise RuntimeError("synth_normal_f32_device failed: CUDA error %d" % rc)
    return out
