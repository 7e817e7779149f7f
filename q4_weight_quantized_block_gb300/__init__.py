"""GB300 (sm_103a) Q4_K weight-only dequantize-and-multiply.

A thin ctypes binding over libfak.so (C ABI in include/fak.h).  Functions keep
the C names and only marshal arguments: torch tensors become device pointers,
the stream defaults to torch's current stream, and a non-zero status raises
FakError.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback: if libfak.so is missing, the first use of
any binding raises ImportError (build it with
q4_weight_quantized_block_gb300.build.build()).
"""
import importlib

__all__ = [
    "FAK_DECODE_ONE_LAUNCH", "FAK_DECODE_PER_MATMUL", "FAK_DECODE_ONE_LAUNCH_I8X", "FAK_DECODE_PER_MATMUL_I8X", "FAK_DECODE_PER_MATMUL_HOST_WAIT", "FAK_ENGINE_MAX_K", "FAK_MLP_NOALLOC_MAX_FF", "FAK_LAYER_FA", "FAK_LAYER_GDN",
    "STATUS", "DecodeContext", "PrefillContext", "FakError", "LIB_PATH", "fak_decode_create", "fak_device_status",
    "fak_mlp_decode", "fak_mlp_decode_noalloc", "fak_mlp_workspace_bytes", "fak_q4k_gemm", "fak_q4k_gemm_swiglu",
    "fak_q4k_gemv", "fak_q4k_gemv_batch", "fak_q4k_gemv_i8x", "fak_q4k_interleave_gate_up",
    "fak_q4k_pack", "fak_q4k_pack_device", "fak_q8_0_gemv", "fak_q8_0_pack", "fak_q8_0_pack_device", "fak_strerror", "fak_swiglu_bf16", "fak_version", "lib",
]


def __getattr__(name):
    if name in __all__:
        return getattr(importlib.import_module("._lib", __name__), name)
    raise AttributeError(name)
