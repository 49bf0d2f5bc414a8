"""Device twin of the generator (libcsa2_synth.so), filling torch CUDA tensors."""

import ctypes as C
import os

import torch

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa2_synth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(_PATH):
            raise RuntimeError(f"{_PATH} missing: run `python -m compressed_sparse_attention_04_gb300.build`")
        lib = C.CDLL(_PATH)
        u64, u32, vp, f32 = C.c_uint64, C.c_uint32, C.c_void_p, C.c_float
        lib.synth_normal_bf16.argtypes = [vp, u64, u64, u32, u32, f32, vp]
        lib.synth_normal_f32.argtypes = [vp, u64, u64, u32, u32, f32, vp]
        lib.synth_u32.argtypes = [vp, u64, u64, u32, u32, vp]
        for f in (lib.synth_normal_bf16, lib.synth_normal_f32, lib.synth_u32):
            f.restype = C.c_int
        _lib = lib
    return _lib


def _s(t):
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def fill_normal(t, seed, stream, start=0, sigma=1.0):
    """Fill a contiguous bf16 or float32 CUDA tensor with elements start.. of (seed, stream)."""
    assert t.is_cuda and t.is_contiguous()
    lib = _load()
    if t.dtype == torch.bfloat16:
        rc = lib.synth_normal_bf16(t.data_ptr(), t.numel(), start, seed, stream, sigma, _s(t))
    elif t.dtype == torch.float32:
        rc = lib.synth_normal_f32(t.data_ptr(), t.numel(), start, seed, stream, sigma, _s(t))
    else:
        raise TypeError(t.dtype)
    if rc != 0:
        raise RuntimeError(f"synth kernel launch failed: cudaError {rc}")
    return t


def fill_u32(t, seed, stream, start=0):
    assert t.is_cuda and t.is_contiguous() and t.dtype == torch.int32
    rc = _load().synth_u32(t.data_ptr(), t.numel(), start, seed, stream, _s(t))
    if rc != 0:
        raise RuntimeError(f"synth kernel launch failed: cudaError {rc}")
    return t
