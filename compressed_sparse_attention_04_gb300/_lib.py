"""ctypes declarations of libcsa2.so (the C ABI in include/csa2.h).

Argument marshalling only: every step of the hot path runs in the library's CUDA
kernels.  Loading fails loudly when the library has not been built.
"""

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_CHECK = range(7)
MODE_SWA, MODE_FULL, MODE_REINDEX, MODE_REUSE = range(4)
STAGES = 6   # compress, index_k, scores, top-k, HSI, attention

vp, i32, f32, sz = C.c_void_p, C.c_int, C.c_float, C.c_size_t
u32 = C.c_uint


class LayerIO(C.Structure):
    """Mirror of csa2_layer_io."""
    _fields_ = [
        ("x", vp), ("w_kv", vp), ("w_gate", vp), ("norm_w", vp), ("w_ik", vp),
        ("kv_cache", vp), ("idx_codes", vp), ("idx_scales", vp),
        ("q_idx", vp), ("w_idx", vp),
        ("q", vp), ("swa_kv", vp), ("sink", vp), ("out", vp),
        ("topk_out", vp), ("cand_out", vp),
        ("kv_codes", vp), ("kv_scales", vp), ("swa_codes", vp), ("swa_scales", vp),
        ("compress_state", vp),
        ("x_tokens", i32), ("x_pos0", i32), ("n_cap", i32), ("swa_len", i32),
        ("swa_pos0", i32), ("reserved0", i32),
    ]


class StepParams(C.Structure):
    """Mirror of csa2_step_params."""
    _fields_ = [
        ("B", i32), ("Tq", i32), ("q_pos0", i32), ("H", i32), ("hidden", i32), ("k", i32),
        ("window", i32), ("reserved0", i32), ("scale", f32), ("eps", f32), ("rope_base", f32),
        ("reserved1", f32),
    ]


# name -> (restype, argtypes); every symbol include/csa2.h declares
SIGNATURES = {
    "csa2_status_str": (C.c_char_p, [i32]),
    "csa2_last_error_message": (C.c_char_p, []),
    "csa2_version": (C.c_char_p, []),
    "csa2_kernel_launches": (C.c_ulonglong, []),
    "csa2_last_device_status": (i32, [vp]),
    "csa2_compress_workspace_size": (sz, [i32, i32, i32, i32]),
    "csa2_compress": (i32, [vp, i32, i32, i32, i32, i32, vp, vp, vp, f32, f32, vp, i32, vp,
                            vp, sz, vp]),
    "csa2_compress_chunk": (i32, [vp, i32, i32, i32, i32, i32, vp, vp, vp, f32, f32, vp, vp, i32,
                                  vp, vp, sz, vp]),
    "csa2_index_k_quant": (i32, [vp, i32, i32, i32, i32, vp, f32, vp, vp, i32, vp, vp]),
    "csa2_main_kv_quant_fp4": (i32, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "csa2_swa_kv_quant_fp8": (i32, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "csa2_indexer_workspace_size": (sz, [i32, i32, i32, i32, i32, i32]),
    "csa2_indexer_score_topk": (i32, [vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, vp, i32,
                                      i32, i32, vp, vp, vp, vp, sz, vp]),
    "csa2_indexer_score_topk_bounded": (i32, [vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, i32,
                                              vp, vp, sz, u32, i32, vp]),
    "csa2_indexer_noalloc_max_scratch_bytes": (sz, []),
    "csa2_indexer_score_topk_noalloc": (i32, [vp, vp, i32, i32, i32, vp, vp, i32, i32, i32, vp,
                                              i32, i32, i32, vp, vp, vp]),
    "csa2_hsi_candidates": (i32, [vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]),
    "csa2_sparse_attn_workspace_size": (sz, [i32, i32, i32, i32, i32]),
    "csa2_sparse_attn": (i32, [vp, i32, i32, i32, i32, vp, i32, i32, vp, i32, vp, i32, i32,
                               i32, vp, f32, vp, vp, vp, sz, vp]),
    "csa2_sparse_attn_fp4kv": (i32, [vp, i32, i32, i32, i32, vp, vp, i32, i32, vp, i32, vp, i32,
                                     i32, i32, vp, f32, vp, vp, vp, sz, vp]),
    "csa2_sparse_attn_ex": (i32, [vp, i32, i32, i32, i32, vp, vp, vp, i32, i32, vp, i32, vp, vp,
                                  vp, i32, i32, i32, vp, f32, vp, vp, vp, sz, vp]),
    "csa2_runner_create": (i32, [i32, vp, vp, vp, i32, i32, C.POINTER(vp)]),
    "csa2_runner_destroy": (None, [vp]),
    "csa2_runner_layer_mode": (i32, [vp, i32]),
    "csa2_runner_workspace_size": (sz, [vp, C.POINTER(StepParams), i32, i32]),
    "csa2_runner_set_timing": (i32, [vp, vp, i32]),
    "csa2_runner_step": (i32, [vp, C.POINTER(StepParams), C.POINTER(LayerIO), vp, sz, vp]),
}

_lib = None


def load():
    """Load libcsa2.so once; raises if it is missing (no fallback path exists)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m compressed_sparse_attention_04_gb300.build`")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


class CSA2Error(RuntimeError):
    def __init__(self, status, where):
        lib = load()
        self.status = status
        msg = lib.csa2_last_error_message().decode()
        super().__init__(f"{where}: {lib.csa2_status_str(status).decode()}: {msg}")


def check(status, where):
    if status != OK:
        raise CSA2Error(status, where)
