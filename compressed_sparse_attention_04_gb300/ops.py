"""Torch-tensor front end of the C ABI (argument marshalling only).

Each function checks dtype / shape / contiguity / device, then calls the library
entry point of the same name on the current CUDA stream.  bf16 tensors are
``torch.bfloat16``; indices ``torch.int32``; codes and scales ``torch.uint8``.
"""

import ctypes as C

import torch

from . import _lib as L

ENTRY, IDX_H, IDX_D = 512, 32, 128


def _p(t):
    return C.c_void_p(0) if t is None else C.c_void_p(t.data_ptr())


def _stream(dev=None):
    return C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _req(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: must be a contiguous CUDA tensor")


def _ws(nbytes, device):
    if nbytes == 0:
        return None
    return torch.empty(nbytes + 256, dtype=torch.uint8, device=device)


def _ws_ptr(buf):
    if buf is None:
        return C.c_void_p(0)
    p = buf.data_ptr()
    return C.c_void_p((p + 255) // 256 * 256)


def compress(x, w_kv, w_gate, norm_w, m, pos0, kv_cache, kv_pre=None, eps=1e-6, rope_base=10000.0,
             workspace=None):
    """Stage 1 into kv_cache [B, n_cap, 512]; returns kv_pre (f32 [B, T/m, 512])."""
    lib = L.load()
    B, T, hid = x.shape
    G = T // m
    _req(x, torch.bfloat16, (B, T, hid), "x")
    _req(w_kv, torch.bfloat16, (ENTRY, hid), "w_kv")
    if w_gate is not None:
        _req(w_gate, torch.bfloat16, (ENTRY, hid), "w_gate")
    _req(norm_w, torch.float32, (ENTRY,), "norm_w")
    n_cap = kv_cache.shape[1]
    _req(kv_cache, torch.bfloat16, (B, n_cap, ENTRY), "kv_cache")
    if kv_pre is None:
        kv_pre = torch.empty(B, G, ENTRY, dtype=torch.float32, device=x.device)
    _req(kv_pre, torch.float32, (B, G, ENTRY), "kv_pre")
    need = lib.csa2_compress_workspace_size(B, T, hid, m)
    buf = workspace if workspace is not None else _ws(need, x.device)
    L.check(lib.csa2_compress(_p(x), B, T, hid, m, pos0, _p(w_kv), _p(w_gate), _p(norm_w), eps,
                              rope_base, _p(kv_cache), n_cap, _p(kv_pre), _ws_ptr(buf),
                              need, _stream(x.device)), "csa2_compress")
    return kv_pre


def compress_chunk(x, w_kv, w_gate, norm_w, m, pos0, kv_cache, state=None, kv_pre=None, eps=1e-6,
                   rope_base=10000.0, workspace=None):
    """Stage 1 over tokens pos0 .. pos0+T-1 (x bf16 [B, T, hidden]) with the group state
    carried across calls (m == 2: state f32 [B, 1024]).  Writes entries pos0 // m ..
    (pos0 + T) // m - 1; returns kv_pre (f32 [B, that many, 512])."""
    lib = L.load()
    B, T, hid = x.shape
    _req(x, torch.bfloat16, (B, T, hid), "x")
    _req(w_kv, torch.bfloat16, (ENTRY, hid), "w_kv")
    if w_gate is not None:
        _req(w_gate, torch.bfloat16, (ENTRY, hid), "w_gate")
    _req(norm_w, torch.float32, (ENTRY,), "norm_w")
    n_cap = kv_cache.shape[1]
    _req(kv_cache, torch.bfloat16, (B, n_cap, ENTRY), "kv_cache")
    if m == 2:
        if state is None:
            raise ValueError("state: m == 2 needs a float32 [B, 1024] state buffer")
        _req(state, torch.float32, (B, 2 * ENTRY), "state")
    n = (pos0 + T) // m - pos0 // m
    if kv_pre is None:
        kv_pre = torch.empty(B, n, ENTRY, dtype=torch.float32, device=x.device)
    _req(kv_pre, torch.float32, (B, n, ENTRY), "kv_pre")
    need = lib.csa2_compress_workspace_size(B, T, hid, m)
    buf = workspace if workspace is not None else _ws(need, x.device)
    L.check(lib.csa2_compress_chunk(_p(x), B, T, hid, m, pos0, _p(w_kv), _p(w_gate), _p(norm_w),
                                    eps, rope_base, _p(state), _p(kv_cache), n_cap, _p(kv_pre),
                                    _ws_ptr(buf), need, _stream(x.device)),
            "csa2_compress_chunk")
    return kv_pre


def index_k_quant(kv_pre, entry0, m, w_ik, codes, scales, k_out=None, rope_base=10000.0):
    """Stage 2 into codes [B, n_cap, 64] / scales [B, n_cap, 4]."""
    lib = L.load()
    B, G, _ = kv_pre.shape
    _req(kv_pre, torch.float32, (B, G, ENTRY), "kv_pre")
    _req(w_ik, torch.bfloat16, (IDX_D, ENTRY), "w_ik")
    n_cap = codes.shape[1]
    _req(codes, torch.uint8, (B, n_cap, 64), "codes")
    _req(scales, torch.uint8, (B, n_cap, 4), "scales")
    if k_out is not None:
        _req(k_out, torch.float32, (B, G, IDX_D), "k_out")
    L.check(lib.csa2_index_k_quant(_p(kv_pre), B, G, entry0, m, _p(w_ik), rope_base, _p(codes),
                                   _p(scales), n_cap, _p(k_out), _stream(kv_pre.device)),
            "csa2_index_k_quant")


def main_kv_quant_fp4(kv_cache, entry0, G, codes, scales):
    """FP4 main KV: rows entry0 .. entry0+G-1 of kv_cache [B, n_cap, 512] (bf16) into
    codes [B, n_cap, 256] / scales [B, n_cap, 32] (u8)."""
    lib = L.load()
    B, n_cap = kv_cache.shape[:2]
    _req(kv_cache, torch.bfloat16, (B, n_cap, ENTRY), "kv_cache")
    _req(codes, torch.uint8, (B, n_cap, ENTRY // 2), "codes")
    _req(scales, torch.uint8, (B, n_cap, ENTRY // 16), "scales")
    L.check(lib.csa2_main_kv_quant_fp4(_p(kv_cache), B, n_cap, entry0, G, _p(codes), _p(scales),
                                       _stream(kv_cache.device)), "csa2_main_kv_quant_fp4")


def swa_kv_quant_fp8(swa_kv, row0, n_rows, codes, scales):
    """FP8 window KV: rows row0 .. row0+n_rows-1 of swa_kv [B, S, 512] (bf16) into
    codes [B, S, 512] / scales [B, S, 8] (u8)."""
    lib = L.load()
    B, S = swa_kv.shape[:2]
    _req(swa_kv, torch.bfloat16, (B, S, ENTRY), "swa_kv")
    _req(codes, torch.uint8, (B, S, ENTRY), "codes")
    _req(scales, torch.uint8, (B, S, ENTRY // 64), "scales")
    L.check(lib.csa2_swa_kv_quant_fp8(_p(swa_kv), B, S, row0, n_rows, _p(codes), _p(scales),
                                      _stream(swa_kv.device)), "csa2_swa_kv_quant_fp8")


def indexer_score_topk(q_idx, w, q_pos0, codes, scales, n_entries, m, k, cand=None, blk=64,
                       topk_out=None, blockmax_out=None, scores_out=None, workspace=None):
    """Stage 3: returns topk [B, Tq, k] (int32, ascending, -1 padded)."""
    lib = L.load()
    B, Tq = q_idx.shape[:2]
    _req(q_idx, torch.bfloat16, (B, Tq, IDX_H, IDX_D), "q_idx")
    _req(w, torch.float32, (B, Tq, IDX_H), "w")
    n_cap = codes.shape[1]
    _req(codes, torch.uint8, (B, n_cap, 64), "codes")
    _req(scales, torch.uint8, (B, n_cap, 4), "scales")
    nb = 0
    if cand is not None:
        nb = cand.shape[2]
        _req(cand, torch.int32, (B, Tq, nb), "cand")
    if topk_out is None:
        topk_out = torch.empty(B, Tq, k, dtype=torch.int32, device=q_idx.device)
    _req(topk_out, torch.int32, (B, Tq, k), "topk_out")
    if blockmax_out is not None:
        _req(blockmax_out, torch.float32, (B, Tq, -(-n_entries // blk)), "blockmax_out")
    if scores_out is not None:
        row = nb * blk if cand is not None else n_entries
        _req(scores_out, torch.float32, (B, Tq, row), "scores_out")
    need = lib.csa2_indexer_workspace_size(B, Tq, n_entries, nb, blk, int(cand is not None))
    buf = workspace if workspace is not None else _ws(need, q_idx.device)
    L.check(lib.csa2_indexer_score_topk(_p(q_idx), _p(w), B, Tq, q_pos0, _p(codes), _p(scales),
                                        n_cap, n_entries, m, _p(cand), nb, blk, k, _p(topk_out),
                                        _p(blockmax_out), _p(scores_out), _ws_ptr(buf),
                                        need if buf is not None else 0, _stream(q_idx.device)),
            "csa2_indexer_score_topk")
    return topk_out


def hsi_candidates(blockmax, q_pos0, n_entries, m, blk, nb, cand_out=None):
    """Stage 3b: returns candidate block ids [B, Tq, nb] (ascending, -1 padded)."""
    lib = L.load()
    B, Tq, nblk = blockmax.shape
    _req(blockmax, torch.float32, (B, Tq, -(-n_entries // blk)), "blockmax")
    if cand_out is None:
        cand_out = torch.empty(B, Tq, nb, dtype=torch.int32, device=blockmax.device)
    _req(cand_out, torch.int32, (B, Tq, nb), "cand_out")
    L.check(lib.csa2_hsi_candidates(_p(blockmax), B, Tq, q_pos0, n_entries, m, blk, nb,
                                    _p(cand_out), _stream(blockmax.device)), "csa2_hsi_candidates")
    return cand_out


def sparse_attn(q, q_pos0, kv_cache, n_entries, topk, swa_kv, swa_pos0, window=128, sink=None,
                scale=ENTRY ** -0.5, out=None, lse_out=None, kv_fp4=None, swa_fp8=None):
    """Stage 4: returns out bf16 [B, Tq, H, 512].  kv_fp4 = (codes, scales): FP4 main-KV
    entries in place of the bf16 kv_cache; swa_fp8 = (codes, scales): FP8 window rows in
    place of the bf16 swa_kv (which is then None)."""
    lib = L.load()
    B, Tq, H, _ = q.shape
    _req(q, torch.bfloat16, (B, Tq, H, ENTRY), "q")
    k, n_cap = 0, 0
    if topk is not None:
        k = topk.shape[2]
        _req(topk, torch.int32, (B, Tq, k), "topk")
        if kv_fp4 is not None:
            n_cap = kv_fp4[0].shape[1]
            _req(kv_fp4[0], torch.uint8, (B, n_cap, ENTRY // 2), "kv codes")
            _req(kv_fp4[1], torch.uint8, (B, n_cap, ENTRY // 16), "kv scales")
        else:
            n_cap = kv_cache.shape[1]
            _req(kv_cache, torch.bfloat16, (B, n_cap, ENTRY), "kv_cache")
    if swa_fp8 is not None:
        if swa_kv is not None:
            raise ValueError("swa_kv: give the window rows either as bf16 or as FP8, not both")
        S = swa_fp8[0].shape[1]
        _req(swa_fp8[0], torch.uint8, (B, S, ENTRY), "swa codes")
        _req(swa_fp8[1], torch.uint8, (B, S, ENTRY // 64), "swa scales")
    else:
        S = swa_kv.shape[1]
        _req(swa_kv, torch.bfloat16, (B, S, ENTRY), "swa_kv")
    if sink is not None:
        _req(sink, torch.float32, (H,), "sink")
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.bfloat16, (B, Tq, H, ENTRY), "out")
    if lse_out is not None:
        _req(lse_out, torch.float32, (B, Tq, H), "lse_out")
    need = lib.csa2_sparse_attn_workspace_size(B, Tq, H, k, window)
    buf = _ws(need, q.device)
    if swa_fp8 is not None:
        kc, ks = kv_fp4 if kv_fp4 is not None else (None, None)
        L.check(lib.csa2_sparse_attn_ex(_p(q), B, Tq, H, q_pos0,
                                        _p(kv_cache if (k and kv_fp4 is None) else None), _p(kc),
                                        _p(ks), n_cap, n_entries, _p(topk), k, _p(None),
                                        _p(swa_fp8[0]), _p(swa_fp8[1]), S, swa_pos0, window,
                                        _p(sink), scale, _p(out), _p(lse_out), _ws_ptr(buf), need,
                                        _stream(q.device)), "csa2_sparse_attn_ex")
        return out
    if kv_fp4 is not None:
        L.check(lib.csa2_sparse_attn_fp4kv(_p(q), B, Tq, H, q_pos0, _p(kv_fp4[0]), _p(kv_fp4[1]),
                                           n_cap, n_entries, _p(topk), k, _p(swa_kv), S, swa_pos0,
                                           window, _p(sink), scale, _p(out), _p(lse_out),
                                           _ws_ptr(buf), need, _stream(q.device)),
                "csa2_sparse_attn_fp4kv")
        return out
    L.check(lib.csa2_sparse_attn(_p(q), B, Tq, H, q_pos0, _p(kv_cache if k else None), n_cap,
                                 n_entries, _p(topk), k, _p(swa_kv), S, swa_pos0, window, _p(sink),
                                 scale, _p(out), _p(lse_out), _ws_ptr(buf), need,
                                 _stream(q.device)), "csa2_sparse_attn")
    return out


def last_device_status(stream=None):
    lib = L.load()
    s = C.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
    return lib.csa2_last_device_status(s)


class Runner:
    """Full / Reindex / Reuse layer runtime over the C ABI (csa2_runner_*)."""

    def __init__(self, kv_src, idx_src, ratio, hsi_blk=64, hsi_nb=64):
        lib = L.load()
        n = len(kv_src)
        self.n_layers = n
        arr = C.c_int32 * n
        self._h = C.c_void_p()
        L.check(lib.csa2_runner_create(n, arr(*kv_src), arr(*idx_src), arr(*ratio), hsi_blk,
                                       hsi_nb, C.byref(self._h)), "csa2_runner_create")
        self.hsi_blk, self.hsi_nb = hsi_blk, hsi_nb

    def mode(self, layer):
        return L.load().csa2_runner_layer_mode(self._h, layer)

    @staticmethod
    def params(B, Tq, q_pos0, H, hidden, k, window=128, scale=ENTRY ** -0.5, eps=1e-6,
               rope_base=10000.0):
        return L.StepParams(B, Tq, q_pos0, H, hidden, k, window, 0, scale, eps, rope_base, 0.0)

    def workspace_size(self, params, max_x_tokens, max_entries):
        return L.load().csa2_runner_workspace_size(self._h, C.byref(params), max_x_tokens,
                                                   max_entries)

    def step(self, params, ios, workspace, stream=None):
        """ios: sequence of LayerIO (one per layer); workspace: CUDA uint8 tensor."""
        lib = L.load()
        arr = (L.LayerIO * self.n_layers)(*ios)
        s = C.c_void_p(stream if stream is not None else torch.cuda.current_stream().cuda_stream)
        L.check(lib.csa2_runner_step(self._h, C.byref(params), arr, _ws_ptr(workspace),
                                     workspace.numel() - 256 if workspace is not None else 0, s),
                "csa2_runner_step")

    def __del__(self):
        try:
            if self._h:
                L.load().csa2_runner_destroy(self._h)
        except Exception:
            pass


def layer_io(**kw):
    """Build a LayerIO from tensors (None -> NULL) and ints."""
    io = L.LayerIO()
    for name, _ in L.LayerIO._fields_:
        if name not in kw:
            continue
        v = kw[name]
        if isinstance(v, torch.Tensor):
            setattr(io, name, v.data_ptr())
        elif v is None:
            setattr(io, name, None)
        else:
            setattr(io, name, v)
    return io
