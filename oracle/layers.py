"""Full / Reindex / Reuse layer runtime -- oracle side (test infrastructure only).

[P1 §一层全局注意力算四样东西], [P1 §共享池里有四样东西], [P2 §CSA2], [P4 §Les trois modes]:
a global-attention layer computes main KV, indexer K, top-k indices and the
attention itself; the first three may come from an earlier layer.  Whether a
layer makes its own main KV (is_kv_source) and whether it makes its own
indices (is_index_source) are static config, given as two source-id tables.
Sharing goes through one object with four slots (compress_kv, index_k,
topk_idxs, candidates) that the latest writer overwrites.
"""

import numpy as np

from . import csa2_ref as R

SWA, FULL, REINDEX, REUSE = "swa", "full", "reindex", "reuse"


def layer_modes(kv_src, idx_src):
    """Classify layers from kv_source_layer_ids / index_source_layer_ids.

    -1 = no global branch (sliding window only).  Full: own KV and own index.
    Reindex: shared KV, own index.  Reuse: shared KV and shared index.  Own KV
    with a foreign index is rejected: indices address one particular KV
    [P1 §一层全局注意力算四样东西].  Raises ValueError on an invalid table.
    """
    n = len(kv_src)
    if len(idx_src) != n:
        raise ValueError("table lengths differ")
    modes = []
    for l in range(n):
        f, r = int(kv_src[l]), int(idx_src[l])
        if f == -1:
            if r != -1:
                raise ValueError(f"layer {l}: index source without a KV source")
            modes.append(SWA)
        elif f == l:
            if r != l:
                raise ValueError(f"layer {l}: own KV with a foreign index")
            modes.append(FULL)
        elif 0 <= f < l and modes[f] == FULL:
            if r == l:
                modes.append(REINDEX)
            elif 0 <= r < l and modes[r] in (FULL, REINDEX) and int(kv_src[r]) == f:
                modes.append(REUSE)
            else:
                raise ValueError(f"layer {l}: index source {r} invalid for KV source {f}")
        else:
            raise ValueError(f"layer {l}: KV source {f} is not an earlier Full layer")
    return modes


def v41_flash_tables():
    """The 40-layer pattern of DeepSeek-V4.1-Flash.

    [P1 §40 层只有 4 个 Full], [P2 §CED], [P4 §Mode Full / Mode Reindex]: layers
    0-1 sliding window only; encoder groups of six layers led by Full layers 2,
    8 and 14 (m = 2); decoder Full layer 20 (m = 1, built from H20); Reindex at
    24, 28, 32, 36; every other layer reuses the newest index source of its KV.
    Returns (kv_src, idx_src, ratio) lists of length 40 (ratio 0 = no entries).
    """
    kv_src, idx_src, ratio = [], [], []
    full_enc, full_dec, reindex = (2, 8, 14), (20,), (24, 28, 32, 36)
    cur_kv, cur_idx = -1, -1
    for l in range(40):
        if l < 2:
            kv_src.append(-1); idx_src.append(-1); ratio.append(0)
            continue
        if l in full_enc or l in full_dec:
            cur_kv, cur_idx = l, l
            ratio.append(2 if l in full_enc else 1)
        elif l in reindex:
            cur_idx = l
            ratio.append(0)
        else:
            ratio.append(0)
        kv_src.append(cur_kv); idx_src.append(cur_idx)
    return kv_src, idx_src, ratio


def entries_per_token(kv_src, idx_src, ratio):
    """Global-KV entries stored per token: each Full layer stores 1/m entries."""
    modes = layer_modes(kv_src, idx_src)
    return sum(1.0 / ratio[l] for l, md in enumerate(modes) if md == FULL)


def bytes_per_token(kv_src, idx_src, ratio, entry_bytes=356):
    """Global-KV bytes per token for a given entry size (356 B = 288 + 68 in FP4)."""
    return entry_bytes * entries_per_token(kv_src, idx_src, ratio)


def run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k, hsi_blk=64, hsi_nb=64,
             window=R.WINDOW, scale=R.ATTN_SCALE, use_hsi=True, main_kv_fp4=False, swa_fp8=False):
    """One pass of all layers for Tq queries per sequence at positions q_pos0..

    ``layers[l]`` is a dict of float64 inputs:
      all:      q [B,Tq,H,512], swa [B,S,512], swa_pos0
      Full:     x [B,Tx,hidden] (tokens x_pos0..), x_pos0, w_kv, w_gate (None if m=1),
                gamma, w_ik, prev_kv [B,n0,512] (bf16-valued), prev_codes [B,n0,64],
                prev_scales [B,n0,4] with n0 = x_pos0 // m
      Full / Reindex: q_idx [B,Tq,32,128], w_idx [B,Tq,32]
    Stored formats ([P3] section 六 and section 七 "FP4 Main KV"): with main_kv_fp4 the
    attention reads every main-KV entry through its FP4 form (csa2_ref.main_kv_fp4), with
    swa_fp8 every window row through its FP8 form (csa2_ref.swa_kv_fp8).
    Returns (outs, trace): outs[l] = [B,Tq,H,512] float64; trace[l] holds the
    layer's top-k [B,Tq,k], its scores / competing masks per (b, i), and candidates for
    a Full layer that builds a pool.
    """
    modes = layer_modes(kv_src, idx_src)
    builds_pool = {l: use_hsi and any(modes[r] == REINDEX and kv_src[r] == l
                                      for r in range(len(modes)))
                   for l in range(len(modes))}
    caches = {}
    slots = {"compress_kv": None, "index_k": None, "topk_idxs": None, "candidates": None}
    outs, trace = [], []
    for l, md in enumerate(modes):
        L = layers[l]
        tr = {}
        if md == FULL:
            m = ratio[l]
            kv_new, pre_new = R.compress(L["x"], L["w_kv"], L["w_gate"], L["gamma"], m,
                                         L["x_pos0"])
            G = kv_new.shape[1]
            pos = L["x_pos0"] + m * np.arange(G)
            kq = R.index_k(pre_new, L["w_ik"], np.broadcast_to(pos, (B, G)))
            codes, scales = R.index_k_quant(kq)
            kv_all = np.concatenate([L["prev_kv"], R.bf16_to_f64(R.f64_to_bf16_bits(kv_new))], 1)
            codes_all = np.concatenate([L["prev_codes"], codes], 1)
            scales_all = np.concatenate([L["prev_scales"], scales], 1)
            caches[l] = (kv_all, codes_all, scales_all, m)
            slots["compress_kv"] = l
            slots["index_k"] = l
            tr["kv_new"], tr["kv_pre_new"], tr["codes_new"], tr["scales_new"] = \
                kv_new, pre_new, codes, scales
        if md in (FULL, REINDEX):
            src = l if md == FULL else kv_src[l]
            kv_all, codes_all, scales_all, m = caches[src]
            N = kv_all.shape[1]
            k_hat = R.fp4.dequantize_rows(codes_all, scales_all)          # [B, N, 128]
            topk_out = np.full((B, Tq, k), -1, dtype=np.int32)
            tr["scores"], tr["valid"] = {}, {}
            cand_out = None
            if md == FULL and builds_pool[l]:
                cand_out = np.full((B, Tq, hsi_nb), -1, dtype=np.int32)
            for b in range(B):
                for i in range(Tq):
                    t = q_pos0 + i
                    nv = R.n_visible(t, m, N)
                    qh = R.quant_query(L["q_idx"][b, i])
                    sc = R.indexer_scores(qh, L["w_idx"][b, i], k_hat[b, :nv])
                    valid = np.ones(nv, dtype=bool)
                    if md == REINDEX and use_hsi:
                        valid = R.pool_mask(slots["candidates"][b, i], nv, hsi_blk, nv)
                    topk_out[b, i] = R.topk(sc, valid, k)
                    tr["scores"][b, i], tr["valid"][b, i] = sc, valid
                    if cand_out is not None:
                        bm = R.block_max(sc, nv, hsi_blk)
                        cand_out[b, i] = R.hsi_candidates(bm, nv, hsi_blk, hsi_nb)
            slots["topk_idxs"] = topk_out
            if cand_out is not None:
                slots["candidates"] = cand_out
                tr["candidates"] = cand_out
            tr["topk"] = topk_out
        # attention (every layer)
        H = L["q"].shape[2]
        o = np.zeros((B, Tq, H, R.D_ENTRY))
        for b in range(B):
            for i in range(Tq):
                t = q_pos0 + i
                if md == SWA:
                    sel = []
                    kv_rows = np.zeros((0, R.D_ENTRY))
                else:
                    kv_rows = caches[kv_src[l]][0][b]
                    if main_kv_fp4:
                        kv_rows = R.main_kv_dequant(*R.main_kv_fp4(kv_rows))
                    sel = slots["topk_idxs"][b, i]
                swa_rows = L["swa"][b]
                if swa_fp8:
                    swa_rows = R.swa_kv_dequant(*R.swa_kv_fp8(swa_rows))
                rows = R.attention_rows(kv_rows, sel, swa_rows, L["swa_pos0"], t, window)
                o[b, i] = R.sparse_attention(L["q"][b, i], rows, scale)
        outs.append(o)
        trace.append(tr)
    return outs, trace
