"""Float64 oracle of the CSA2 hot path (test infrastructure only).

Page abbreviations (full titles in ``oracle/__init__.py``):
[P1] javazero "CSA2 的三种模式", [P2] myhz0606 "架构篇", [P3] junki.cn "分级缓存",
[P4] reaper.mx "CSA2 — l'attention creuse compressée".

Everything is float64; inputs arrive as exact float64 widenings of the bf16 /
float32 bits the GPU consumes.  Where a float decides an integer (an FP4 code),
the value is first rounded to float32, the precision the GPU decides it in.
"""

import numpy as np

from . import fp4
from . import fp8

# ---- constants / readings -------------------------------------------------------------
D_ENTRY = 512        # main-KV entry width, K = V            [P1 §一层全局注意力算四样东西]
D_ROPE = 64          # RoPE on the last 64 dims              [P1 §压缩算子去掉了重叠和位置偏置, last para]
H_IDX = 32           # indexer heads                          [P1 §indexer K 改由 main KV 投影]
D_IDX = 128          # indexer head dim / indexer-K width     [same]
WINDOW = 128         # sliding window                         [P1 §一层全局注意力算四样东西, item 4]
RMS_EPS = 1e-6       # READING: epsilon not printed on the pages (parity unpinned)
ROPE_BASE = 10000.0  # READING: RoPE base (workload definition)
ATTN_SCALE = 1.0 / np.sqrt(D_ENTRY)   # READING: softmax(c.q / sqrt(d)) with d = 512 [P3 §四]


def bf16_to_f64(bits):
    """bf16 bit patterns (uint16) -> exact float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x):
    """Round float64 -> float32 -> bf16 (nearest-even both times), as the GPU stores
    its float32 results.  Pinned by hand-worked values (ties both ways, signed zeros,
    subnormals, overflow, and inputs where the two-step rounding differs from one step):
    tests/golden/bf16_rounding.txt."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


# ---- RMSNorm / RoPE ---------------------------------------------------------------------
def rmsnorm(v, gamma, eps=RMS_EPS):
    """y = gamma * v / sqrt(mean(v^2) + eps) over the last axis.

    [P1 §压缩算子去掉了重叠和位置偏置]: the pooled entry goes through RMSNorm.
    """
    v = np.asarray(v, dtype=np.float64)
    r = np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)
    return np.asarray(gamma, dtype=np.float64) * v / r


def rope_freqs(n_pairs=D_ROPE // 2, base=ROPE_BASE):
    """theta_i = base^(-2i / 64), i = 0..31."""
    i = np.arange(n_pairs, dtype=np.float64)
    return base ** (-2.0 * i / (2 * n_pairs))


def rope(v, pos, base=ROPE_BASE):
    """Rotate the last 64 dims of v[..., D] in interleaved pairs (2i, 2i+1) by pos*theta_i.

    [P1 §压缩算子去掉了重叠和位置偏置]: RoPE on the last 64 dims at the position of
    the group's first token.  READING: interleaved pair layout (parity unpinned).
    pos broadcasts against v[..., 0].
    """
    v = np.array(v, dtype=np.float64, copy=True)
    d = v.shape[-1]
    th = rope_freqs(base=base)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * th           # [..., 32]
    c, s = np.cos(ang), np.sin(ang)
    a = v[..., d - D_ROPE::2].copy()
    b = v[..., d - D_ROPE + 1::2].copy()
    v[..., d - D_ROPE::2] = a * c - b * s
    v[..., d - D_ROPE + 1::2] = a * s + b * c
    return v


# ---- stage 1: compressor ---------------------------------------------------------------
def compress(x, w_kv, w_gate, gamma, m, pos0=0, eps=RMS_EPS, base=ROPE_BASE):
    """CSA2 compressor over disjoint groups of m tokens.

    [P1 §压缩算子去掉了重叠和位置偏置] and [P2 §Compressor]: kv = wkv(x),
    score = wgate(x); each entry pools only its own group of m tokens (no overlap,
    no position bias) with a softmax over the group taken separately for every
    one of the 512 channels; then RMSNorm, then RoPE on the last 64 dims at the
    position of the group's first token.  m = 1 is the gate-less special case
    norm(wkv(x)) [P1 same section; P2: "对于 decoder ... 无需计算压缩权重"].

    x: [B, T, hidden] float64 for tokens at absolute positions pos0..pos0+T-1
    (pos0 a multiple of m); tokens of an incomplete trailing group make no entry.
    Returns (kv_rope, kv_pre), each [B, T // m, 512] float64; kv_pre is the
    normalised entry before RoPE (input of the indexer-K projection).
    """
    x = np.asarray(x, dtype=np.float64)
    B, T, _ = x.shape
    G = T // m
    x = x[:, : G * m]
    kv = x @ np.asarray(w_kv, dtype=np.float64).T                          # [B, G*m, 512]
    if m == 1:
        pooled = kv
    else:
        z = x @ np.asarray(w_gate, dtype=np.float64).T
        kv = kv.reshape(B, G, m, D_ENTRY)
        z = z.reshape(B, G, m, D_ENTRY)
        z = z - z.max(axis=2, keepdims=True)
        p = np.exp(z)
        p = p / p.sum(axis=2, keepdims=True)                               # per channel
        pooled = (p * kv).sum(axis=2)
    kv_pre = rmsnorm(pooled, gamma, eps)
    pos = pos0 + m * np.arange(G)
    kv_rope = rope(kv_pre, np.broadcast_to(pos, (B, G)), base)
    return kv_rope, kv_pre


# ---- stage 2: indexer K ------------------------------------------------------------------
def index_k(kv_pre, w_ik, entry_pos, base=ROPE_BASE):
    """k = W_IK . kv_pre (512 -> 128), then RoPE on k's last 64 dims.

    [P1 §indexer K 改由 main KV 投影]: the projection reads the main-KV entry
    before its RoPE; the indexer key then gets its own RoPE on its last 64 dims;
    no Hadamard rotation.  READING: the key's RoPE uses the entry's position.
    """
    k = np.asarray(kv_pre, dtype=np.float64) @ np.asarray(w_ik, dtype=np.float64).T
    return rope(k, entry_pos, base)


def index_k_quant(k):
    """Quantise indexer keys [..., 128]: decide in float32 (the kernel's precision)."""
    return fp4.quantize_rows(np.asarray(k, dtype=np.float64).astype(np.float32))


def quant_query(q_idx):
    """READING (parity unpinned): indexer queries [..., 32, 128] use the same FP4
    format as the keys, one E4M3 scale per 32 dims of each head.
    Returns the dequantised float64 values."""
    q = np.asarray(q_idx, dtype=np.float64).astype(np.float32)
    codes, scales = fp4.quantize_rows(q)
    return fp4.dequantize_rows(codes, scales)


MAIN_KV_BLOCK = 16


def main_kv_fp4(kv):
    """FP4 main-KV entries [..., 512] -> (codes [..., 256], scales [..., 32]).

    [P3] section 六: a main-KV entry takes 288 bytes; section 七 "FP4 Main KV": E2M1 data,
    channel groups share an E4M3 scale, dequantised before the attention.  READING: groups of
    16 channels (256 B codes + 32 one-byte scales = 288 B), the indexer keys' rounding rules,
    quantising the stored entry (its bf16 value; decisions in float32, the kernel's precision).
    """
    return fp4.quantize_rows(np.asarray(kv, dtype=np.float64).astype(np.float32), block=MAIN_KV_BLOCK)


def main_kv_dequant(codes, scales):
    """FP4 main-KV entries back to float64 (what the attention reads)."""
    return fp4.dequantize_rows(codes, scales)


def swa_kv_fp8(rows):
    """FP8 window-KV rows [..., 512] (bf16 values) -> (codes [..., 512], scales [..., 8]).

    [P3] section 七: the window KV stays FP8.  READING (the format is not given): E4M3
    elements, one power-of-two scale per 64 channels (fp8.py states the rules)."""
    return fp8.quantize_rows(rows)


def swa_kv_dequant(codes, scales):
    """FP8 window-KV rows back to float64 (what the attention reads)."""
    return fp8.dequantize_rows(codes, scales)


# ---- stage 3: lightning indexer, top-k, HSI -----------------------------------------------
def indexer_scores(q_hat, w, k_hat):
    """I[s] = sum_j w[j] * ReLU(q_hat[j] . k_hat[s]).

    [P1 §indexer K 改由 main KV 投影]: the scoring formula is unchanged from V4
    (per-head ReLU dot products weighted by per-head weights decided by the
    token, 32 heads of 128 dims).  READING: the ReLU lightning-indexer form.
    q_hat [H, 128], w [H], k_hat [N, 128] -> [N].
    """
    d = np.asarray(k_hat, np.float64) @ np.asarray(q_hat, np.float64).T    # [N, H]
    return np.maximum(d, 0.0) @ np.asarray(w, np.float64)


def n_visible(t, m, n_entries):
    """Entries visible to a query at position t: entry s covers tokens s*m..s*m+m-1
    and is visible once complete, s*m + m - 1 <= t.  [P2 §Indexer: 因果可见位置集合]
    READING: incomplete groups are invisible."""
    return int(max(0, min(n_entries, (t + 1) // m)))


def topk(scores, valid, k):
    """Top-k of the entries flagged valid, by (score desc, index asc).

    [P1 §一层全局注意力算四样东西, item 3] selects the k highest-scoring entries.
    READING: equal scores rank the lower index first; fewer than k valid entries
    pad with -1.  Output ascending entry indices, int32 [k].
    """
    scores = np.asarray(scores, dtype=np.float64)
    idx = np.nonzero(np.asarray(valid, dtype=bool))[0]
    order = np.lexsort((idx, -scores[idx]))            # primary: -score, then index
    sel = np.sort(idx[order[:k]])
    out = np.full(k, -1, dtype=np.int32)
    out[: len(sel)] = sel
    return out


def block_max(scores, n_vis, blk):
    """HSI block score: max index score of the visible entries of each block.

    [P2 §CSA2-ReIndex]: entries are split into blocks of size s and a block's score
    is the highest index score inside it.  Returns [ceil(n_vis / blk)] float64.
    """
    nb_vis = -(-n_vis // blk)
    out = np.empty(nb_vis)
    for b in range(nb_vis):
        out[b] = np.max(scores[b * blk: min((b + 1) * blk, n_vis)])
    return out


def hsi_candidates(bmax, n_vis, blk, nb):
    """Top-nb blocks of the block scores, the newest visible block forced in.

    [P2 §CSA2-ReIndex] and [P3 §五 HSI]: the highest-scoring blocks form the
    candidate pool; the block holding the newest causally visible entry is always
    kept.  READING: its score is set to +inf (the printed value is garbled); ties
    rank the lower block first; output ascending block ids padded with -1.
    """
    bmax = np.array(bmax, dtype=np.float64, copy=True)
    nb_vis = -(-n_vis // blk)
    bmax = bmax[:nb_vis]
    if nb_vis > 0:
        bmax[(n_vis - 1) // blk] = np.inf
    return topk(bmax, np.ones(nb_vis, dtype=bool), nb)


def pool_mask(cand, n_vis, blk, n_entries):
    """Entries inside the candidate blocks and visible. [P2 §CSA2-ReIndex]: entries
    outside the pool are scored -inf so they cannot be chosen."""
    mask = np.zeros(n_entries, dtype=bool)
    for b in np.asarray(cand):
        if b >= 0:
            mask[b * blk: min((b + 1) * blk, n_vis)] = True
    return mask


# ---- stage 4: sparse attention ------------------------------------------------------------
def sparse_attention(q, rows, scale=ATTN_SCALE, sink=None):
    """Shared K = V attention of H heads over the rows of the set A.

    [P3 §四]: p_j = exp(c_j.q / sqrt d) / sum_k exp(c_k.q / sqrt d), o = sum_j p_j c_j;
    [P2 §CSA2-FULL]: key and value are the same vector, taken from the selected
    compressed entries concatenated with the sliding-window rows.
    READING: optional per-head sink adds exp(sink_h) to the denominator only.
    q [H, 512], rows [n, 512] -> [H, 512] float64.
    """
    q = np.asarray(q, np.float64)
    rows = np.asarray(rows, np.float64)
    lg = (q @ rows.T) * scale                                     # [H, n]
    mx = lg.max(axis=1, keepdims=True)
    if sink is not None:
        mx = np.maximum(mx, np.asarray(sink, np.float64)[:, None])
    e = np.exp(lg - mx)
    den = e.sum(axis=1, keepdims=True)
    if sink is not None:
        den = den + np.exp(np.asarray(sink, np.float64)[:, None] - mx)
    return (e / den) @ rows


def attention_rows(kv_entries, topk_idx, swa_rows, swa_pos0, t, window=WINDOW):
    """Rows of A for a query at position t: the selected entries (valid indices, in
    the order given) followed by the window rows of positions max(0, t-W+1)..t.
    [P1 §一层全局注意力算四样东西, item 4]: the k selected entries plus the layer's
    own 128 window rows.  READING: a multiset (no de-duplication; the window rows
    come from a separate per-layer projection) and the window includes t."""
    sel = [int(s) for s in topk_idx if s >= 0]
    lo = max(0, t - window + 1)
    w = [swa_rows[p - swa_pos0] for p in range(lo, t + 1)]
    parts = []
    if sel:
        parts.append(np.asarray(kv_entries, np.float64)[sel])
    if w:
        parts.append(np.asarray(w, np.float64))
    return np.concatenate(parts, axis=0)
