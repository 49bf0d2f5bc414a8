"""Pins for the oracle's compressor, RoPE, indexer, selection, attention and layer
runtime (no GPU).  Each test checks the oracle against a closed form, an
invariant, a special case that reduces to a simpler definition, a hand-worked
example, or brute force -- never against a re-typing of the same formula.
"""

import itertools

import numpy as np
import pytest

from conftest import read_golden
from oracle import csa2_ref as R
from oracle import fp4
from oracle import layers as Lr


def _rng(s):
    return np.random.default_rng(s)


# ---------------------------------------------------------------- compressor
def test_compressor_m2_identical_tokens_equals_m1():
    # softmax weights sum to one: a group of two equal tokens pools to that token
    rng = _rng(0)
    x1 = rng.standard_normal((2, 3, 96))
    wkv = rng.standard_normal((512, 96)) * 0.1
    wg = rng.standard_normal((512, 96)) * 0.1
    g = np.ones(512)
    x2 = np.repeat(x1, 2, axis=1)                                # tokens 2i, 2i+1 equal
    kv2, pre2 = R.compress(x2, wkv, wg, g, m=2, pos0=0)
    # m = 1 entries of x1 at positions 0, 2, 4 (the group's first token)
    for gidx in range(3):
        kv1, pre1 = R.compress(x1[:, gidx:gidx + 1], wkv, None, g, m=1, pos0=2 * gidx)
        np.testing.assert_allclose(pre2[:, gidx], pre1[:, 0], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(kv2[:, gidx], kv1[:, 0], rtol=1e-12, atol=1e-12)


def test_compressor_gate_closed_form():
    # W_kv copies hidden dims 0..511, W_gate reads dims 512..1023.  Token 0 carries
    # gate ln 3, token 1 gate 0: weights 3/4, 1/4 per channel.  Pooled = constant 2
    # per channel -> RMSNorm gives 2 / sqrt(4 + eps) in every channel; position 0.
    hid = 1024
    wkv = np.zeros((512, hid)); wkv[np.arange(512), np.arange(512)] = 1.0
    wg = np.zeros((512, hid)); wg[np.arange(512), 512 + np.arange(512)] = 1.0
    x = np.zeros((1, 2, hid))
    x[0, 0, :512] = 2.5          # 0.75 * 2.5 + 0.25 * 0.5 = 2.0
    x[0, 1, :512] = 0.5
    x[0, 0, 512:] = np.log(3.0)
    kv, pre = R.compress(x, wkv, wg, np.ones(512), m=2, pos0=0)
    np.testing.assert_allclose(pre[0, 0], 2.0 / np.sqrt(4.0 + 1e-6), rtol=1e-14)
    np.testing.assert_allclose(kv[0, 0], pre[0, 0], rtol=1e-14)   # RoPE at pos 0 = identity


def test_compressor_zero_gate_is_plain_mean_and_channel_box():
    rng = _rng(1)
    x = rng.standard_normal((2, 8, 64))
    wkv = rng.standard_normal((512, 64)) * 0.2
    wg = rng.standard_normal((512, 64)) * 0.5
    g = np.ones(512)
    # zero gate: uniform weights -> pooled = mean, so entry = RMSNorm of the mean
    kv0, pre0 = R.compress(x, wkv, np.zeros_like(wg), g, m=2)
    kvi = (x @ wkv.T).reshape(2, 4, 2, 512)
    mean = kvi.mean(axis=2)
    scale = pre0 / mean
    assert np.allclose(scale, scale[..., :1], rtol=1e-10)          # one factor per entry
    # eps = 0: every entry has unit RMS after the norm
    _, pre = R.compress(x, wkv, wg, g, m=2, eps=0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(pre ** 2, axis=-1)), 1.0, rtol=1e-12)


def test_compressor_pooled_channel_box_exact():
    # with gamma = 1 and eps = 0 the pooled vector is pre * rms(pooled); recover the
    # pooled vector with a second, gate-identical call on scaled input and check
    # min <= pooled <= max per channel (the weights are a per-channel convex combination)
    rng = _rng(2)
    x = rng.standard_normal((1, 6, 32))
    wkv = rng.standard_normal((512, 32)) * 0.3
    wg = rng.standard_normal((512, 32))
    kvi = (x @ wkv.T).reshape(1, 3, 2, 512)
    _, pre = R.compress(x, wkv, wg, np.ones(512), m=2, eps=0.0)
    # pooled = pre * c with c = rms(pooled); c is the unique value making every
    # channel lie in its box; check a c exists (interval intersection non-empty)
    lo, hi = kvi.min(axis=2), kvi.max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        a = np.where(pre > 0, lo / pre, np.where(pre < 0, hi / pre, -np.inf))
        b = np.where(pre > 0, hi / pre, np.where(pre < 0, lo / pre, np.inf))
    assert np.all(a.max(axis=-1) <= b.min(axis=-1) * (1 + 1e-12))


def test_incomplete_trailing_group_makes_no_entry():
    rng = _rng(3)
    x = rng.standard_normal((1, 5, 16))
    kv, pre = R.compress(x, rng.standard_normal((512, 16)), rng.standard_normal((512, 16)),
                         np.ones(512), m=2)
    assert kv.shape == (1, 2, 512)


# ---------------------------------------------------------------- RoPE
def test_rope_matches_complex_rotation_and_properties():
    rng = _rng(4)
    v = rng.standard_normal((3, 512))
    pos = np.array([0, 7, 1_000_003])
    out = R.rope(v, pos)
    np.testing.assert_array_equal(out[:, :448], v[:, :448])
    np.testing.assert_allclose(out[0], v[0], rtol=0, atol=0)              # pos 0: identity
    # interleaved pair i as a complex number times exp(i * pos * base^(-i/32))
    z = v[:, 448::2] + 1j * v[:, 449::2]
    th = np.array([10000.0 ** (-(i / 32.0)) for i in range(32)])
    zr = z * np.exp(1j * pos[:, None] * th)
    np.testing.assert_allclose(out[:, 448::2], zr.real, atol=1e-12)
    np.testing.assert_allclose(out[:, 449::2], zr.imag, atol=1e-12)
    # relative-position property on the rotated part
    a, b = rng.standard_normal(512), rng.standard_normal(512)
    d1 = R.rope(a, 100)[448:] @ R.rope(b, 37)[448:]
    d2 = R.rope(a, 1100)[448:] @ R.rope(b, 1037)[448:]
    assert abs(d1 - d2) < 1e-9


def test_compressor_rope_position_is_group_first_token():
    # identity-like W_kv, zero gate: entry g of tokens at pos0 + 2g is rotated by pos0 + 2g
    hid = 512
    wkv = np.eye(512)
    x = np.zeros((1, 4, hid))
    x[0, :, 448] = 1.0                       # pair 0 = (1, 0) before norm
    kv, pre = R.compress(x, wkv, np.zeros((512, hid)), np.ones(512), m=2, pos0=6)
    for gidx, p in enumerate([6, 8]):
        r = pre[0, gidx, 448]
        np.testing.assert_allclose(kv[0, gidx, 448:450], [r * np.cos(p), r * np.sin(p)],
                                   atol=1e-12)


def test_index_k_is_linear_map_of_pre_rope_entry():
    rng = _rng(5)
    pre = rng.standard_normal((4, 512))
    sel = rng.permutation(512)[:128]
    w = np.zeros((128, 512)); w[np.arange(128), sel] = 1.0
    k = R.index_k(pre, w, entry_pos=np.zeros(4))
    np.testing.assert_array_equal(k, pre[:, sel])
    k2 = R.index_k(2.0 * pre, w, entry_pos=np.full(4, 9))
    k1 = R.index_k(pre, w, entry_pos=np.full(4, 9))
    np.testing.assert_allclose(k2, 2.0 * k1, rtol=1e-14)


# ---------------------------------------------------------------- indexer scores
def test_indexer_score_hand_example():
    # q = k = 1.5 everywhere: amax/6 = 0.25 exactly, codes 6 -> dequantised 1.5 exactly.
    # dot = 128 * 2.25 = 288 per head; I = 288 * sum(w) when all w > 0; ReLU kills k = -q.
    q = np.full((32, 128), 1.5)
    qh = R.quant_query(q)
    np.testing.assert_array_equal(qh, q)
    codes, scales = R.index_k_quant(np.stack([np.full(128, 1.5), np.full(128, -1.5)]))
    kh = fp4.dequantize_rows(codes, scales)
    w = np.arange(1, 33, dtype=np.float64) / 8
    I = R.indexer_scores(qh, w, kh)
    assert I[0] == 288.0 * w.sum() and I[1] == 0.0


def test_indexer_one_hot_weight_and_permutation():
    rng = _rng(6)
    qh = rng.standard_normal((32, 128))
    kh = rng.standard_normal((50, 128))
    for j in (0, 13, 31):
        w = np.zeros(32); w[j] = 1.0
        I = R.indexer_scores(qh, w, kh)
        # single head: ReLU of one dot product, computed element by element
        for s in (0, 7, 49):
            d = sum(qh[j, i] * kh[s, i] for i in range(128))
            assert abs(I[s] - max(d, 0.0)) < 1e-9
    perm = rng.permutation(50)
    w = rng.standard_normal(32)
    np.testing.assert_allclose(R.indexer_scores(qh, w, kh[perm]),
                               R.indexer_scores(qh, w, kh)[perm], rtol=1e-13)


def test_visibility():
    assert R.n_visible(0, 2, 100) == 0 and R.n_visible(1, 2, 100) == 1
    assert R.n_visible(0, 1, 100) == 1 and R.n_visible(131071, 1, 131072) == 131072
    assert R.n_visible(2 * 524288 - 1, 2, 524288) == 524288
    assert R.n_visible(10, 2, 3) == 3


# ---------------------------------------------------------------- selection
def test_topk_hand_examples():
    g = read_golden("selection_examples.txt")
    sc = np.array([float(v) for v in g["topk_scores"][0]])
    for row in g["topk"]:
        nv, k = int(row[0]), int(row[1])
        exp = [int(v) for v in row[3:]]
        valid = np.arange(len(sc)) < nv
        np.testing.assert_array_equal(R.topk(sc, valid, k), exp)


@pytest.mark.parametrize("seed", range(6))
def test_topk_equals_brute_force_full_sort(seed):
    rng = _rng(100 + seed)
    for n in (1, 5, 17, 64):
        # integer-valued scores plant many exact ties
        sc = rng.integers(-4, 5, size=n).astype(np.float64)
        for k in (1, 3, n, n + 4):
            for nv in (0, n // 2, n):
                valid = np.arange(n) < nv
                brute = sorted(range(nv), key=lambda s: (-sc[s], s))[:k]
                exp = sorted(brute) + [-1] * (k - len(brute))
                np.testing.assert_array_equal(R.topk(sc, valid, k), exp)


def test_topk_tiny_exhaustive_permutations():
    # every ordering of 5 distinct scores, k = 2: the top two are the two largest
    vals = [0.5, -1.0, 3.0, 2.0, 7.0]
    for perm in itertools.permutations(range(5)):
        sc = np.array([vals[p] for p in perm])
        top = {i for i in range(5) if sc[i] >= 3.0}
        assert set(R.topk(sc, np.ones(5, bool), 2).tolist()) == top


def test_hsi_hand_examples():
    g = read_golden("selection_examples.txt")
    sc = np.array([float(v) for v in g["hsi_scores"][0]])
    exp_bm = [float(v) for v in g["hsi_blockmax"][0]]
    np.testing.assert_array_equal(R.block_max(sc, 14, 4), exp_bm)
    for row in g["hsi"]:
        nv, blk, nb = int(row[0]), int(row[1]), int(row[2])
        exp = [int(v) for v in row[4:]]
        np.testing.assert_array_equal(R.hsi_candidates(R.block_max(sc, nv, blk), nv, blk, nb), exp)
    sc = np.array([float(v) for v in g["hsi_tie_scores"][0]])
    for row in g["hsi_tie"]:
        nv, blk, nb = int(row[0]), int(row[1]), int(row[2])
        exp = [int(v) for v in row[4:]]
        np.testing.assert_array_equal(R.hsi_candidates(R.block_max(sc, nv, blk), nv, blk, nb), exp)
    sc = np.array([float(v) for v in g["reindex_scores"][0]])
    for row in g["reindex"]:
        nv, blk, k = int(row[0]), int(row[1]), int(row[2])
        exp = [int(v) for v in row[4:]]
        mask = R.pool_mask([1, 3], nv, blk, nv)
        np.testing.assert_array_equal(R.topk(sc[:nv], mask, k), exp)


def test_pool_covering_everything_reduces_to_plain_topk():
    rng = _rng(7)
    sc = rng.standard_normal(300)
    nv, blk = 257, 16
    cand = R.hsi_candidates(R.block_max(sc, nv, blk), nv, blk, 64)
    assert set(cand[cand >= 0].tolist()) == set(range(17))
    mask = R.pool_mask(cand, nv, blk, nv)
    np.testing.assert_array_equal(R.topk(sc[:nv], mask, 40),
                                  R.topk(sc[:nv], np.ones(nv, bool), 40))


# ---------------------------------------------------------------- attention
def test_attention_special_cases():
    rng = _rng(8)
    c = rng.standard_normal((1, 512))
    q = rng.standard_normal((4, 512))
    np.testing.assert_allclose(R.sparse_attention(q, c), np.repeat(c, 4, 0), rtol=1e-14)
    rows = rng.standard_normal((9, 512))
    np.testing.assert_allclose(R.sparse_attention(np.zeros((2, 512)), rows),
                               np.repeat(rows.mean(0, keepdims=True), 2, 0), rtol=1e-12)
    # two keys whose logits differ by ln 3: weights 3/4 and 1/4
    c2 = np.zeros((2, 512)); c2[0, 0] = 1.0; c2[1, 1] = 1.0
    qq = np.zeros((1, 512)); qq[0, 0] = np.log(3.0) * np.sqrt(512)
    np.testing.assert_allclose(R.sparse_attention(qq, c2)[0, :2], [0.75, 0.25], rtol=1e-13)


def test_attention_convex_hull_and_sink():
    rng = _rng(9)
    rows = rng.standard_normal((40, 512))
    q = 3.0 * rng.standard_normal((8, 512))
    o = R.sparse_attention(q, rows)
    assert np.all(o <= rows.max(0) + 1e-12) and np.all(o >= rows.min(0) - 1e-12)
    # sink with one key: o = c * e^l / (e^l + e^sink)
    c = rng.standard_normal((1, 512))
    qq = rng.standard_normal((2, 512))
    lg = qq @ c[0] / np.sqrt(512)
    sink = np.array([0.3, -2.0])
    got = R.sparse_attention(qq, c, sink=sink)
    frac = np.exp(lg) / (np.exp(lg) + np.exp(sink))
    np.testing.assert_allclose(got, frac[:, None] * c, rtol=1e-12)


def test_exponential_tilting_identity():
    # [P3] §四: p_j(q0 + dq) is proportional to p_j(q0) * exp(c_j . dq / sqrt d).
    # Rows c_j = e_j make o_j = p_j, so the weights can be read off the output.
    n = 30
    rows = np.zeros((n, 512)); rows[np.arange(n), np.arange(n)] = 1.0
    rng = _rng(10)
    q0 = 4.0 * rng.standard_normal((1, 512))
    dq = 4.0 * rng.standard_normal((1, 512))
    p0 = R.sparse_attention(q0, rows)[0, :n]
    p1 = R.sparse_attention(q0 + dq, rows)[0, :n]
    tilt = p0 * np.exp(rows @ dq[0] / np.sqrt(512))
    np.testing.assert_allclose(p1, tilt / tilt.sum(), rtol=1e-11)


def test_attention_rows_window_and_selection():
    kv = np.arange(20 * 512, dtype=np.float64).reshape(20, 512)
    swa = -np.arange(300 * 512, dtype=np.float64).reshape(300, 512)
    rows = R.attention_rows(kv, np.array([3, 9, -1]), swa, swa_pos0=100, t=250, window=128)
    assert rows.shape[0] == 2 + 128
    np.testing.assert_array_equal(rows[0], kv[3])
    np.testing.assert_array_equal(rows[2], swa[250 - 127 - 100])
    np.testing.assert_array_equal(rows[-1], swa[150])
    rows = R.attention_rows(kv, np.array([-1]), swa, swa_pos0=0, t=5, window=128)
    assert rows.shape[0] == 6            # window clipped at position 0, includes t


# ---------------------------------------------------------------- layer runtime
def test_v41_layer_pattern_and_accounting():
    g = read_golden("layer_pattern.txt")
    kv_src, idx_src, ratio = Lr.v41_flash_tables()
    modes = Lr.layer_modes(kv_src, idx_src)
    assert len(modes) == int(g["n_layers"][0][0])
    assert [l for l, m in enumerate(modes) if m == Lr.FULL] == [int(v) for v in g["full"][0]]
    assert [l for l, m in enumerate(modes) if m == Lr.REINDEX] == [int(v) for v in g["reindex"][0]]
    assert modes.count(Lr.REUSE) == int(g["n_reuse"][0][0])
    assert modes.count(Lr.SWA) == int(g["n_swa_only"][0][0])
    assert Lr.entries_per_token(kv_src, idx_src, ratio) == float(g["entries_per_token"][0][0])
    assert Lr.bytes_per_token(kv_src, idx_src, ratio) == float(g["bytes_per_token"][0][0])
    for l, b in g["per_layer_bytes"]:
        assert int(g["entry_bytes"][0][0]) / ratio[int(l)] == float(b)
    enc = sum(356 / ratio[l] for l, m in enumerate(modes) if m == Lr.FULL and ratio[l] == 2)
    assert enc == float(g["encoder_bytes"][0][0])
    # V4-Flash: 41 own-KV layers, 21 at ratio 4 and 20 at ratio 128
    v4_kv = list(range(41))
    v4_ratio = [4] * 21 + [128] * 20
    e = Lr.entries_per_token(v4_kv, v4_kv, v4_ratio)
    assert round(e, 2) == float(g["v4_entries_per_token"][0][0])
    # one more Full layer: +0.5 entry/token in the encoder (ratio 2), +1 in the decoder
    kv2, idx2, r2 = list(kv_src), list(idx_src), list(ratio)
    kv2[5], idx2[5], r2[5] = 5, 5, 2
    for l in (6, 7):
        kv2[l], idx2[l] = 5, 5
    assert Lr.entries_per_token(kv2, idx2, r2) - 2.5 == float(g["extra_entries_encoder_full"][0][0])
    kv3, idx3, r3 = list(kv_src), list(idx_src), list(ratio)
    kv3[30], idx3[30], r3[30] = 30, 30, 1
    for l in (31,):
        kv3[l], idx3[l] = 30, 30
    assert Lr.entries_per_token(kv3, idx3, r3) - 2.5 == float(g["extra_entries_decoder_full"][0][0])


def test_invalid_tables_rejected():
    with pytest.raises(ValueError):
        Lr.layer_modes([0, 1], [0, 0])            # own KV with a foreign index
    with pytest.raises(ValueError):
        Lr.layer_modes([0, 2, 2], [0, 1, 2])      # forward KV source
    with pytest.raises(ValueError):
        Lr.layer_modes([0, 1, 0], [0, 1, 1])      # reuses an index made for another KV
    with pytest.raises(ValueError):
        Lr.layer_modes([-1, 0], [-1, 0])          # source is not Full
    with pytest.raises(ValueError):
        Lr.layer_modes([-1], [0])
    assert Lr.layer_modes([-1, 1, 1, 1, 1], [-1, 1, 1, 3, 3]) == \
        [Lr.SWA, Lr.FULL, Lr.REUSE, Lr.REINDEX, Lr.REUSE]


def _tiny_stack_inputs(rng, kv_src, ratio, B, Tq, q_pos0, n0_tokens, hid=64, H=2):
    """Small float64 inputs for oracle run_step (bf16 values not needed here)."""
    layers = []
    for l in range(len(kv_src)):
        L = {"q": rng.standard_normal((B, Tq, H, 512)),
             "swa": rng.standard_normal((B, q_pos0 + Tq, 512)), "swa_pos0": 0,
             "q_idx": rng.standard_normal((B, Tq, 32, 128)),
             "w_idx": rng.standard_normal((B, Tq, 32))}
        if kv_src[l] == l:
            m = ratio[l]
            xall = rng.standard_normal((B, q_pos0 + Tq, hid))
            L.update(w_kv=rng.standard_normal((512, hid)) * 0.2,
                     w_gate=rng.standard_normal((512, hid)) * 0.2 if m > 1 else None,
                     gamma=np.ones(512), w_ik=rng.standard_normal((128, 512)) * 0.05)
            n0 = n0_tokens // m
            kv_p, pre_p = R.compress(xall[:, : n0 * m], L["w_kv"], L["w_gate"], L["gamma"], m)
            pos = m * np.arange(n0)
            c, s = R.index_k_quant(R.index_k(pre_p, L["w_ik"], np.broadcast_to(pos, (B, n0))))
            L.update(prev_kv=R.bf16_to_f64(R.f64_to_bf16_bits(kv_p)), prev_codes=c,
                     prev_scales=s, x=xall[:, n0 * m:], x_pos0=n0 * m)
        layers.append(L)
    return layers


def test_runner_reuse_with_source_query_reproduces_source():
    rng = _rng(11)
    kv_src, idx_src, ratio = [0, 0, 0], [0, 0, 0], [2, 0, 0]
    B, Tq, q_pos0 = 2, 3, 40
    layers = _tiny_stack_inputs(rng, kv_src, ratio, B, Tq, q_pos0, n0_tokens=40)
    for l in (1, 2):
        layers[l]["swa"] = layers[0]["swa"]
    layers[1]["q"] = layers[0]["q"]                  # same query as the source
    outs, trace = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=8)
    np.testing.assert_array_equal(outs[1], outs[0])
    assert not np.allclose(outs[2], outs[0])         # own query -> different output


def test_runner_reindex_with_full_pool_equals_full_topk():
    # nb covering every block: Reindex = plain top-k with that layer's indexer query
    rng = _rng(12)
    kv_src, idx_src, ratio = [0, 0, 0], [0, 1, 1], [1, 0, 0]
    B, Tq, q_pos0 = 1, 2, 60
    layers = _tiny_stack_inputs(rng, kv_src, ratio, B, Tq, q_pos0, n0_tokens=60)
    outs, trace = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=10,
                              hsi_blk=8, hsi_nb=64)
    outs2, trace2 = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=10,
                                use_hsi=False)
    np.testing.assert_array_equal(trace[1]["topk"], trace2[1]["topk"])
    # and a small pool restricts the choice to its blocks
    outs3, trace3 = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=10,
                                hsi_blk=8, hsi_nb=2)
    cand = trace3[0]["candidates"]
    for i in range(Tq):
        sel = trace3[1]["topk"][0, i]
        blocks = set((sel[sel >= 0] // 8).tolist())
        assert blocks <= set(cand[0, i][cand[0, i] >= 0].tolist())
    # the newest visible block is always in the pool
    for i in range(Tq):
        nv = R.n_visible(q_pos0 + i, 1, 62)
        assert (nv - 1) // 8 in cand[0, i]


def _fp4_exact_rows(rng, shape):
    """Rows whose 16-channel groups are E2M1 values times an E4M3 scale with one element at
    6 x scale: the FP4 main-KV quantiser reproduces them exactly."""
    mags = fp4.E2M1_MAG
    v = rng.choice(mags, size=shape + (512,)) * rng.choice([-1.0, 1.0], size=shape + (512,))
    g = v.reshape(shape + (32, 16))
    g[..., 0] = 6.0
    scale = fp4.e4m3_value(rng.integers(0x18, 0x30, size=shape + (32,)))   # 2^-4 .. 0.875
    return (g * scale[..., None]).reshape(shape + (512,))


def _fp8_exact_rows(rng, shape):
    """Rows whose 64-channel groups are E4M3 grid values times 2^k with one element in
    (224, 448] x 2^k: the FP8 window quantiser reproduces them exactly."""
    grid = fp4._E4M3_GRID
    c = rng.integers(0, 127, size=shape + (8, 64))
    c[..., 0] = rng.integers(0x70, 0x7F, size=shape + (8,))
    k = rng.integers(-12, -8, size=shape + (8,))                          # |v| < 1.75
    v = grid[c] * np.where(rng.random(c.shape) < 0.5, -1.0, 1.0) * np.exp2(k)[..., None]
    return v.reshape(shape + (512,))


def test_run_step_stored_formats_reduce_to_plain_on_representable_rows():
    """[P3] section 七: attention reads FP4 entries and FP8 window rows after dequantisation;
    on rows the two formats hold exactly, the stored-format step equals the plain step, and
    moving one window value off the FP8 grid changes it."""
    rng = _rng(21)
    kv_src, idx_src, ratio = [-1, 1, 1], [-1, 1, 1], [0, 2, 0]
    B, Tq = 2, 1
    q_pos0 = 80                                     # token 80 starts a group: no new entry
    layers = _tiny_stack_inputs(rng, kv_src, ratio, B, Tq, q_pos0, n0_tokens=80)
    n0 = layers[1]["prev_kv"].shape[1]
    layers[1]["prev_kv"] = _fp4_exact_rows(rng, (B, n0))
    for L in layers:
        L["swa"] = _fp8_exact_rows(rng, L["swa"].shape[:2])
    assert layers[1]["x"].shape[1] == 1
    plain, _ = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=8)
    stored, _ = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=8,
                            main_kv_fp4=True, swa_fp8=True)
    for a, b in zip(plain, stored):
        np.testing.assert_array_equal(a, b)
    layers[0]["swa"][:, q_pos0, 5] += 1e-3 * np.sign(layers[0]["swa"][:, q_pos0, 5] + 0.5)  # off the grid
    moved, _ = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=8,
                           main_kv_fp4=True, swa_fp8=True)
    plain2, _ = Lr.run_step(kv_src, idx_src, ratio, layers, B, Tq, q_pos0, k=8)
    assert not np.array_equal(moved[0], plain2[0])


# ---- bf16 store rounding ----------------------------------------------------------------
def test_bf16_store_rounding_golden():
    """f64_to_bf16_bits against hand-worked values (tests/golden/bf16_rounding.txt): ties
    to even in both directions, signed zeros, subnormals (including a tie), overflow to
    infinity at bf16 max + half an ulp, and two float64 inputs where rounding through
    float32 (the GPU's path: a float32 result stored as bf16) differs from rounding float64
    to bf16 in one step -- so truncation, a lost tie rule or one-step rounding each fail."""
    g = read_golden("bf16_rounding.txt")
    rows = g["round"]
    assert len(rows) >= 18
    xs = np.array([float.fromhex(r[1]) for r in rows])
    want = np.array([int(r[2], 16) for r in rows], dtype=np.uint16)
    got = R.f64_to_bf16_bits(xs)
    bad = [(r[0], hex(int(a)), hex(int(b))) for r, a, b in zip(rows, got, want) if a != b]
    assert not bad, bad
    # elementwise on any shape, one value at a time the same
    assert (R.f64_to_bf16_bits(xs.reshape(2, -1)).ravel() == want).all()
    assert all(R.f64_to_bf16_bits(np.float64(x)) == w for x, w in zip(xs, want))


def test_bf16_widening_golden_and_round_trip():
    g = read_golden("bf16_rounding.txt")
    for bits, val in g["widen"]:
        v = R.bf16_to_f64(np.uint16(int(bits, 16)))
        want = float("inf") if val == "inf" else float.fromhex(val)
        assert v == want and np.signbit(v) == np.signbit(want), (bits, v, want)
    # every finite bf16 widens exactly and rounds back to itself
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = R.bf16_to_f64(allb)
    fin = np.isfinite(v)
    assert (R.f64_to_bf16_bits(v[fin]) == allb[fin]).all()
    # widening is monotone over the positive finite patterns
    pos = v[: 0x7F80]
    assert (np.diff(pos) > 0).all()
