"""Parity at the full sizes of the decode and prefill workloads, through the same entry points
and launch shapes the benchmark step uses (persistent FP4 scorer, threshold-filtered top-k,
clustered attention).

The device inputs are filled by the generator's device twin; the oracle regenerates only the
sampled rows on the host (same generator, same element offsets) and checks them one by one.
No oracle input comes from the CUDA path.

Workloads covered (all at their stated sizes):
  * 40-layer decode, batch 64 at 131072 tokens: encoder Full (m = 2, 65536 entries), decoder
    Full (m = 1, 131072 entries, block maxima), Reindex over a 64-block pool, HSI, attention
    over 512 + 128 rows with 64 heads, the per-step compressor.
  * decoder-group decode, batch 32 at 65536 entries: Full with block maxima, Reindex.
  * the HSI variant with 8-entry blocks: Reindex over 2048-block (16 384-entry) pools and HSI
    over 64 x 16 384 blocks.
  * long-context decode, batch 4, 524288 entries (m = 2): indexer and attention.
  * encoder prefill, 16384 tokens, 8192 entries: compressor, index keys, causal indexer,
    attention.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import csa2_ref as R
from oracle import fp4

import helpers as Hp

pytestmark = pytest.mark.gpu

ZERO_SCALE_EVERY = 97


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from compressed_sparse_attention_04_gb300 import build
    build.build_all()


def _ops():
    from compressed_sparse_attention_04_gb300 import ops
    return ops


def _ok():
    assert _ops().last_device_status() == 0


# ---------------------------------------------------------------- generated caches
def _device_index_cache(seed, stream, B, n_cap):
    """Device copy of the FP4 index cache of helpers.index_cache_input: the same words
    through the same transform (codes = low byte, scale = 0x18 + low 6 bits, every 97th
    entry's scales zero)."""
    from synth import gpu as sg
    codes = torch.empty(B, n_cap, 64, dtype=torch.uint8, device="cuda")
    scales = torch.empty(B, n_cap, 4, dtype=torch.uint8, device="cuda")
    per = max(1, (1 << 28) // (n_cap * 68))          # sequences per generator chunk
    for b0 in range(0, B, per):
        nb = min(per, B - b0)
        r = torch.empty(nb * n_cap * 68, dtype=torch.int32, device="cuda")
        sg.fill_u32(r, seed, stream, b0 * n_cap * 68)
        r = r.view(nb, n_cap, 68)
        codes[b0:b0 + nb] = (r[..., :64] & 0xFF).to(torch.uint8)
        scales[b0:b0 + nb] = (0x18 + (r[..., 64:] & 0x3F)).to(torch.uint8)
        del r
    scales.view(-1, 4)[::ZERO_SCALE_EVERY] = 0
    return codes, scales


def _host_index_rows(seed, stream, b, n_cap, n):
    """Entries 0..n-1 of sequence b of the same cache, regenerated on the host."""
    r = synth.uniform_u32(seed, stream, b * n_cap * 68, n * 68).reshape(n, 68)
    codes = (r[:, :64] & 0xFF).astype(np.uint8)
    scales = (0x18 + (r[:, 64:] % 0x40)).astype(np.uint8)
    rows = b * n_cap + np.arange(n)
    scales[rows % ZERO_SCALE_EVERY == 0] = 0
    return codes, scales


def test_host_index_rows_match_the_small_cache_generator():
    # the row regenerator reproduces helpers.index_cache_input, sequence by sequence
    codes, scales = Hp.index_cache_input(31, 3, 3, 500)
    for b in range(3):
        c_b, s_b = _host_index_rows(31, 3, b, 500, 500)
        np.testing.assert_array_equal(c_b, codes[b])
        np.testing.assert_array_equal(s_b, scales[b])


def test_device_index_cache_matches_the_small_cache_generator():
    codes, scales = Hp.index_cache_input(31, 3, 3, 500)
    dc, ds = _device_index_cache(31, 3, 3, 500)
    np.testing.assert_array_equal(dc.cpu().numpy(), codes)
    np.testing.assert_array_equal(ds.cpu().numpy(), scales)


def _oracle_row_scores(qi64, w64, codes, scales):
    return R.indexer_scores(R.quant_query(qi64), w64, fp4.dequantize_rows(codes, scales))


# ---------------------------------------------------------------- indexer
@pytest.mark.parametrize("B,n_entries,m,blockmax,rows", [
    (64, 131072, 1, True, (0, 37, 63)),   # 40-layer decode: decoder Full (HSI source)
    (64, 65536, 2, False, (5, 50)),       # 40-layer decode: encoder Full
    (32, 65536, 1, True, (0, 31)),        # decoder-group decode: Full
    (4, 524288, 2, False, (2,)),          # long-context decode at 1M tokens
])
def test_indexer_full_size_sampled_rows(B, n_entries, m, blockmax, rows):
    ops = _ops()
    k, seed = 512, 9000 + n_entries // 1024 + B
    q_pos0 = m * n_entries - 1            # decode: every entry complete and visible
    codes, scales = _device_index_cache(seed, 3, B, n_entries)
    qi, qi64 = Hp.bf16_input(seed, 1, (B, 1, 32, 128), 1.28)
    w, w64 = Hp.f32_input(seed, 2, (B, 1, 32), 1.28)
    bm = (torch.empty(B, 1, n_entries // 64, dtype=torch.float32, device="cuda")
          if blockmax else None)
    topk = ops.indexer_score_topk(qi, w, q_pos0, codes, scales, n_entries, m, k, blk=64,
                                  blockmax_out=bm)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    bm = bm.cpu().numpy() if blockmax else None
    del codes, scales
    for b in rows:
        c_b, s_b = _host_index_rows(seed, 3, b, n_entries, n_entries)
        so = _oracle_row_scores(qi64[b, 0], w64[b, 0], c_b, s_b)
        Hp.check_topk_row(topk[b, 0], so, np.ones(n_entries, bool), k, f"sequence {b}")
        if blockmax:
            np.testing.assert_allclose(bm[b, 0], R.block_max(so, n_entries, 64), rtol=1e-5,
                                       atol=1e-5 * np.max(np.abs(so)))


def _pool(seed, B, n_blocks, nb):
    """nb distinct ascending blocks per sequence, the newest block always included."""
    r = synth.uniform_u32(seed, 5, 0, B * n_blocks).reshape(B, n_blocks)
    out = np.empty((B, nb), np.int32)
    for b in range(B):
        order = np.argsort(r[b], kind="stable")
        take = order[:nb]
        if n_blocks - 1 not in take:
            take = np.concatenate([order[:nb - 1], [n_blocks - 1]])
        out[b] = np.sort(take)
    return out


@pytest.mark.parametrize("B,n_entries,rows", [
    (64, 131072, (3, 60)),    # 40-layer decode: Reindex layer
    (32, 65536, (7,)),        # decoder-group decode: Reindex layer
])
def test_reindex_pool_full_size_sampled_rows(B, n_entries, rows):
    ops = _ops()
    nb, blk, k, seed = 64, 64, 512, 9300 + B
    codes, scales = _device_index_cache(seed, 3, B, n_entries)
    qi, qi64 = Hp.bf16_input(seed, 1, (B, 1, 32, 128), 1.28)
    w, w64 = Hp.f32_input(seed, 2, (B, 1, 32), 1.28)
    cand = _pool(seed, B, n_entries // blk, nb)
    topk = ops.indexer_score_topk(qi, w, n_entries - 1, codes, scales, n_entries, 1, k,
                                  cand=Hp.to_dev(cand.reshape(B, 1, nb), torch.int32), blk=blk)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    del codes, scales
    for b in rows:
        c_b, s_b = _host_index_rows(seed, 3, b, n_entries, n_entries)
        so = _oracle_row_scores(qi64[b, 0], w64[b, 0], c_b, s_b)
        mask = R.pool_mask(cand[b], n_entries, blk, n_entries)
        Hp.check_topk_row(topk[b, 0], so, mask, k, f"sequence {b}")


def test_reindex_8_key_block_pools_full_size_sampled_rows():
    # 64 sequences x 131072 entries, pools of 2048 blocks of 8 entries (16 384 entries)
    ops = _ops()
    B, n_entries, nb, blk, k, seed = 64, 131072, 2048, 8, 512, 9350
    codes, scales = _device_index_cache(seed, 3, B, n_entries)
    qi, qi64 = Hp.bf16_input(seed, 1, (B, 1, 32, 128), 1.28)
    w, w64 = Hp.f32_input(seed, 2, (B, 1, 32), 1.28)
    cand = _pool(seed, B, n_entries // blk, nb)
    topk = ops.indexer_score_topk(qi, w, n_entries - 1, codes, scales, n_entries, 1, k,
                                  cand=Hp.to_dev(cand.reshape(B, 1, nb), torch.int32), blk=blk)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    del codes, scales
    for b in (11, 52):
        c_b, s_b = _host_index_rows(seed, 3, b, n_entries, n_entries)
        so = _oracle_row_scores(qi64[b, 0], w64[b, 0], c_b, s_b)
        mask = R.pool_mask(cand[b], n_entries, blk, n_entries)
        Hp.check_topk_row(topk[b, 0], so, mask, k, f"sequence {b}")


def test_hsi_8_key_blocks_full_size():
    # block maxima of 64 sequences x 16 384 blocks of 8 entries, 2048 candidates each
    ops = _ops()
    B, n_entries, blk, nb = 64, 131072, 8, 2048
    bm, bm64 = Hp.f32_input(9410, 1, (B, 1, n_entries // blk))
    cand = ops.hsi_candidates(bm, n_entries - 1, n_entries, 1, blk, nb).cpu().numpy()
    _ok()
    for b in range(0, B, 9):
        np.testing.assert_array_equal(cand[b, 0], R.hsi_candidates(bm64[b, 0], n_entries, blk, nb))


def test_hsi_full_size():
    # block maxima of 64 sequences x 2048 blocks: the decoder Full layer at 131072 entries
    ops = _ops()
    B, n_entries, blk, nb = 64, 131072, 64, 64
    bm, bm64 = Hp.f32_input(9400, 1, (B, 1, n_entries // blk))
    cand = ops.hsi_candidates(bm, n_entries - 1, n_entries, 1, blk, nb).cpu().numpy()
    _ok()
    for b in range(0, B, 7):
        np.testing.assert_array_equal(cand[b, 0], R.hsi_candidates(bm64[b, 0], n_entries, blk, nb))


def test_prefill_indexer_full_size_sampled_rows():
    # the 16384-token encoder prefill: 8192 entries (m = 2), causal visibility per query
    from synth import gpu as sg
    ops = _ops()
    Tq, n_entries, m, k, seed = 16384, 8192, 2, 512, 9500
    codes, scales = _device_index_cache(seed, 3, 1, n_entries)
    qi = sg.fill_normal(torch.empty(1, Tq, 32, 128, dtype=torch.bfloat16, device="cuda"),
                        seed, 1, 0, 1.28)
    w = sg.fill_normal(torch.empty(1, Tq, 32, dtype=torch.float32, device="cuda"), seed, 2, 0, 1.28)
    topk = ops.indexer_score_topk(qi, w, 0, codes, scales, n_entries, m, k)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    c_all, s_all = _host_index_rows(seed, 3, 0, n_entries, n_entries)
    k_all = fp4.dequantize_rows(c_all, s_all)
    for i in (0, 1, 2, 1023, 1024, 4097, 16383):
        nv = R.n_visible(i, m, n_entries)
        if nv == 0:
            assert np.all(topk[0, i] == -1)
            continue
        q_i = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, i * 4096, 4096, 1.28)).reshape(32, 128)
        w_i = synth.normal_f32(seed, 2, i * 32, 32, 1.28).astype(np.float64)
        so = R.indexer_scores(R.quant_query(q_i), w_i, k_all[:nv])
        Hp.check_topk_row(topk[0, i], so, np.ones(nv, bool), k, f"query {i}")


# ---------------------------------------------------------------- attention
def _spread_topk(B, Tq, k, n_vis):
    """Distinct ascending selected entries spread over each query's visible range, with a
    per-(sequence, query) offset; fewer than k visible entries take them all, -1 padded."""
    out = np.full((B, Tq, k), -1, np.int32)
    n_vis = np.broadcast_to(np.asarray(n_vis), (Tq,))
    for i in range(Tq):
        n = int(n_vis[i])
        if n <= k:
            out[:, i, :n] = np.arange(n)
            continue
        gap = n // k                                  # consecutive picks are >= gap apart
        base = (np.arange(k, dtype=np.int64) * n) // k
        off = (np.arange(B) * 7 + i * 13) % gap
        out[:, i] = base[None, :] + off[:, None]
    return out


def _entry_rows(seed, stream, b, n_cap, sel):
    return np.stack([R.bf16_to_f64(synth.normal_bf16_bits(seed, stream, (b * n_cap + int(e)) * 512, 512))
                     for e in sel]) if len(sel) else np.zeros((0, 512))


@pytest.mark.parametrize("B,n_cap,q_pos0,rows", [
    (64, 65536, 131071, (0, 31, 63)),     # 40-layer decode, encoder layers (65536 entries)
    (64, 131072, 131071, (17,)),          # 40-layer decode, decoder layers (131072 entries)
    (4, 524288, 1048575, (1, 3)),         # long-context decode at 1M tokens
])
def test_sparse_attention_full_size_sampled_rows(B, n_cap, q_pos0, rows):
    from synth import gpu as sg
    ops = _ops()
    H, k, W, S, seed = 64, 512, 128, 256, 9600 + B + n_cap // 65536
    swa_pos0 = q_pos0 - S + 1
    q = sg.fill_normal(torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda"), seed, 1, 0, 1.28)
    kv = sg.fill_normal(torch.empty(B, n_cap, 512, dtype=torch.bfloat16, device="cuda"), seed, 2)
    swa = sg.fill_normal(torch.empty(B, S, 512, dtype=torch.bfloat16, device="cuda"), seed, 3)
    tk = _spread_topk(B, 1, k, n_cap)
    lse = torch.empty(B, 1, H, dtype=torch.float32, device="cuda")
    out = ops.sparse_attn(q, q_pos0, kv, n_cap, Hp.to_dev(tk, torch.int32), swa, swa_pos0,
                          window=W, lse_out=lse)
    torch.cuda.synchronize()
    _ok()
    del kv
    g = Hp.bf16_of(out)
    lse = lse.cpu().numpy()
    for b in rows:
        q64 = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, b * H * 512, H * 512, 1.28)).reshape(H, 512)
        swa_b = R.bf16_to_f64(synth.normal_bf16_bits(seed, 3, b * S * 512, S * 512)).reshape(S, 512)
        rows_ = np.concatenate([_entry_rows(seed, 2, b, n_cap, tk[b, 0]),
                                R.attention_rows(np.zeros((0, 512)), [], swa_b, swa_pos0, q_pos0, W)])
        Hp.check_attention(g[b, 0], R.sparse_attention(q64, rows_, R.ATTN_SCALE, None), f"sequence {b}")
        lg = (q64 @ rows_.T) * R.ATTN_SCALE
        mx = lg.max(axis=1)
        np.testing.assert_allclose(lse[b, 0], np.log(np.exp(lg - mx[:, None]).sum(1)) + mx,
                                   rtol=1e-4, atol=1e-4)


def test_prefill_attention_full_size_sampled_rows():
    # the 16384-token encoder prefill: 64 heads over 512 selected entries + the window
    from synth import gpu as sg
    ops = _ops()
    Tq, H, n_entries, m, k, W, seed = 16384, 64, 8192, 2, 512, 128, 9700
    q = sg.fill_normal(torch.empty(1, Tq, H, 512, dtype=torch.bfloat16, device="cuda"), seed, 1, 0, 1.28)
    kv = sg.fill_normal(torch.empty(1, n_entries, 512, dtype=torch.bfloat16, device="cuda"), seed, 2)
    swa = sg.fill_normal(torch.empty(1, Tq, 512, dtype=torch.bfloat16, device="cuda"), seed, 3)
    tk = _spread_topk(1, Tq, k, [R.n_visible(i, m, n_entries) for i in range(Tq)])
    out = ops.sparse_attn(q, 0, kv, n_entries, Hp.to_dev(tk, torch.int32), swa, 0, window=W)
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    for i in (0, 1, 127, 128, 1500, 9999, 16383):
        q64 = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, i * H * 512, H * 512, 1.28)).reshape(H, 512)
        kv_rows = _entry_rows(seed, 2, 0, n_entries, tk[0, i][tk[0, i] >= 0])
        lo = max(0, i - W + 1)
        swa_rows = R.bf16_to_f64(synth.normal_bf16_bits(seed, 3, lo * 512, (i - lo + 1) * 512)).reshape(-1, 512)
        o = R.sparse_attention(q64, np.concatenate([kv_rows, swa_rows]), R.ATTN_SCALE, None)
        Hp.check_attention(g[0, i], o, f"query {i}")


# ---------------------------------------------------------------- compressor + index keys
def _check_cache_rows(got, kv_o):
    exp = R.bf16_to_f64(R.f64_to_bf16_bits(kv_o))
    rms = np.sqrt(np.mean(exp * exp, axis=-1, keepdims=True))
    bound = np.abs(exp) * 2.0 ** -7 + Hp.COMPRESS_REL * np.maximum(np.abs(exp), rms)
    assert np.all(np.abs(got - exp) <= bound), "bf16 cache beyond rounding + 1e-3 relative"


@pytest.mark.parametrize("B,T,m,n_cap", [
    (64, 2, 2, 65536),      # 40-layer decode: one new pair per sequence, encoder layers
    (64, 1, 1, 131072),     # 40-layer decode: decoder layer from its hidden state
])
def test_decode_compressor_and_index_k_full_batch(B, T, m, n_cap):
    ops = _ops()
    hidden, seed = 4096, 9850 + m
    pos0 = 131072 - T
    x, x64 = Hp.bf16_input(seed, 1, (B, T, hidden))
    wkv, wkv64 = Hp.bf16_input(seed, 2, (512, hidden), 0.02)
    wg, wg64 = Hp.bf16_input(seed, 3, (512, hidden), 0.02) if m == 2 else (None, None)
    wik, wik64 = Hp.bf16_input(seed, 4, (128, 512), 0.02)
    gam = torch.ones(512, dtype=torch.float32, device="cuda")
    cache = torch.zeros(B, n_cap, 512, dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros(B, n_cap, 64, dtype=torch.uint8, device="cuda")
    scl = torch.zeros(B, n_cap, 4, dtype=torch.uint8, device="cuda")
    e0 = pos0 // m
    pre = ops.compress(x, wkv, wg, gam, m, pos0, cache)
    ops.index_k_quant(pre, e0, m, wik, codes, scl)
    torch.cuda.synchronize()
    _ok()
    kv_o, pre_o = R.compress(x64, wkv64, wg64, np.ones(512), m, pos0)
    Hp.check_compress_f32(pre.cpu().numpy(), pre_o, "kv_pre")
    _check_cache_rows(Hp.bf16_of(cache[:, e0:e0 + 1]), kv_o)
    k_o = R.index_k(pre_o, wik64, np.full((B, 1), pos0))
    sf, cf = Hp.check_codes(codes[:, e0:e0 + 1].cpu().numpy(), scl[:, e0:e0 + 1].cpu().numpy(), k_o)
    assert sf + cf <= 4, (sf, cf)


def test_prefill_compressor_and_index_k_full_size_sampled_entries():
    # the 16384-token encoder prefill: 8192 entries (m = 2), hidden 4096
    from synth import gpu as sg
    ops = _ops()
    T, hidden, m, seed = 16384, 4096, 2, 9800
    G = T // m
    x = sg.fill_normal(torch.empty(1, T, hidden, dtype=torch.bfloat16, device="cuda"), seed, 1)
    wkv, wkv64 = Hp.bf16_input(seed, 2, (512, hidden), 0.02)
    wg, wg64 = Hp.bf16_input(seed, 3, (512, hidden), 0.02)
    wik, wik64 = Hp.bf16_input(seed, 4, (128, 512), 0.02)
    gam, gam64 = Hp.f32_input(seed, 5, (512,), 0.1)
    gam, gam64 = gam + 1.0, gam64 + 1.0
    cache = torch.zeros(1, G, 512, dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros(1, G, 64, dtype=torch.uint8, device="cuda")
    scl = torch.zeros(1, G, 4, dtype=torch.uint8, device="cuda")
    pre = ops.compress(x, wkv, wg, gam, m, 0, cache)
    ops.index_k_quant(pre, 0, m, wik, codes, scl)
    torch.cuda.synchronize()
    _ok()
    del x
    pre, kvc = pre.cpu().numpy(), Hp.bf16_of(cache)
    codes, scl = codes.cpu().numpy(), scl.cpu().numpy()
    flips = 0
    for e in (0, 1, 777, 4095, 4096, 8191):
        xg = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, e * m * hidden, m * hidden)).reshape(1, m, hidden)
        kv_o, pre_o = R.compress(xg, wkv64, wg64, gam64, m, pos0=e * m)
        Hp.check_compress_f32(pre[0, e], pre_o[0, 0], f"entry {e}")
        _check_cache_rows(kvc[0, e], kv_o[0, 0])
        k_o = R.index_k(pre_o, wik64, np.array([[e * m]]))
        sf, cf = Hp.check_codes(codes[0, e][None, None], scl[0, e][None, None], k_o)
        flips += sf + cf
    assert flips <= 4, flips


# ---------------------------------------------------------------- FP4 main KV
def _device_main_kv_fp4(seed, stream, B, n_cap):
    """Device copy of helpers.main_kv_fp4_input (same words, same bytes)."""
    from synth import gpu as sg
    r = torch.empty(B * n_cap * 72, dtype=torch.int32, device="cuda")
    sg.fill_u32(r, seed, stream)
    r8 = r.view(torch.uint8).view(B, n_cap, 288)
    codes = r8[..., :256].contiguous()
    scales = (0x28 + (r8[..., 256:] % 16)).to(torch.uint8).contiguous()
    return codes, scales


def _host_main_kv_rows(seed, stream, b, n_cap, entries):
    out = []
    for e in entries:
        w = synth.uniform_u32(seed, stream, (b * n_cap + int(e)) * 72, 72)
        by = np.ascontiguousarray(w).view(np.uint8)
        out.append(R.main_kv_dequant(by[None, :256], (0x28 + by[None, 256:] % 16).astype(np.uint8))[0])
    return np.stack(out) if out else np.zeros((0, 512))


def test_sparse_attention_fp4kv_full_size_sampled_rows():
    # 40-layer decode shape with FP4 main-KV entries: 64 rows x (512 entries + 128 window rows)
    from synth import gpu as sg
    ops = _ops()
    B, n_cap, q_pos0, H, k, W, S, seed = 64, 65536, 131071, 64, 512, 128, 256, 9660
    swa_pos0 = q_pos0 - S + 1
    q = sg.fill_normal(torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda"), seed, 1, 0, 1.28)
    codes, scales = _device_main_kv_fp4(seed, 2, B, n_cap)
    swa = sg.fill_normal(torch.empty(B, S, 512, dtype=torch.bfloat16, device="cuda"), seed, 3)
    tk = _spread_topk(B, 1, k, n_cap)
    out = ops.sparse_attn(q, q_pos0, None, n_cap, Hp.to_dev(tk, torch.int32), swa, swa_pos0,
                          window=W, kv_fp4=(codes, scales))
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    for b in (0, 29, 63):
        q64 = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, b * H * 512, H * 512, 1.28)).reshape(H, 512)
        swa_b = R.bf16_to_f64(synth.normal_bf16_bits(seed, 3, b * S * 512, S * 512)).reshape(S, 512)
        rows_ = np.concatenate([_host_main_kv_rows(seed, 2, b, n_cap, tk[b, 0]),
                                R.attention_rows(np.zeros((0, 512)), [], swa_b, swa_pos0, q_pos0, W)])
        Hp.check_attention(g[b, 0], R.sparse_attention(q64, rows_, R.ATTN_SCALE, None), f"sequence {b}")


def test_sparse_attention_fp4kv_fp8_window_full_size_sampled_rows():
    # the pages' stored formats at the 40-layer decode shape: FP4 main-KV entries and FP8
    # window rows (generator rows quantised by the oracle on the host), 64 rows x (512 + 128)
    from synth import gpu as sg
    ops = _ops()
    B, n_cap, q_pos0, H, k, W, S, seed = 64, 65536, 131071, 64, 512, 128, 256, 9661
    swa_pos0 = q_pos0 - S + 1
    q = sg.fill_normal(torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda"), seed, 1, 0, 1.28)
    codes, scales = _device_main_kv_fp4(seed, 2, B, n_cap)
    wbits = synth.normal_bf16_bits(seed, 3, 0, B * S * 512).reshape(B, S, 512)
    wc, ws = R.swa_kv_fp8(R.bf16_to_f64(wbits))
    tk = _spread_topk(B, 1, k, n_cap)
    out = ops.sparse_attn(q, q_pos0, None, n_cap, Hp.to_dev(tk, torch.int32), None, swa_pos0,
                          window=W, kv_fp4=(codes, scales),
                          swa_fp8=(Hp.to_dev(wc, torch.uint8), Hp.to_dev(ws, torch.uint8)))
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    for b in (0, 37, 63):
        q64 = R.bf16_to_f64(synth.normal_bf16_bits(seed, 1, b * H * 512, H * 512, 1.28)).reshape(H, 512)
        swa_b = R.swa_kv_dequant(wc[b], ws[b])
        rows_ = np.concatenate([_host_main_kv_rows(seed, 2, b, n_cap, tk[b, 0]),
                                R.attention_rows(np.zeros((0, 512)), [], swa_b, swa_pos0, q_pos0, W)])
        Hp.check_attention(g[b, 0], R.sparse_attention(q64, rows_, R.ATTN_SCALE, None), f"sequence {b}")


# ---------------------------------------------------------------- runner, full decoder group
def test_runner_decoder_group_full_size_sampled_sequences():
    # The decoder group of the benchmark (Full m = 1 building the HSI pool, Reindex, two Reuse
    # layers) through csa2_runner_step at its stated size: batch 32, token 65535 completing
    # entry 65535 of a 65536-entry cache (prefix entries and index keys from the generator).
    # The oracle's run_step replays sequences 0 and 31 alone (sequences are independent) from
    # the same generator rows, and every layer's top-k, the pool and the outputs are compared.
    from synth import gpu as sg
    from oracle import layers as Lr
    from test_gpu_runner import run_gpu
    B, t, n_cap, hidden, H, k, W, seed = 32, 65535, 65536, 4096, 64, 512, 128, 9900
    kv_src, idx_src, ratio = [0, 0, 0, 0], [0, 1, 1, 1], [1, 0, 0, 0]
    n0, S, swa_pos0 = t, W, t - W + 1
    kv = sg.fill_normal(torch.empty(B, n_cap, 512, dtype=torch.bfloat16, device="cuda"), seed, 20)
    codes, scales = _device_index_cache(seed, 21, B, n_cap)
    gpu, orc = [], []
    for l in range(4):
        s = seed + 10 * l
        q, q64 = Hp.bf16_input(s, 5, (B, 1, H, 512), 1.28)
        swa, swa64 = Hp.bf16_input(s, 8, (B, S, 512))
        g = dict(q=q, swa_kv=swa, swa_len=S, swa_pos0=swa_pos0, out=torch.empty_like(q))
        o = dict(q=q64, swa=swa64, swa_pos0=swa_pos0)
        if l in (0, 1):
            qi, qi64 = Hp.bf16_input(s, 6, (B, 1, 32, 128), 1.28)
            wi, wi64 = Hp.f32_input(s, 7, (B, 1, 32), 1.28)
            g.update(q_idx=qi, w_idx=wi, topk_out=None)
            o.update(q_idx=qi64, w_idx=wi64)
        if l == 0:
            x, x64 = Hp.bf16_input(s, 1, (B, 1, hidden))
            wkv, wkv64 = Hp.bf16_input(s, 2, (512, hidden), 0.02)
            wik, wik64 = Hp.bf16_input(s, 4, (128, 512), 0.02)
            gam = torch.ones(512, dtype=torch.float32, device="cuda")
            g.update(x=x, w_kv=wkv, w_gate=None, norm_w=gam, w_ik=wik, kv_cache=kv, idx_codes=codes,
                     idx_scales=scales, n_cap=n_cap, x_tokens=1, x_pos0=n0)
            o.update(x=x64, x_pos0=n0, w_kv=wkv64, w_gate=None, gamma=np.ones(512), w_ik=wik64)
        gpu.append(g)
        orc.append(o)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, gpu, B, 1, t, H, hidden, k, 64, 64)
    _ok()
    got_top = {l: topks[l].cpu().numpy() for l in topks}
    got_cand = cands[0].cpu().numpy()
    got_out = [Hp.bf16_of(g["out"]) for g in gpu]
    del kv, codes, scales
    for b in (0, 31):
        ob = []
        for l, o in enumerate(orc):
            d = {key: (v[b:b + 1] if isinstance(v, np.ndarray) and v.ndim >= 3 else v)
                 for key, v in o.items()}
            if l == 0:
                prev = synth.normal_bf16_bits(seed, 20, b * n_cap * 512, n0 * 512, 1.0)
                d["prev_kv"] = R.bf16_to_f64(prev).reshape(1, n0, 512)
                pc, ps = _host_index_rows(seed, 21, b, n_cap, n0)
                d["prev_codes"], d["prev_scales"] = pc[None], ps[None]
            ob.append(d)
        outs, trace = Lr.run_step(kv_src, idx_src, ratio, ob, 1, 1, t, k, hsi_blk=64, hsi_nb=64)
        for l in (0, 1):
            for (_, i), sc in trace[l]["scores"].items():
                Hp.check_topk_row(got_top[l][b, i], sc, trace[l]["valid"][0, i], k,
                                  f"layer {l} sequence {b}")
        np.testing.assert_array_equal(got_cand[b], trace[0]["candidates"][0])
        for l in range(4):
            Hp.check_attention(got_out[l][b:b + 1], outs[l], f"layer {l} sequence {b}")
