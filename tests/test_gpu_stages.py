"""Parity of each C-ABI entry point against the oracle, on seeded inputs both sides
draw from the generator module.  Sizes span several tiles with ragged tails."""

import numpy as np
import pytest
import torch

import synth
from oracle import csa2_ref as R
from oracle import fp4

import helpers as Hp

pytestmark = pytest.mark.gpu

cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


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


# ---------------------------------------------------------------- generator twin
def test_gpu_generator_matches_host():
    from synth import gpu as sg
    for seed, stream, start, n, sigma in [(0, 1, 0, 100_003, 1.0), (5, 9, 2**33 + 7, 4097, 0.02),
                                          (123456, 4, 17, 65536, 1.28)]:
        t = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        sg.fill_normal(t, seed, stream, start, sigma)
        host = synth.normal_bf16_bits(seed, stream, start, n, sigma)
        np.testing.assert_array_equal(t.cpu().view(torch.int16).numpy().view(np.uint16), host)
        f = torch.empty(n, dtype=torch.float32, device="cuda")
        sg.fill_normal(f, seed, stream, start, sigma)
        np.testing.assert_array_equal(f.cpu().numpy(), synth.normal_f32(seed, stream, start, n, sigma))
        u = torch.empty(n, dtype=torch.int32, device="cuda")
        sg.fill_u32(u, seed, stream, start)
        np.testing.assert_array_equal(u.cpu().numpy().view(np.uint32),
                                      synth.uniform_u32(seed, stream, start, n))


# ---------------------------------------------------------------- stage 1
@pytest.mark.parametrize("B,T,hidden,m,pos0,n_cap", [
    (1, 256, 4096, 2, 0, 128),        # config-1 like slice
    (3, 37, 192, 2, 10, 40),          # ragged: odd T, trailing token ignored, offset entries
    (2, 130, 256, 1, 7, 200),         # m = 1, rows not a multiple of the 128-row tile
    (4, 2, 4096, 2, 131070, 65536),   # a decode step: one new pair per sequence
])
def test_compress_parity(B, T, hidden, m, pos0, n_cap):
    ops = _ops()
    seed = 11 + T + m
    x, x64 = Hp.bf16_input(seed, 1, (B, T, hidden))
    wkv, wkv64 = Hp.bf16_input(seed, 2, (512, hidden), 0.02)
    wg, wg64 = Hp.bf16_input(seed, 3, (512, hidden), 0.02) if m == 2 else (None, None)
    gam, gam64 = Hp.f32_input(seed, 4, (512,), 0.1)
    gam = gam + 1.0
    gam64 = gam64 + 1.0
    cache = torch.full((B, n_cap, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    pre = ops.compress(x, wkv, wg, gam, m, pos0, cache)
    torch.cuda.synchronize()
    _ok()
    kv_o, pre_o = R.compress(x64, wkv64, wg64, gam64.astype(np.float64), m, pos0)
    Hp.check_compress_f32(pre.cpu().numpy(), pre_o, "kv_pre")
    G = T // m
    e0 = pos0 // m
    got = Hp.bf16_of(cache[:, e0:e0 + G])
    exp = R.bf16_to_f64(R.f64_to_bf16_bits(kv_o))
    # one bf16 rounding step plus the float32 compressor tolerance (1e-3 relative,
    # with the row RMS as floor for near-zero channels)
    rms = np.sqrt(np.mean(exp * exp, axis=-1, keepdims=True))
    bound = np.abs(exp) * 2.0 ** -7 + Hp.COMPRESS_REL * np.maximum(np.abs(exp), rms)
    assert np.all(np.abs(got - exp) <= bound), "bf16 cache beyond rounding + 1e-3 relative"
    assert np.mean(got == exp) > 0.99
    # rows outside the written range are untouched
    untouched = torch.ones(n_cap, dtype=torch.bool)
    untouched[e0:e0 + G] = False
    assert torch.all(cache[:, untouched.cuda()] == 7.0)


@pytest.mark.parametrize("B,T,hidden,m,pos0,n_cap,chunks", [
    (5, 6, 512, 2, 2, 16, [1] * 6),              # decode: one token per call, split-K projection
    (3, 4, 320, 2, 131070, 65538, [1] * 4),      # hidden not a multiple of 256: plain projection
    (4, 3, 4096, 1, 9, 20, [1] * 3),             # m = 1: every token completes its entry
    (2, 41, 256, 2, 4, 40, [3, 1, 2, 7, 1, 1, 9, 16, 1]),   # prefill chunks cutting groups
    (3, 130, 4096, 2, 0, 80, [129, 1]),          # chunk ends inside a group; next completes it
])
def test_compress_chunk_matches_batch(B, T, hidden, m, pos0, n_cap, chunks):
    """The compressor fed in chunks (down to one token per call), with the group state carried
    between calls, writes the entries the oracle's compressor gives over whole groups."""
    assert sum(chunks) == T
    ops = _ops()
    seed = 31 + T + m
    x, x64 = Hp.bf16_input(seed, 1, (B, T, hidden))
    wkv, wkv64 = Hp.bf16_input(seed, 2, (512, hidden), 0.02)
    wg, wg64 = Hp.bf16_input(seed, 3, (512, hidden), 0.02) if m == 2 else (None, None)
    gam, gam64 = Hp.f32_input(seed, 4, (512,), 0.1)
    gam = gam + 1.0
    gam64 = gam64 + 1.0
    cache = torch.full((B, n_cap, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    state = torch.zeros(B, 1024, dtype=torch.float32, device="cuda") if m == 2 else None
    pres = []
    t0 = 0
    for c in chunks:
        p0 = pos0 + t0
        before = cache.clone()
        pre = ops.compress_chunk(x[:, t0:t0 + c].contiguous(), wkv, wg, gam, m, p0, cache,
                                 state=state)
        torch.cuda.synchronize()
        _ok()
        first, last = p0 // m, (p0 + c) // m          # entries this chunk completes
        assert pre.shape[1] == last - first
        pres.append(pre.cpu().numpy())
        changed = set(torch.any(cache != before, dim=-1).any(dim=0).nonzero().flatten().tolist())
        assert changed <= set(range(first, last))
        t0 += c
    kv_o, pre_o = R.compress(x64, wkv64, wg64, gam64.astype(np.float64), m, pos0)
    G = T // m
    Hp.check_compress_f32(np.concatenate(pres, axis=1)[:, :G], pre_o, "kv_pre (chunked)")
    e0 = pos0 // m
    got = Hp.bf16_of(cache[:, e0:e0 + G])
    exp = R.bf16_to_f64(R.f64_to_bf16_bits(kv_o))
    rms = np.sqrt(np.mean(exp * exp, axis=-1, keepdims=True))
    bound = np.abs(exp) * 2.0 ** -7 + Hp.COMPRESS_REL * np.maximum(np.abs(exp), rms)
    assert np.all(np.abs(got - exp) <= bound), "chunked entry beyond rounding + 1e-3 relative"
    assert np.mean(got == exp) > 0.99
    untouched = torch.ones(n_cap, dtype=torch.bool)
    untouched[e0:e0 + G] = False
    assert torch.all(cache[:, untouched.cuda()] == 7.0)


def test_compress_chunk_rejects_bad_state():
    ops = _ops()
    x = torch.zeros(2, 1, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(512, 256, dtype=torch.bfloat16, device="cuda")
    gam = torch.ones(512, dtype=torch.float32, device="cuda")
    cache = torch.zeros(2, 4, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):   # m = 2 needs a state buffer
        ops.compress_chunk(x, w, w, gam, 2, 0, cache, state=None)
    with pytest.raises(RuntimeError):   # entry 4 lies beyond the 4-entry cache
        ops.compress_chunk(x, w, w, gam, 2, 9, cache, state=torch.zeros(2, 1024, device="cuda"))
    with pytest.raises(RuntimeError):   # m = 1 carries no state
        ops.compress_chunk(x, w, None, gam, 1, 0, cache, state=torch.zeros(2, 1024, device="cuda"))


# ---------------------------------------------------------------- stage 2
def _wide_range_kv(seed, B, G):
    """float32 entries whose 32-blocks span subnormal scales to saturation, with planted
    exact E2M1 midpoints (amax = 6 s, elements s * midpoint)."""
    z = synth.normal_f32(seed, 21, 0, B * G * 512).reshape(B, G, 512)
    e = (synth.uniform_u32(seed, 22, 0, B * G * 16) % 27).astype(np.int64) - 15   # 2^-15..2^11
    scale = np.ldexp(np.ones(B * G * 16, np.float32), e).reshape(B, G, 16, 1)
    v = (z.reshape(B, G, 16, 32) * scale).reshape(B, G, 512).astype(np.float32)
    # plant midpoint blocks in dims 0..31 of every 3rd entry: s = 2^-3
    s = np.float32(0.125)
    mids = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 0.0, 0.0] + [0.5] * 20,
                    np.float32) * s
    v.reshape(-1, 512)[::3, :32] = mids
    return v


def test_index_k_quant_bit_exact_quantiser():
    """W_IK copies 64 entry dims into key dims 0..63 (exact in float32) and zeros dims
    64..127: the GPU quantises exactly the generated values, so every code and scale
    must match the oracle's quantiser bit for bit."""
    ops = _ops()
    B, G, n_cap, entry0, m = 3, 301, 320, 5, 2
    v = _wide_range_kv(3, B, G)
    sel = (np.arange(64) * 7) % 512
    sel[0] = 0                                    # dims 0..31 hold the planted midpoints
    sel[1:32] = np.arange(1, 32)
    w = np.zeros((128, 512), np.float32)
    w[np.arange(64), sel] = 1.0
    w_t = Hp.to_dev(synth.f32_to_bf16_bits(w).view(np.int16), torch.int16).view(torch.bfloat16)
    kv = Hp.to_dev(v, torch.float32)
    codes = torch.zeros(B, n_cap, 64, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, n_cap, 4, dtype=torch.uint8, device="cuda")
    kout = torch.empty(B, G, 128, dtype=torch.float32, device="cuda")
    ops.index_k_quant(kv, entry0, m, w_t, codes, scales, k_out=kout)
    torch.cuda.synchronize()
    _ok()
    k_exp = np.zeros((B, G, 128), np.float32)
    k_exp[..., :64] = v[..., sel]
    np.testing.assert_array_equal(kout.cpu().numpy(), k_exp)
    oc, os_ = fp4.quantize_rows(k_exp)
    np.testing.assert_array_equal(codes[:, entry0:entry0 + G].cpu().numpy(), oc)
    np.testing.assert_array_equal(scales[:, entry0:entry0 + G].cpu().numpy(), os_)
    assert not codes[:, :entry0].any() and not codes[:, entry0 + G:].any()
    # the planted block hit every midpoint: codes of row 0 block 0
    c = fp4.unpack_codes(oc[0, 0])[:12]
    np.testing.assert_array_equal(c, [7, 0, 2, 2, 4, 4, 6, 6, 8, 14, 0, 0])


@pytest.mark.parametrize("B,G,entry0,m", [(2, 129, 0, 2), (1, 1000, 65535, 1), (4, 1, 524287, 2)])
def test_index_k_quant_parity(B, G, entry0, m):
    ops = _ops()
    seed = 40 + G
    kv, kv64 = Hp.f32_input(seed, 1, (B, G, 512))
    w, w64 = Hp.bf16_input(seed, 2, (128, 512), 0.02)
    n_cap = entry0 + G
    codes = torch.zeros(B, n_cap, 64, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, n_cap, 4, dtype=torch.uint8, device="cuda")
    kout = torch.empty(B, G, 128, dtype=torch.float32, device="cuda")
    ops.index_k_quant(kv, entry0, m, w, codes, scales, k_out=kout)
    torch.cuda.synchronize()
    _ok()
    pos = (entry0 + np.arange(G)) * m
    k_o = R.index_k(kv64, w64, np.broadcast_to(pos, (B, G)))
    g = kout.cpu().numpy().astype(np.float64)
    rms = np.sqrt(np.mean(k_o ** 2, axis=-1, keepdims=True))
    assert np.max(np.abs(g - k_o) / rms) < 1e-5
    sf, cf = Hp.check_codes(codes[:, entry0:].cpu().numpy(), scales[:, entry0:].cpu().numpy(), k_o)
    assert sf + cf <= max(2, B * G * 128 // 20000)


# ---------------------------------------------------------------- stage 3
def _indexer_inputs(seed, B, Tq, n_cap, plant_ties=True):
    """Query, weights and a random FP4 cache of n_cap rows per sequence (ties planted)."""
    qi, qi64 = Hp.bf16_input(seed, 1, (B, Tq, 32, 128), 1.28)
    w, w64 = Hp.f32_input(seed, 2, (B, Tq, 32), 1.28)
    codes, scales = Hp.index_cache_input(seed, 3, B, n_cap)
    if plant_ties:
        # duplicate some key rows: exactly equal scores, tie broken by the lower index
        for b in range(B):
            src = np.arange(0, n_cap, 37)
            dst = (src * 11 + 5) % n_cap
            codes[b, dst] = codes[b, src]
            scales[b, dst] = scales[b, src]
    return qi, qi64, w, w64, codes, scales


def _oracle_scores(qi64, w64, codes, scales, n):
    k_hat = fp4.dequantize_rows(codes[:n], scales[:n])
    qh = R.quant_query(qi64)
    return R.indexer_scores(qh, w64, k_hat)


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,m,k", [
    (3, 1, 9999, 5000, 1, 512),       # decode, m = 1, several chunks, ragged tail
    (2, 1, 20001, 10001, 2, 128),     # decode, m = 2
    (1, 1, 29999, 30000, 1, 512),     # row longer than the shared-memory staging
    (1, 300, 0, 150, 2, 64),          # causal prefill: early rows see fewer than k entries
    (2, 5, 2040, 2048, 1, 2048),      # k = 2048 (maximum)
    (2, 1, 69999, 70000, 1, 512),     # chunked selection pruned by the caller's block maxima
    (1, 3, 79997, 40000, 2, 2048),    # chunked, rows of different lengths, k = 2048
])
def test_indexer_full_parity(B, Tq, q_pos0, n_entries, m, k):
    ops = _ops()
    seed = 70 + n_entries + Tq
    # capacities that are a multiple of 64 take the TMA path, others the per-thread copies
    n_cap = n_entries + 3 if n_entries % 2 else -(-n_entries // 64) * 64 + 64
    qi, qi64, w, w64, codes, scales = _indexer_inputs(seed, B, Tq, n_cap)
    blk = 64
    nblk = -(-n_entries // blk)
    scores = torch.full((B, Tq, n_entries), np.nan, dtype=torch.float32, device="cuda")
    bmax = torch.empty(B, Tq, nblk, dtype=torch.float32, device="cuda")
    topk = ops.indexer_score_topk(qi, w, q_pos0, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, m, k, blk=blk,
                                  blockmax_out=bmax, scores_out=scores)
    torch.cuda.synchronize()
    _ok()
    topk, scores, bmax = topk.cpu().numpy(), scores.cpu().numpy(), bmax.cpu().numpy()
    swaps = 0
    for b in range(B):
        for i in range(Tq):
            nv = R.n_visible(q_pos0 + i, m, n_entries)
            so = _oracle_scores(qi64[b, i], w64[b, i], codes[b], scales[b], nv)
            if nv:
                scale_row = np.max(np.abs(so))
                assert np.max(np.abs(scores[b, i, :nv] - so)) <= 1e-5 * max(scale_row, 1e-3), "scores"
            swaps += Hp.check_topk_row(topk[b, i], so, np.ones(nv, bool), k, f"row {b},{i}")
            bm_o = R.block_max(so, nv, blk)
            np.testing.assert_allclose(bmax[b, i, :len(bm_o)], bm_o, rtol=1e-5,
                                       atol=1e-5 * max(np.max(np.abs(so)) if nv else 0, 1e-3))
            assert np.all(bmax[b, i, len(bm_o):] == -np.inf)
    assert swaps <= max(1, B * Tq // 50)


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,m,k", [
    (2, 301, 0, 150, 2, 64),        # causal prefill, two sequences, last group of 4 ragged
    (1, 1030, 0, 515, 2, 128),      # several 128-key tiles, ragged tile and group
    (2, 77, 1000, 538, 2, 256),     # a later prefill chunk (q_pos0 > 0), k above the early rows
    (1, 200, 0, 200, 1, 64),        # m = 1
])
def test_indexer_prefill_groups_parity(B, Tq, q_pos0, n_entries, m, k):
    # Prefill calls without block maxima take the grouped scorer (four queries per key
    # tile); every visible score and every top-k row is checked against the oracle.
    ops = _ops()
    seed = 90 + n_entries + Tq
    n_cap = -(-n_entries // 64) * 64 + 64        # a multiple of 64: the tensor-map path
    qi, qi64, w, w64, codes, scales = _indexer_inputs(seed, B, Tq, n_cap)
    scores = torch.full((B, Tq, n_entries), np.nan, dtype=torch.float32, device="cuda")
    topk = ops.indexer_score_topk(qi, w, q_pos0, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, m, k, scores_out=scores)
    torch.cuda.synchronize()
    _ok()
    topk, scores = topk.cpu().numpy(), scores.cpu().numpy()
    swaps = 0
    for b in range(B):
        for i in range(Tq):
            nv = R.n_visible(q_pos0 + i, m, n_entries)
            so = _oracle_scores(qi64[b, i], w64[b, i], codes[b], scales[b], nv)
            if nv:
                scale_row = np.max(np.abs(so))
                assert np.max(np.abs(scores[b, i, :nv] - so)) <= 1e-5 * max(scale_row, 1e-3), f"scores {b},{i}"
            swaps += Hp.check_topk_row(topk[b, i], so, np.ones(nv, bool), k, f"row {b},{i}")
    assert swaps <= max(1, B * Tq // 50)


def test_indexer_non_staged_no_scores_out_uses_workspace():
    ops = _ops()
    B, n_entries, k = 2, 40000, 512
    qi, qi64, w, w64, codes, scales = _indexer_inputs(5, B, 1, n_entries)
    topk = ops.indexer_score_topk(qi, w, n_entries - 1, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, 1, k)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    for b in range(B):
        so = _oracle_scores(qi64[b, 0], w64[b, 0], codes[b], scales[b], n_entries)
        Hp.check_topk_row(topk[b, 0], so, np.ones(n_entries, bool), k)


def test_indexer_long_rows_with_32_key_blocks():
    # block maxima of 32-key blocks: the top-k threshold uses its own 64-key maxima
    ops = _ops()
    B, Tq, n_entries, m, k, blk = 2, 2, 50000, 1, 256, 32
    q_pos0 = n_entries - 2
    qi, qi64, w, w64, codes, scales = _indexer_inputs(11, B, Tq, n_entries)
    nblk = -(-n_entries // blk)
    bmax = torch.empty(B, Tq, nblk, dtype=torch.float32, device="cuda")
    topk = ops.indexer_score_topk(qi, w, q_pos0, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, m, k, blk=blk,
                                  blockmax_out=bmax)
    torch.cuda.synchronize()
    _ok()
    topk, bmax = topk.cpu().numpy(), bmax.cpu().numpy()
    for b in range(B):
        for i in range(Tq):
            nv = R.n_visible(q_pos0 + i, m, n_entries)
            so = _oracle_scores(qi64[b, i], w64[b, i], codes[b], scales[b], nv)
            Hp.check_topk_row(topk[b, i], so, np.ones(nv, bool), k, f"row {b},{i}")
            bm_o = R.block_max(so, nv, blk)
            np.testing.assert_allclose(bmax[b, i, :len(bm_o)], bm_o, rtol=1e-5,
                                       atol=1e-5 * max(np.max(np.abs(so)), 1e-3))


def test_indexer_long_rows_all_tied_take_the_lowest_positions():
    # identical keys: every score ties, so the threshold admits the whole row (more
    # candidates than the list holds) and the selection must return positions 0 .. k-1
    ops = _ops()
    B, n_entries, k = 2, 40000, 512
    qi, qi64, w, w64, codes, scales = _indexer_inputs(17, B, 1, n_entries)
    codes[:] = codes[:, :1]
    scales[:] = scales[:, :1]
    bmax = torch.empty(B, 1, -(-n_entries // 64), dtype=torch.float32, device="cuda")
    topk = ops.indexer_score_topk(qi, w, n_entries - 1, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, 1, k, blk=64,
                                  blockmax_out=bmax)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    for b in range(B):
        so = _oracle_scores(qi64[b, 0], w64[b, 0], codes[b], scales[b], n_entries)
        assert np.all(so == so[0])
        np.testing.assert_array_equal(topk[b, 0], np.arange(k))


def _cand_input(seed, B, Tq, n_blocks, nb, n_vis):
    """Ascending distinct candidate blocks among the visible ones, -1 padded."""
    out = np.full((B, Tq, nb), -1, np.int32)
    nbv = -(-n_vis // 64) if np.isscalar(n_vis) else None
    r = synth.uniform_u32(seed, 30, 0, B * Tq * n_blocks).reshape(B, Tq, n_blocks)
    for b in range(B):
        for i in range(Tq):
            nbv_i = nbv if nbv is not None else -(-n_vis[i] // 64)
            order = np.argsort(r[b, i, :nbv_i], kind="stable")
            take = np.sort(order[: min(nb - (i % 3), nbv_i)])
            out[b, i, : len(take)] = take
    return out


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,m,nb,k", [
    (3, 1, 65535, 65536, 1, 64, 512),      # decode Reindex, pool of 4096
    (2, 4, 1000, 1001, 1, 10, 128),        # pool slots past the visible range (-inf)
    (1, 1, 999, 1000, 1, 2, 512),          # pool smaller than k: padding
])
def test_indexer_reindex_pool_parity(B, Tq, q_pos0, n_entries, m, nb, k):
    ops = _ops()
    blk = 64
    seed = 90 + nb
    qi, qi64, w, w64, codes, scales = _indexer_inputs(seed, B, Tq, n_entries)
    n_blocks = -(-n_entries // blk)
    nvis = [R.n_visible(q_pos0 + i, m, n_entries) for i in range(Tq)]
    cand = _cand_input(seed, B, Tq, n_blocks, nb, nvis)
    scores = torch.empty(B, Tq, nb * blk, dtype=torch.float32, device="cuda")
    topk = ops.indexer_score_topk(qi, w, q_pos0, Hp.to_dev(codes, torch.uint8),
                                  Hp.to_dev(scales, torch.uint8), n_entries, m, k,
                                  cand=Hp.to_dev(cand, torch.int32), blk=blk, scores_out=scores)
    torch.cuda.synchronize()
    _ok()
    topk = topk.cpu().numpy()
    for b in range(B):
        for i in range(Tq):
            nv = nvis[i]
            so = _oracle_scores(qi64[b, i], w64[b, i], codes[b], scales[b], nv)
            mask = R.pool_mask(cand[b, i], nv, blk, nv)
            Hp.check_topk_row(topk[b, i], so, mask, k, f"pool row {b},{i}")


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,m,blk,nb", [
    (4, 1, 131071, 131072, 1, 64, 64),
    (2, 3, 2000, 1000, 2, 8, 2048 // 8),
    (1, 2, 0, 5, 1, 4, 3),
])
def test_hsi_candidates_parity(B, Tq, q_pos0, n_entries, m, blk, nb):
    ops = _ops()
    nblk = -(-n_entries // blk)
    bm, bm64 = Hp.f32_input(7 + nblk, 1, (B, Tq, nblk))
    bm64 = bm64.copy()
    # planted ties
    bm_np = bm.cpu().numpy()
    bm_np[..., 1::5] = bm_np[..., 0::5][..., : bm_np[..., 1::5].shape[-1]]
    bm = Hp.to_dev(bm_np, torch.float32)
    bm64 = bm_np.astype(np.float64)
    cand = ops.hsi_candidates(bm, q_pos0, n_entries, m, blk, nb).cpu().numpy()
    torch.cuda.synchronize()
    _ok()
    for b in range(B):
        for i in range(Tq):
            nv = R.n_visible(q_pos0 + i, m, n_entries)
            exp = R.hsi_candidates(bm64[b, i], nv, blk, nb)
            np.testing.assert_array_equal(cand[b, i], exp)


# ---------------------------------------------------------------- stage 4
def _topk_input(seed, B, Tq, k, n_entries, holes=True):
    r = synth.uniform_u32(seed, 40, 0, B * Tq * n_entries).reshape(B, Tq, n_entries)
    out = np.full((B, Tq, k), -1, np.int32)
    for b in range(B):
        for i in range(Tq):
            take = np.sort(np.argsort(r[b, i], kind="stable")[: min(k, n_entries) - (i % 2 if holes else 0)])
            out[b, i, : len(take)] = take
    return out


@pytest.mark.parametrize("B,Tq,H,q_pos0,n_entries,k,S,swa_pos0,sink", [
    (2, 1, 64, 131071, 3000, 512, 128, 131071 - 127, False),   # decode
    (1, 40, 16, 0, 20, 128, 40, 0, False),                      # prefill, window clipped at 0
    (3, 2, 12, 500, 700, 64, 200, 370, True),                   # H not a multiple of 8, sink
    (2, 1, 8, 300, 0, 0, 128, 173, False),                      # window only (k = 0)
    # 64 heads (tensor-core path): holes + clipped window + empty tiles + sink, ragged k,
    # window only
    (1, 40, 64, 0, 20, 128, 40, 0, True),
    (2, 3, 64, 500, 700, 300, 200, 370, False),
    (2, 1, 64, 300, 0, 0, 128, 173, True),
    # fewer heads on the tensor-core path (query rows past H are zero in its 64-row tile):
    # 16 heads at the decode batch (two CTAs per row) with a sink, 32 heads over a prefill chunk
    (64, 1, 16, 131071, 3000, 512, 128, 131071 - 127, True),
    (3, 5, 32, 900, 800, 200, 256, 700, False),
    # more rows than SMs: one persistent CTA per SM walks several rows (window rows gathered,
    # rows of different lengths, 64 and 16 heads)
    (1, 400, 64, 0, 300, 128, 400, 0, True),
    (200, 1, 64, 4095, 2000, 256, 128, 4095 - 127, False),
    (1, 300, 16, 500, 700, 64, 720, 100, False),
    # enough rows for one CTA per row, and the decode batch (two CTAs per row)
    (80, 1, 64, 4095, 2000, 256, 128, 4095 - 127, False),
    (64, 1, 64, 131071, 3000, 512, 128, 131071 - 127, True),
])
def test_sparse_attn_parity(B, Tq, H, q_pos0, n_entries, k, S, swa_pos0, sink):
    ops = _ops()
    seed = 120 + H + k
    q, q64 = Hp.bf16_input(seed, 1, (B, Tq, H, 512), 1.28)
    n_cap = max(n_entries, 1) + 2
    kv, kv64 = Hp.bf16_input(seed, 2, (B, n_cap, 512))
    swa, swa64 = Hp.bf16_input(seed, 3, (B, S, 512))
    topk_np = _topk_input(seed, B, Tq, k, n_entries) if k else None
    sk, sk64 = Hp.f32_input(seed, 4, (H,)) if sink else (None, None)
    lse = torch.empty(B, Tq, H, dtype=torch.float32, device="cuda")
    out = ops.sparse_attn(q, q_pos0, kv if k else None, n_entries,
                          Hp.to_dev(topk_np, torch.int32) if k else None, swa, swa_pos0,
                          window=128, sink=sk, lse_out=lse)
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    for b in range(B):
        for i in range(Tq):
            t = q_pos0 + i
            sel = topk_np[b, i] if k else []
            rows = R.attention_rows(kv64[b], sel, swa64[b], swa_pos0, t, 128)
            o = R.sparse_attention(q64[b, i], rows, R.ATTN_SCALE, sk64)
            Hp.check_attention(g[b, i], o, f"row {b},{i}")
            lg = (q64[b, i] @ rows.T) * R.ATTN_SCALE
            mx = lg.max(axis=1)
            if sink:
                mx = np.maximum(mx, sk64)
            l_o = np.log(np.exp(lg - mx[:, None]).sum(1) + (np.exp(sk64 - mx) if sink else 0)) + mx
            np.testing.assert_allclose(lse[b, i].cpu().numpy(), l_o, rtol=1e-4, atol=1e-4)


def _bf16_dev(x64):
    bits = R.f64_to_bf16_bits(x64)
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16), R.bf16_to_f64(bits)


@pytest.mark.parametrize("B", [1, 64])
def test_sparse_attn_rising_logits_move_the_running_max(B):
    # logits rise by about 50 (log2 units) from one 64-row chunk to the next, so every
    # chunk moves each head's running maximum and rescales what was accumulated so far
    ops = _ops()
    H, k, n_entries, S, t = 64, 512, 1024, 128, 2047
    g = np.random.default_rng(7)   # seeded structure on top of the synthetic streams
    u = np.zeros(512); u[0] = 1.0
    e = np.arange(n_entries)
    kv64 = np.empty((B, n_entries, 512))
    kv64[:] = 0.1 * g.standard_normal((B, n_entries, 512))
    kv64[:, :, 0] = e / n_entries
    swa64 = 0.1 * g.standard_normal((B, S, 512))
    swa64[:, :, 0] = -0.5
    gamma = np.linspace(400.0, 800.0, H) * np.sqrt(512)
    q64 = np.zeros((B, 1, H, 512))
    q64[:, 0] = gamma[:, None] * u[None, :] + 0.05 * g.standard_normal((B, H, 512))
    q, q64 = _bf16_dev(q64)
    kv, kv64 = _bf16_dev(kv64)
    swa, swa64 = _bf16_dev(swa64)
    topk_np = np.broadcast_to(np.arange(k, dtype=np.int32), (B, 1, k)).copy()
    out = ops.sparse_attn(q, t, kv, n_entries, Hp.to_dev(topk_np, torch.int32), swa, t - 127,
                          window=128)
    torch.cuda.synchronize()
    _ok()
    gout = Hp.bf16_of(out)
    for b in range(B):
        rows = R.attention_rows(kv64[b], topk_np[b, 0], swa64[b], t - 127, t, 128)
        Hp.check_attention(gout[b, 0], R.sparse_attention(q64[b, 0], rows, R.ATTN_SCALE, None),
                           f"row {b}")


def test_sparse_attn_out_of_range_index_is_reported_and_skipped():
    ops = _ops()
    B, H, n_entries, k = 1, 8, 100, 16
    q, q64 = Hp.bf16_input(1, 1, (B, 1, H, 512))
    kv, kv64 = Hp.bf16_input(1, 2, (B, n_entries, 512))
    swa, swa64 = Hp.bf16_input(1, 3, (B, 128, 512))
    tk = np.full((B, 1, k), -1, np.int32)
    tk[0, 0, :3] = [5, 50, 100]           # 100 == n_entries: out of range
    out = ops.sparse_attn(q, 127, kv, n_entries, Hp.to_dev(tk, torch.int32), swa, 0)
    assert ops.last_device_status() == 6          # CSA2_ERR_DEVICE_CHECK
    assert ops.last_device_status() == 0          # cleared after reading
    rows = R.attention_rows(kv64[0], [5, 50], swa64[0], 0, 127, 128)
    Hp.check_attention(Hp.bf16_of(out)[0, 0], R.sparse_attention(q64[0, 0], rows))


# ---------------------------------------------------------------- FP4 main KV
def test_main_kv_quant_fp4_bit_exact():
    """The quantiser reads the stored bf16 entries; both sides decide in float32, so every
    code and scale matches; rows outside the range stay untouched."""
    ops = _ops()
    B, n_cap, entry0, G = 3, 300, 7, 250
    v = synth.normal_f32(61, 1, 0, B * n_cap * 512).reshape(B, n_cap, 512)
    v *= np.exp2((synth.uniform_u32(61, 2, 0, B * n_cap * 32) % 24).astype(np.float32) - 12.0).reshape(
        B, n_cap, 32).repeat(16, axis=-1)                    # groups spanning 2^-12 .. 2^11
    bits = synth.f32_to_bf16_bits(v.astype(np.float32))
    kv = Hp.to_dev(bits.view(np.int16), torch.int16).view(torch.bfloat16)
    codes = torch.zeros(B, n_cap, 256, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, n_cap, 32, dtype=torch.uint8, device="cuda")
    ops.main_kv_quant_fp4(kv, entry0, G, codes, scales)
    torch.cuda.synchronize()
    _ok()
    oc, os_ = R.main_kv_fp4(R.bf16_to_f64(bits[:, entry0:entry0 + G]))
    np.testing.assert_array_equal(codes[:, entry0:entry0 + G].cpu().numpy(), oc)
    np.testing.assert_array_equal(scales[:, entry0:entry0 + G].cpu().numpy(), os_)
    assert not codes[:, :entry0].any() and not codes[:, entry0 + G:].any()
    assert not scales[:, :entry0].any() and not scales[:, entry0 + G:].any()


def test_swa_kv_quant_fp8_bit_exact():
    """Window rows to FP8: the scale exponent and every E4M3 code match the oracle bit for
    bit (the element decision is on an exact product); rows outside the range untouched."""
    ops = _ops()
    B, S, row0, n = 3, 200, 5, 180
    v = synth.normal_f32(62, 1, 0, B * S * 512).reshape(B, S, 512)
    v *= np.exp2((synth.uniform_u32(62, 2, 0, B * S * 8) % 40).astype(np.float32) - 20.0).reshape(
        B, S, 8).repeat(64, axis=-1)                      # groups spanning 2^-20 .. 2^19
    v[0, 10, 64:128] = 0.0                                # an all-zero group
    v[1, 11, :64] = 0.0
    v[1, 11, 3] = 448.0 * 2.0 ** -5                       # amax exactly on a power-of-two bound
    v[2, 12, 128:192] *= 2.0 ** -110                      # bf16 subnormal elements
    bits = synth.f32_to_bf16_bits(v.astype(np.float32))
    swa = Hp.to_dev(bits.view(np.int16), torch.int16).view(torch.bfloat16)
    codes = torch.zeros(B, S, 512, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(B, S, 8, dtype=torch.uint8, device="cuda")
    ops.swa_kv_quant_fp8(swa, row0, n, codes, scales)
    torch.cuda.synchronize()
    _ok()
    oc, os_ = R.swa_kv_fp8(R.bf16_to_f64(bits[:, row0:row0 + n]))
    np.testing.assert_array_equal(scales[:, row0:row0 + n].cpu().numpy(), os_)
    np.testing.assert_array_equal(codes[:, row0:row0 + n].cpu().numpy(), oc)
    assert not codes[:, :row0].any() and not codes[:, row0 + n:].any()
    assert not scales[:, :row0].any() and not scales[:, row0 + n:].any()


def _swa_fp8_input(seed, stream, B, S):
    """Window rows as FP8: generator bf16 rows quantised by the oracle (host side)."""
    bits = synth.normal_bf16_bits(seed, stream, 0, B * S * 512).reshape(B, S, 512)
    codes, scales = R.swa_kv_fp8(R.bf16_to_f64(bits))
    return codes, scales


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,k,S,swa_pos0,main", [
    (2, 1, 131071, 3000, 512, 128, 131071 - 127, "fp4"),   # decode, the pages' stored formats
    (2, 1, 131071, 3000, 512, 128, 131071 - 127, "bf16"),  # FP8 window, bf16 entries
    (1, 40, 0, 20, 128, 40, 0, "fp4"),                     # prefill, window clipped at 0
    (3, 2, 500, 700, 300, 200, 370, "bf16"),               # odd sizes, masked slots
    (2, 3, 1000, 0, 0, 140, 870, None),                    # window only (k = 0)
])
def test_sparse_attn_fp8_window_parity(B, Tq, q_pos0, n_entries, k, S, swa_pos0, main):
    ops = _ops()
    H, seed = 64, 170 + n_entries
    q, q64 = Hp.bf16_input(seed, 1, (B, Tq, H, 512), 1.28)
    wc, ws = _swa_fp8_input(seed, 3, B, S)
    swa64 = R.swa_kv_dequant(wc, ws)
    kv_fp4, kv, kv64, topk = None, None, None, None
    topk_np = np.zeros((B, Tq, 0), np.int32)
    if main == "fp4":
        codes, scales = Hp.main_kv_fp4_input(seed, 2, B, n_entries)
        kv_fp4 = (Hp.to_dev(codes, torch.uint8), Hp.to_dev(scales, torch.uint8))
        kv64 = R.main_kv_dequant(codes, scales)
    elif main == "bf16":
        kv, kv64 = Hp.bf16_input(seed, 2, (B, n_entries, 512))
    if main is not None:
        topk_np = _topk_input(seed, B, Tq, k, n_entries)
        topk = Hp.to_dev(topk_np, torch.int32)
    lse = torch.empty(B, Tq, H, dtype=torch.float32, device="cuda")
    out = ops.sparse_attn(q, q_pos0, kv, n_entries, topk, None, swa_pos0, window=128, lse_out=lse,
                          kv_fp4=kv_fp4,
                          swa_fp8=(Hp.to_dev(wc, torch.uint8), Hp.to_dev(ws, torch.uint8)))
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    lse = lse.cpu().numpy()
    for b in range(B):
        for i in range(Tq):
            t = q_pos0 + i
            ent = kv64[b] if kv64 is not None else np.zeros((0, 512))
            rows = R.attention_rows(ent, topk_np[b, i], swa64[b], swa_pos0, t)
            Hp.check_attention(g[b, i], R.sparse_attention(q64[b, i], rows, R.ATTN_SCALE, None),
                               f"row {b},{i}")
            lg = (q64[b, i] @ rows.T) * R.ATTN_SCALE
            mx = lg.max(axis=1)
            np.testing.assert_allclose(lse[b, i], np.log(np.exp(lg - mx[:, None]).sum(1)) + mx,
                                       rtol=1e-4, atol=1e-4)


def test_sparse_attn_ex_rejects_ambiguous_operands():
    ops = _ops()
    from compressed_sparse_attention_04_gb300 import _lib as L
    lib = L.load()
    q = torch.zeros(1, 1, 64, 512, dtype=torch.bfloat16, device="cuda")
    swa = torch.zeros(1, 8, 512, dtype=torch.bfloat16, device="cuda")
    wc = torch.zeros(1, 8, 512, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(1, 8, 8, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    p = lambda t: ops._p(t)
    # both forms of the window rows
    st = lib.csa2_sparse_attn_ex(p(q), 1, 1, 64, 7, p(None), p(None), p(None), 0, 0, p(None), 0,
                                 p(swa), p(wc), p(ws), 8, 0, 8, p(None), 0.05, p(out), p(None),
                                 p(None), 0, ops._stream(q.device))
    assert st == L.ERR_INVALID_ARG
    # neither form
    st = lib.csa2_sparse_attn_ex(p(q), 1, 1, 64, 7, p(None), p(None), p(None), 0, 0, p(None), 0,
                                 p(None), p(None), p(None), 8, 0, 8, p(None), 0.05, p(out), p(None),
                                 p(None), 0, ops._stream(q.device))
    assert st == L.ERR_INVALID_ARG
    # quantised rows need the tensor-core kernel: H a multiple of 8 up to 64
    q12 = torch.zeros(1, 1, 12, 512, dtype=torch.bfloat16, device="cuda")
    st = lib.csa2_sparse_attn_ex(p(q12), 1, 1, 12, 7, p(None), p(None), p(None), 0, 0, p(None), 0,
                                 p(None), p(wc), p(ws), 8, 0, 8, p(None), 0.05, p(q12), p(None),
                                 p(None), 0, ops._stream(q.device))
    assert st == L.ERR_UNSUPPORTED


@pytest.mark.parametrize("H", [16, 32])
def test_sparse_attn_fewer_heads_quantised_rows_equal_their_bf16_values(H):
    # With fewer than 64 heads the stored formats run on the same tensor-core kernel: FP8
    # window rows and FP4 entries dequantise exactly into the bf16 tile, so the output equals,
    # bit for bit, the bf16 path over the dequantised values (computed by the oracle's
    # decoders on the host).
    ops = _ops()
    B, Tq, q_pos0, n_entries, k, S = 64, 1, 131071, 1500, 512, 128
    swa_pos0 = q_pos0 - 127
    seed = 260 + H
    q, _ = Hp.bf16_input(seed, 1, (B, Tq, H, 512), 1.28)
    kv_b, kv64 = Hp.bf16_input(seed, 2, (B, n_entries, 512))
    swa_b, swa64 = Hp.bf16_input(seed, 3, (B, S, 512))
    kc, ks = R.main_kv_fp4(kv64)
    wc, wsc = R.swa_kv_fp8(swa64)
    kv_deq, _ = _bf16_dev(R.main_kv_dequant(kc, ks))
    swa_deq, _ = _bf16_dev(R.swa_kv_dequant(wc, wsc))
    topk = Hp.to_dev(_topk_input(seed, B, Tq, k, n_entries), torch.int32)
    quant = ops.sparse_attn(q, q_pos0, None, n_entries, topk, None, swa_pos0, window=128,
                            kv_fp4=(Hp.to_dev(kc, torch.uint8), Hp.to_dev(ks, torch.uint8)),
                            swa_fp8=(Hp.to_dev(wc, torch.uint8), Hp.to_dev(wsc, torch.uint8)))
    plain = ops.sparse_attn(q, q_pos0, kv_deq, n_entries, topk, swa_deq, swa_pos0, window=128)
    torch.cuda.synchronize()
    _ok()
    np.testing.assert_array_equal(quant.view(torch.int16).cpu().numpy(),
                                  plain.view(torch.int16).cpu().numpy())


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,k,S,swa_pos0", [
    (2, 1, 131071, 3000, 512, 128, 131071 - 127),   # decode: 512 entries + 128 window rows
    (1, 40, 0, 20, 128, 40, 0),                     # prefill, window clipped at 0
    (3, 2, 500, 700, 300, 200, 370),                # odd sizes, masked slots
])
def test_sparse_attn_fp4kv_parity(B, Tq, q_pos0, n_entries, k, S, swa_pos0):
    ops = _ops()
    H, seed = 64, 130 + n_entries
    q, q64 = Hp.bf16_input(seed, 1, (B, Tq, H, 512), 1.28)
    codes, scales = Hp.main_kv_fp4_input(seed, 2, B, n_entries)
    swa, swa64 = Hp.bf16_input(seed, 3, (B, S, 512))
    topk_np = _topk_input(seed, B, Tq, k, n_entries)
    lse = torch.empty(B, Tq, H, dtype=torch.float32, device="cuda")
    out = ops.sparse_attn(q, q_pos0, None, n_entries, Hp.to_dev(topk_np, torch.int32), swa, swa_pos0,
                          window=128, lse_out=lse,
                          kv_fp4=(Hp.to_dev(codes, torch.uint8), Hp.to_dev(scales, torch.uint8)))
    torch.cuda.synchronize()
    _ok()
    g = Hp.bf16_of(out)
    lse = lse.cpu().numpy()
    kv64 = R.main_kv_dequant(codes, scales)
    for b in range(B):
        for i in range(Tq):
            t = q_pos0 + i
            rows = R.attention_rows(kv64[b], topk_np[b, i], swa64[b], swa_pos0, t)
            Hp.check_attention(g[b, i], R.sparse_attention(q64[b, i], rows, R.ATTN_SCALE, None),
                               f"row {b},{i}")
            lg = (q64[b, i] @ rows.T) * R.ATTN_SCALE
            mx = lg.max(axis=1)
            np.testing.assert_allclose(lse[b, i], np.log(np.exp(lg - mx[:, None]).sum(1)) + mx,
                                       rtol=1e-4, atol=1e-4)
