"""Full / Reindex / Reuse runtime through csa2_runner_step vs the oracle's run_step,
end to end from seeded hidden states (no value crosses from the GPU into the oracle)."""

import numpy as np
import pytest
import torch

from oracle import csa2_ref as R
from oracle import layers as Lr

import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from compressed_sparse_attention_04_gb300 import build
    build.build_all()


def make_stack(kv_src, idx_src, ratio, B, Tq, q_pos0, n0_tokens, hidden, H, seed0, S_extra=0,
               window=128, stored_formats=False):
    """Per-layer inputs for both sides.  Full layers get hidden states for tokens
    0..q_pos0+Tq-1: the prefix 0..n0_tokens-1 is compressed beforehand (GPU: by the
    stage calls; oracle: by its own compressor), the rest is the step's input.
    stored_formats: FP4 main KV and FP8 window rows; the prefix entries' FP4 form and the
    window rows' FP8 form come from the oracle's quantisers on the host."""
    from compressed_sparse_attention_04_gb300 import ops
    gpu, orc = [], []
    T_all = q_pos0 + Tq
    swa_pos0 = max(0, q_pos0 - window + 1) - S_extra
    swa_pos0 = max(0, swa_pos0)
    S = T_all - swa_pos0
    for l in range(len(kv_src)):
        s = seed0 + l
        q, q64 = Hp.bf16_input(s, 5, (B, Tq, H, 512), 1.28)
        swa, swa64 = Hp.bf16_input(s, 8, (B, S, 512))
        g = dict(q=q, swa_kv=swa, swa_len=S, swa_pos0=swa_pos0, out=torch.empty_like(q))
        if stored_formats:
            wc, ws_ = R.swa_kv_fp8(swa64)
            g.update(swa_kv=None, swa_codes=Hp.to_dev(wc, torch.uint8),
                     swa_scales=Hp.to_dev(ws_, torch.uint8))
        o = dict(q=q64, swa=swa64, swa_pos0=swa_pos0)
        if kv_src[l] == l or idx_src[l] == l:
            qi, qi64 = Hp.bf16_input(s, 6, (B, Tq, 32, 128), 1.28)
            wi, wi64 = Hp.f32_input(s, 7, (B, Tq, 32), 1.28)
            g.update(q_idx=qi, w_idx=wi, topk_out=None)
            o.update(q_idx=qi64, w_idx=wi64)
        if kv_src[l] == l:
            m = ratio[l]
            x, x64 = Hp.bf16_input(s, 1, (B, T_all, hidden))
            wkv, wkv64 = Hp.bf16_input(s, 2, (512, hidden), 0.02)
            wg, wg64 = Hp.bf16_input(s, 3, (512, hidden), 0.02) if m == 2 else (None, None)
            wik, wik64 = Hp.bf16_input(s, 4, (128, 512), 0.02)
            gam = torch.ones(512, dtype=torch.float32, device="cuda")
            n0 = n0_tokens // m
            n_cap = T_all // m + 1
            cache = torch.zeros(B, n_cap, 512, dtype=torch.bfloat16, device="cuda")
            codes = torch.zeros(B, n_cap, 64, dtype=torch.uint8, device="cuda")
            scl = torch.zeros(B, n_cap, 4, dtype=torch.uint8, device="cuda")
            if n0 > 0:
                pre = ops.compress(x[:, : n0 * m].contiguous(), wkv, wg, gam, m, 0, cache)
                ops.index_k_quant(pre, 0, m, wik, codes, scl)
            xs = x[:, n0 * m:].contiguous()
            g.update(x=xs, w_kv=wkv, w_gate=wg, norm_w=gam, w_ik=wik, kv_cache=cache,
                     idx_codes=codes, idx_scales=scl, n_cap=n_cap, x_tokens=xs.shape[1],
                     x_pos0=n0 * m)
            kv_p, pre_p = R.compress(x64[:, : n0 * m], wkv64, wg64, np.ones(512), m)
            pos = m * np.arange(n0)
            c, sc = R.index_k_quant(R.index_k(pre_p, wik64, np.broadcast_to(pos, (B, n0))))
            if stored_formats:
                kc = np.zeros((B, n_cap, 256), np.uint8)
                ks = np.zeros((B, n_cap, 32), np.uint8)
                if n0 > 0:
                    kc[:, :n0], ks[:, :n0] = R.main_kv_fp4(R.bf16_to_f64(R.f64_to_bf16_bits(kv_p)))
                g.update(kv_codes=Hp.to_dev(kc, torch.uint8), kv_scales=Hp.to_dev(ks, torch.uint8))
            o.update(x=x64[:, n0 * m:], x_pos0=n0 * m, w_kv=wkv64, w_gate=wg64,
                     gamma=np.ones(512), w_ik=wik64,
                     prev_kv=R.bf16_to_f64(R.f64_to_bf16_bits(kv_p)), prev_codes=c,
                     prev_scales=sc)
        gpu.append(g)
        orc.append(o)
    return gpu, orc


def run_gpu(kv_src, idx_src, ratio, gpu_layers, B, Tq, q_pos0, H, hidden, k, blk, nb,
            window=128):
    from compressed_sparse_attention_04_gb300 import ops
    runner = ops.Runner(kv_src, idx_src, ratio, hsi_blk=blk, hsi_nb=nb)
    p = runner.params(B, Tq, q_pos0, H, hidden, k, window)
    topks, cands = {}, {}
    ios = []
    for l, g in enumerate(gpu_layers):
        md = runner.mode(l)
        if md in (1, 2):
            topks[l] = torch.full((B, Tq, k), -7, dtype=torch.int32, device="cuda")
            g["topk_out"] = topks[l]
        if md == 1:
            cands[l] = torch.full((B, Tq, nb), -7, dtype=torch.int32, device="cuda")
            g["cand_out"] = cands[l]
        ios.append(ops.layer_io(**g))
    max_x = max([g.get("x_tokens", 0) for g in gpu_layers] + [0])
    max_n = max([(g["x_pos0"] + g["x_tokens"]) // ratio[l]
                 for l, g in enumerate(gpu_layers) if "x_tokens" in g] + [0])
    ws = torch.empty(runner.workspace_size(p, max_x, max_n) + 256, dtype=torch.uint8, device="cuda")
    runner.step(p, ios, ws)
    torch.cuda.synchronize()
    assert ops.last_device_status() == 0
    return runner, topks, cands


def compare(kv_src, idx_src, ratio, gpu_layers, orc_layers, B, Tq, q_pos0, k, blk, nb, topks,
            cands, stored_formats=False):
    outs, trace = Lr.run_step(kv_src, idx_src, ratio, orc_layers, B, Tq, q_pos0, k, hsi_blk=blk,
                              hsi_nb=nb, main_kv_fp4=stored_formats, swa_fp8=stored_formats)
    modes = Lr.layer_modes(kv_src, idx_src)
    worst = 0.0
    for l, md in enumerate(modes):
        if md in (Lr.FULL, Lr.REINDEX):
            got = topks[l].cpu().numpy()
            for (b, i), sc in trace[l]["scores"].items():
                Hp.check_topk_row(got[b, i], sc, trace[l]["valid"][b, i], k, f"layer {l} row {b},{i}")
        if l in cands and "candidates" in trace[l]:
            np.testing.assert_array_equal(cands[l].cpu().numpy(), trace[l]["candidates"])
        mx, mean = Hp.check_attention(Hp.bf16_of(gpu_layers[l]["out"]), outs[l], f"layer {l}")
        worst = max(worst, mx)
    return worst


def test_runner_prefill_full_and_reuse():
    # one Full layer (m = 2) then two Reuse layers, causal prefill of 256 tokens
    kv_src, idx_src, ratio = [0, 0, 0], [0, 0, 0], [2, 0, 0]
    B, T, hidden, H, k = 1, 256, 256, 16, 32
    g, o = make_stack(kv_src, idx_src, ratio, B, T, 0, 0, hidden, H, seed0=500)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, T, 0, H, hidden, k, 64, 64)
    compare(kv_src, idx_src, ratio, g, o, B, T, 0, k, 64, 64, topks, cands)


def test_runner_decode_mixed_pattern():
    # SWA-only, encoder-style Full m=2 + Reuse, decoder-style Full m=1 + Reindex (HSI) + Reuse
    kv_src = [-1, 1, 1, 1, 4, 4, 4, 4, 4, 4, 4]
    idx_src = [-1, 1, 1, 1, 4, 4, 6, 6, 8, 8, 8]
    ratio = [0, 2, 0, 0, 1, 0, 0, 0, 0, 0, 0]
    B, Tq, hidden, H, k, blk, nb = 2, 1, 128, 8, 48, 16, 8
    C = 1200                                   # context incl. the current token
    q_pos0 = C - 1
    g, o = make_stack(kv_src, idx_src, ratio, B, Tq, q_pos0, q_pos0 - 1, hidden, H, seed0=700)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, Tq, q_pos0, H, hidden, k, blk, nb)
    compare(kv_src, idx_src, ratio, g, o, B, Tq, q_pos0, k, blk, nb, topks, cands)


def test_runner_config1_single_full_layer():
    """Config 1 at full size: one Full layer, prefill of 1024 tokens, hidden 4096,
    m = 2 (512 entries), top-128, window 128, 16 heads, seed 0."""
    kv_src, idx_src, ratio = [0], [0], [2]
    B, T, hidden, H, k = 1, 1024, 4096, 16, 128
    g, o = make_stack(kv_src, idx_src, ratio, B, T, 0, 0, hidden, H, seed0=0)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, T, 0, H, hidden, k, 64, 64)
    compare(kv_src, idx_src, ratio, g, o, B, T, 0, k, 64, 64, topks, cands)


def test_runner_decode_hsi_8_key_blocks():
    """The HSI variant with 8-entry blocks and 2048 candidate blocks (16 384-entry pools):
    decoder Full m = 1 builds the pool, a Reindex layer rescores inside it, a Reuse layer
    reads its selection; 20 000 entries so the pool is a real subset."""
    kv_src, idx_src, ratio = [0, 0, 0], [0, 1, 1], [1, 0, 0]
    B, Tq, hidden, H, k, blk, nb = 1, 1, 128, 8, 512, 8, 2048
    C = 20000
    q_pos0 = C - 1
    g, o = make_stack(kv_src, idx_src, ratio, B, Tq, q_pos0, q_pos0, hidden, H, seed0=900)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, Tq, q_pos0, H, hidden, k, blk, nb)
    compare(kv_src, idx_src, ratio, g, o, B, Tq, q_pos0, k, blk, nb, topks, cands)


def test_runner_decode_stored_formats():
    """The pages' stored formats through the runner: FP4 main KV (the Full layers quantise
    their new entries) and FP8 window rows, 64 heads, encoder-style Full m = 2 + Reuse and
    decoder-style Full m = 1 + Reindex + Reuse."""
    kv_src = [-1, 1, 1, 3, 3, 3]
    idx_src = [-1, 1, 1, 3, 4, 4]
    ratio = [0, 2, 0, 1, 0, 0]
    B, Tq, hidden, H, k, blk, nb = 2, 1, 256, 64, 64, 16, 8
    C = 900
    q_pos0 = C - 1
    g, o = make_stack(kv_src, idx_src, ratio, B, Tq, q_pos0, q_pos0 - 1, hidden, H, seed0=950,
                      stored_formats=True)
    runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, Tq, q_pos0, H, hidden, k, blk, nb)
    # the step's new entries in FP4 against the oracle's quantiser of the oracle's own new
    # entries (both from the seeded hidden states; the bf16 entries agree to within one bf16
    # ulp, so a code may differ where that ulp crosses a rounding boundary)
    for l in (1, 3):
        m = ratio[l]
        kv_new, _ = R.compress(o[l]["x"], o[l]["w_kv"], o[l]["w_gate"], o[l]["gamma"], m,
                               o[l]["x_pos0"])
        oc, os_ = R.main_kv_fp4(R.bf16_to_f64(R.f64_to_bf16_bits(kv_new)))
        e0 = g[l]["x_pos0"] // m
        e1 = e0 + kv_new.shape[1]
        assert np.mean(g[l]["kv_codes"][:, e0:e1].cpu().numpy() == oc) > 0.98
        assert np.mean(g[l]["kv_scales"][:, e0:e1].cpu().numpy() == os_) > 0.98
    compare(kv_src, idx_src, ratio, g, o, B, Tq, q_pos0, k, blk, nb, topks, cands,
            stored_formats=True)


def test_runner_streaming_compressor_one_token_per_step():
    """Decode with m = 2 one token per step through the runner's group state: the first
    step holds its token back (no new entry), the second completes the entry; both steps
    match the oracle's step over the same tokens."""
    kv_src, idx_src, ratio = [0, 0], [0, 0], [2, 0]
    B, Tq, hidden, H, k = 2, 1, 128, 8, 32
    P = 600                                            # first token of a new group
    g, o = make_stack(kv_src, idx_src, ratio, B, Tq, P + 1, P, hidden, H, seed0=990, S_extra=1)
    x2, x2_64 = g[0]["x"], o[0]["x"]                   # tokens P and P + 1
    assert x2.shape[1] == 2 and g[0]["x_pos0"] == P
    state = torch.zeros(B, 1024, dtype=torch.float32, device="cuda")
    e_new = P // 2
    for step, t in enumerate((P, P + 1)):
        g[0].update(x=x2[:, step:step + 1].contiguous(), x_pos0=t, x_tokens=1, compress_state=state)
        before = g[0]["kv_cache"][:, e_new].clone()
        runner, topks, cands = run_gpu(kv_src, idx_src, ratio, g, B, Tq, t, H, hidden, k, 64, 64)
        if step == 0:   # the group is incomplete: its entry is not written yet
            assert torch.equal(g[0]["kv_cache"][:, e_new], before)
        o1 = [dict(o[0], x=x2_64[:, : step + 1], x_pos0=P), o[1]]
        compare(kv_src, idx_src, ratio, g, o1, B, Tq, t, k, 64, 64, topks, cands)


@pytest.mark.parametrize("m,B,x_tokens,pos0,use_state", [
    (2, 8, 2, 1022, False),     # encoder decode step: one new entry per sequence
    (1, 8, 1, 511, False),      # decoder decode step
    (2, 4, 4, 1021, True),      # group state: completes an open group, leaves one open
    (2, 3, 2732, 0, False),     # 4098 entries: above the fused limit, separate indexer-key kernel
])
def test_runner_index_keys_equal_the_separate_stage_calls(m, B, x_tokens, pos0, use_state):
    # The runner writes decode-sized calls' indexer keys from the compressor's epilogue; the
    # entries and keys it leaves in the caches equal, bit for bit, csa2_compress(_chunk)
    # followed by csa2_index_k_quant on the same inputs.
    from compressed_sparse_attention_04_gb300 import ops
    hidden, H, k = 512, 64, 16
    s = 870 + m + x_tokens
    x, _ = Hp.bf16_input(s, 1, (B, x_tokens, hidden))
    wkv, _ = Hp.bf16_input(s, 2, (512, hidden), 0.02)
    wg = Hp.bf16_input(s, 3, (512, hidden), 0.02)[0] if m == 2 else None
    wik, _ = Hp.bf16_input(s, 4, (128, 512), 0.02)
    gam = torch.ones(512, dtype=torch.float32, device="cuda")
    n_cap = (pos0 + x_tokens) // m + 2
    st0 = None
    if use_state:   # the open group's first token, as a previous call would leave it
        st0 = Hp.f32_input(s, 9, (B, 1024))[0]
    caches = []
    for _ in range(2):
        caches.append(dict(kv=torch.zeros(B, n_cap, 512, dtype=torch.bfloat16, device="cuda"),
                           codes=torch.zeros(B, n_cap, 64, dtype=torch.uint8, device="cuda"),
                           scales=torch.zeros(B, n_cap, 4, dtype=torch.uint8, device="cuda"),
                           state=st0.clone() if use_state else None))
    # separate stage calls
    a = caches[0]
    e0 = pos0 // m
    if use_state:
        pre = ops.compress_chunk(x, wkv, wg, gam, m, pos0, a["kv"], state=a["state"])
    else:
        pre = ops.compress(x, wkv, wg, gam, m, pos0, a["kv"])
    ops.index_k_quant(pre, e0, m, wik, a["codes"], a["scales"])
    # the runner (one Full layer; its attention output is not compared here)
    b_ = caches[1]
    Tq = 1
    q = Hp.bf16_input(s, 5, (B, Tq, H, 512), 1.28)[0]
    t_last = pos0 + x_tokens - 1
    swa = Hp.bf16_input(s, 8, (B, 128, 512))[0]
    runner = ops.Runner([0], [0], [m], 64, 64)
    p = runner.params(B, Tq, t_last, H, hidden, k)
    g = dict(q=q, swa_kv=swa, swa_len=128, swa_pos0=t_last - 127, out=torch.empty_like(q),
             q_idx=Hp.bf16_input(s, 6, (B, Tq, 32, 128), 1.28)[0],
             w_idx=Hp.f32_input(s, 7, (B, Tq, 32), 1.28)[0],
             x=x, w_kv=wkv, w_gate=wg, norm_w=gam, w_ik=wik, kv_cache=b_["kv"],
             idx_codes=b_["codes"], idx_scales=b_["scales"], n_cap=n_cap, x_tokens=x_tokens,
             x_pos0=pos0, compress_state=b_["state"])
    ws = torch.empty(runner.workspace_size(p, x_tokens, n_cap) + 256, dtype=torch.uint8, device="cuda")
    runner.step(p, [ops.layer_io(**g)], ws)
    torch.cuda.synchronize()
    assert ops.last_device_status() == 0
    n_new = (pos0 + x_tokens) // m - e0
    sl = slice(e0, e0 + n_new)
    assert n_new >= 1
    for key in ("kv", "codes", "scales"):
        np.testing.assert_array_equal(b_[key][:, sl].contiguous().view(torch.uint8).cpu().numpy(),
                                      a[key][:, sl].contiguous().view(torch.uint8).cpu().numpy(),
                                      err_msg=key)
    if use_state:
        np.testing.assert_array_equal(b_["state"].cpu().numpy(), a["state"].cpu().numpy())
