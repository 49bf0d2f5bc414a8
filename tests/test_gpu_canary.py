"""Canary padding around every output buffer the entry points write.

Each output lives in the middle of a larger allocation whose head and tail hold a sentinel
pattern; after the call (small shapes with ragged tails, decode and prefill forms, pools,
stored formats) the padding must be untouched, so no kernel writes past either end of what it
was given.  The values themselves are checked against the oracle elsewhere."""

import numpy as np
import pytest
import torch

import helpers as Hp

pytestmark = pytest.mark.gpu

PAD = 256   # elements on each side (>= 512 bytes, keeps every view 256-byte aligned)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from compressed_sparse_attention_04_gb300 import build
    build.build_all()


def _ops():
    from compressed_sparse_attention_04_gb300 import ops
    return ops


class Padded:
    """A tensor of `shape` inside a flat buffer with PAD sentinel elements before and after."""

    def __init__(self, shape, dtype, fill=0):
        n = int(np.prod(shape))
        self.flat = torch.empty(n + 2 * PAD, dtype=dtype, device="cuda")
        raw = self.flat.view(torch.uint8)
        raw.fill_(0xA7)   # the sentinel: every byte 0xA7
        self.view = self.flat[PAD:PAD + n].view(shape)
        if fill is not None:
            self.view.fill_(fill)

    def intact(self):
        torch.cuda.synchronize()
        head = self.flat[:PAD].view(torch.uint8)
        tail = self.flat[-PAD:].view(torch.uint8)
        return bool((head == 0xA7).all()) and bool((tail == 0xA7).all())


def test_compress_and_index_keys_stay_inside_their_buffers():
    ops = _ops()
    for (B, T, hidden, m, pos0, n_cap) in [(3, 37, 192, 2, 10, 40), (2, 130, 256, 1, 7, 200),
                                             (4, 2, 4096, 2, 131070, 65536)]:
        x, _ = Hp.bf16_input(7, 1, (B, T, hidden))
        wkv, _ = Hp.bf16_input(7, 2, (512, hidden), 0.02)
        wg = Hp.bf16_input(7, 3, (512, hidden), 0.02)[0] if m == 2 else None
        gam = torch.ones(512, dtype=torch.float32, device="cuda")
        cache = Padded((B, n_cap, 512), torch.bfloat16)
        G = T // m
        pre = Padded((B, G, 512), torch.float32)
        ops.compress(x, wkv, wg, gam, m, pos0, cache.view, kv_pre=pre.view)
        assert cache.intact() and pre.intact(), (B, T, hidden, m)
        wik, _ = Hp.bf16_input(7, 4, (128, 512), 0.02)
        codes = Padded((B, n_cap, 64), torch.uint8)
        scales = Padded((B, n_cap, 4), torch.uint8)
        kout = Padded((B, G, 128), torch.float32)
        ops.index_k_quant(pre.view, pos0 // m, m, wik, codes.view, scales.view, k_out=kout.view)
        assert codes.intact() and scales.intact() and kout.intact(), (B, T, hidden, m)
        assert ops.last_device_status() == 0


@pytest.mark.parametrize("B,Tq,q_pos0,n_entries,m,k,pool", [
    (3, 1, 9999, 5000, 1, 512, False),     # decode, several chunks, ragged tail
    (1, 300, 0, 150, 2, 64, False),        # causal prefill (grouped scorer)
    (2, 1, 69999, 70000, 1, 512, False),   # long row: threshold-filtered selection
    (2, 1, 8191, 8192, 1, 256, True),      # Reindex pool
])
def test_indexer_outputs_stay_inside_their_buffers(B, Tq, q_pos0, n_entries, m, k, pool):
    ops = _ops()
    n_cap = -(-n_entries // 64) * 64
    qi, _ = Hp.bf16_input(11, 1, (B, Tq, 32, 128), 1.28)
    w, _ = Hp.f32_input(11, 2, (B, Tq, 32), 1.28)
    c, s = Hp.index_cache_input(11, 3, B, n_cap)
    codes, scales = Hp.to_dev(c, torch.uint8), Hp.to_dev(s, torch.uint8)
    blk = 64
    nblk = -(-n_entries // blk)
    top = Padded((B, Tq, k), torch.int32)
    if pool:
        nb = 16
        cand = Hp.to_dev(np.tile((np.arange(nb) * 7)[None, None, :], (B, Tq, 1)).astype(np.int32),
                         torch.int32)
        sc = Padded((B, Tq, nb * blk), torch.float32)
        ops.indexer_score_topk(qi, w, q_pos0, codes, scales, n_entries, m, k, cand=cand, blk=blk,
                               topk_out=top.view, scores_out=sc.view)
        assert top.intact() and sc.intact()
    else:
        bm = Padded((B, Tq, nblk), torch.float32) if Tq == 1 else None
        sc = Padded((B, Tq, n_entries), torch.float32)
        ops.indexer_score_topk(qi, w, q_pos0, codes, scales, n_entries, m, k, blk=blk,
                               topk_out=top.view, blockmax_out=None if bm is None else bm.view,
                               scores_out=sc.view)
        assert top.intact() and sc.intact() and (bm is None or bm.intact())
        if bm is not None:
            cand = Padded((B, Tq, 64), torch.int32)
            ops.hsi_candidates(bm.view, q_pos0, n_entries, m, blk, 64, cand_out=cand.view)
            assert cand.intact()
    assert ops.last_device_status() == 0


@pytest.mark.parametrize("B,Tq,H,q_pos0,n_cap,k,stored", [
    (64, 1, 64, 4095, 4096, 512, False),   # decode shape: cluster kernel
    (1, 300, 64, 299, 512, 128, False),    # more rows than SMs: persistent kernel
    (3, 2, 16, 700, 1024, 100, False),     # fewer heads, ragged k
    (8, 1, 64, 2047, 2048, 256, True),     # FP4 entries + FP8 window rows
])
def test_attention_outputs_stay_inside_their_buffers(B, Tq, H, q_pos0, n_cap, k, stored):
    ops = _ops()
    swa_pos0 = max(0, q_pos0 - 127)          # every query's whole window is present
    S = q_pos0 + Tq - swa_pos0
    q, _ = Hp.bf16_input(13, 1, (B, Tq, H, 512), 1.28)
    kv, _ = Hp.bf16_input(13, 2, (B, n_cap, 512))
    swa, _ = Hp.bf16_input(13, 3, (B, S, 512))
    rng = np.random.default_rng(13)
    tk = np.stack([np.sort(rng.choice(n_cap, k, replace=False)) for _ in range(B * Tq)])
    topk = Hp.to_dev(tk.reshape(B, Tq, k).astype(np.int32), torch.int32)
    out = Padded((B, Tq, H, 512), torch.bfloat16)
    lse = Padded((B, Tq, H), torch.float32)
    if stored:
        codes = torch.empty(B, n_cap, 256, dtype=torch.uint8, device="cuda")
        scl = torch.empty(B, n_cap, 32, dtype=torch.uint8, device="cuda")
        ops.main_kv_quant_fp4(kv, 0, n_cap, codes, scl)
        wc = torch.empty(B, S, 512, dtype=torch.uint8, device="cuda")
        wsc = torch.empty(B, S, 8, dtype=torch.uint8, device="cuda")
        ops.swa_kv_quant_fp8(swa, 0, S, wc, wsc)
        ops.sparse_attn(q, q_pos0, None, n_cap, topk, None, swa_pos0, out=out.view, lse_out=lse.view,
                        kv_fp4=(codes, scl), swa_fp8=(wc, wsc))
    else:
        ops.sparse_attn(q, q_pos0, kv, n_cap, topk, swa, swa_pos0, out=out.view, lse_out=lse.view)
    assert out.intact() and lse.intact()
    assert ops.last_device_status() == 0
