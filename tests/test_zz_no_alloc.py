"""The no-allocation indexer entry point (csa2_indexer_score_topk_noalloc).

For callers that cannot allocate device memory, the library keeps the score scratch
in a fixed array of its own.  This test calls it through the C ABI and checks that
two calls in a row give exactly what csa2_indexer_score_topk gives with a caller
workspace (same kernels, same inputs), and that an over-size call is refused.
Kept in a file of its own, collected last."""

import ctypes as C

import numpy as np
import pytest
import torch

import helpers as Hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from compressed_sparse_attention_04_gb300 import build
    from compressed_sparse_attention_04_gb300 import _lib
    build.build_all()
    return _lib.load()


def _inputs(seed, B, n_entries):
    qi, _ = Hp.bf16_input(seed, 1, (B, 1, 32, 128), 1.28)
    w, _ = Hp.f32_input(seed, 2, (B, 1, 32), 1.28)
    codes, scales = Hp.index_cache_input(seed, 3, B, n_entries)
    return qi, w, Hp.to_dev(codes, torch.uint8), Hp.to_dev(scales, torch.uint8)


def _p(t):
    return C.c_void_p(0 if t is None else t.data_ptr())


def test_noalloc_matches_workspace_entry_point_twice(lib):
    from compressed_sparse_attention_04_gb300 import ops
    B, n_entries, k, blk = 4, 70001, 512, 64
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.csa2_indexer_noalloc_max_scratch_bytes() >= B * n_entries * 4
    for call, seed in enumerate((31, 32)):          # two calls in a row, different inputs
        qi, w, codes, scales = _inputs(seed, B, n_entries)
        nblk = -(-n_entries // blk)
        ref_bm = torch.empty(B, 1, nblk, dtype=torch.float32, device="cuda")
        ref = ops.indexer_score_topk(qi, w, n_entries - 1, codes, scales, n_entries, 1, k,
                                     blk=blk, blockmax_out=ref_bm)
        got = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
        got_bm = torch.full((B, 1, nblk), 7.0, dtype=torch.float32, device="cuda")
        st = lib.csa2_indexer_score_topk_noalloc(
            _p(qi), _p(w), B, 1, n_entries - 1, _p(codes), _p(scales), n_entries, n_entries, 1,
            None, 0, blk, k, _p(got), _p(got_bm), stream)
        assert st == 0, lib.csa2_last_error_message()
        torch.cuda.synchronize()
        assert ops.last_device_status() == 0
        np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy(), err_msg=f"call {call}")
        np.testing.assert_array_equal(got_bm.cpu().numpy(), ref_bm.cpu().numpy())


def test_noalloc_pool_mode_and_size_limit(lib):
    from compressed_sparse_attention_04_gb300 import ops
    B, n_entries, k, blk, nb = 3, 8192, 128, 64, 16
    qi, w, codes, scales = _inputs(40, B, n_entries)
    cand = Hp.to_dev(np.tile((np.arange(nb) * 7)[None, None, :], (B, 1, 1)).astype(np.int32),
                     torch.int32)
    ref = ops.indexer_score_topk(qi, w, n_entries - 1, codes, scales, n_entries, 1, k, cand=cand,
                                 blk=blk)
    got = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        assert lib.csa2_indexer_score_topk_noalloc(
            _p(qi), _p(w), B, 1, n_entries - 1, _p(codes), _p(scales), n_entries, n_entries, 1,
            _p(cand), nb, blk, k, _p(got), None, stream) == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())
    # 5 Mi scores do not fit the 16 MiB array: refused before any launch
    big = lib.csa2_indexer_noalloc_max_scratch_bytes() // 4 + 1
    st = lib.csa2_indexer_score_topk_noalloc(
        _p(qi), _p(w), 1, 1, big - 1, _p(codes), _p(scales), big, big, 1, None, 0, blk, k,
        _p(got), None, stream)
    assert st == 2 and b"16777216" in lib.csa2_last_error_message()
