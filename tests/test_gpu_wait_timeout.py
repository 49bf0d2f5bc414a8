"""The bounded-wait error path, on the GPU, without a fault.

The tensor-core decode scorer bounds every mbarrier wait.  Through the diagnostic entry
point csa2_indexer_score_topk_bounded a test gives the launch a short poll limit and makes
its copy thread wait on a barrier that nothing completes: that wait runs out, nothing is
copied, so the producers', the MMA issuer's and the epilogue's first waits run out too;
every role leaves its loop, the CTA frees its tensor memory and exits.  The host then reads
CSA2_ERR_TIMEOUT from csa2_last_device_status, and the same context computes the next call
correctly."""

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


def _p(t):
    return C.c_void_p(0 if t is None else t.data_ptr())


def _case(seed, B=2, n=8192):
    qi, _ = Hp.bf16_input(seed, 1, (B, 1, 32, 128), 1.28)
    w, _ = Hp.f32_input(seed, 2, (B, 1, 32), 1.28)
    codes, scales = Hp.index_cache_input(seed, 3, B, n)
    return qi, w, Hp.to_dev(codes, torch.uint8), Hp.to_dev(scales, torch.uint8)


def test_stalled_scorer_reports_timeout_and_context_stays_usable(lib):
    from compressed_sparse_attention_04_gb300 import _lib as L
    from compressed_sparse_attention_04_gb300 import ops
    B, n, k = 2, 8192, 256
    qi, w, codes, scales = _case(61, B, n)
    stream = torch.cuda.current_stream()
    sp = C.c_void_p(stream.cuda_stream)
    ws_bytes = lib.csa2_indexer_workspace_size(B, 1, n, 0, 64, 0)
    ws = torch.zeros(ws_bytes + 256, dtype=torch.uint8, device="cuda")   # scores read as 0.0
    wp = C.c_void_p((ws.data_ptr() + 255) // 256 * 256)
    assert ops.last_device_status() == 0
    got = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")

    def call(wait_limit, stall):
        return lib.csa2_indexer_score_topk_bounded(
            _p(qi), _p(w), B, 1, n - 1, _p(codes), _p(scales), n, n, 1, k, _p(got), wp,
            ws_bytes, wait_limit, stall, sp)

    # every wait of the stalled launch gives up after 64 polls
    assert call(64, 1) == 0, lib.csa2_last_error_message()
    assert lib.csa2_last_device_status(sp) == L.ERR_TIMEOUT
    assert lib.csa2_last_device_status(sp) == 0          # read and cleared
    # the top-k launch after it ran on the untouched (zero) scores: all tie, so the
    # lowest k indices are chosen -- and it produced a valid index set
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), np.broadcast_to(np.arange(k), (B, 1, k)))

    # the same context: a bounded call without the stall, and the default entry point,
    # give the same selection
    ref = ops.indexer_score_topk(qi, w, n - 1, codes, scales, n, 1, k)
    for limit in (0, 1 << 20):
        got.fill_(-7)
        assert call(limit, 0) == 0, lib.csa2_last_error_message()
        assert lib.csa2_last_device_status(sp) == 0
        np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())
