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


def test_noalloc_at_its_limit(lib):
    # The largest call the array admits (one entry more would be refused) runs and
    # matches the workspace entry point.
    from compressed_sparse_attention_04_gb300 import ops
    from test_abi_host import _noalloc_limit_entries
    B, k, blk = 4, 512, 64
    cap = lib.csa2_indexer_noalloc_max_scratch_bytes()
    n_entries = _noalloc_limit_entries(lib, B, blk)   # the longest rows the array admits
    assert lib.csa2_indexer_workspace_size(B, 1, n_entries, 0, blk, 0) <= cap
    assert lib.csa2_indexer_workspace_size(B, 1, n_entries + 1, 0, blk, 0) > cap
    qi, w, codes, scales = _inputs(33, B, n_entries)
    ref = ops.indexer_score_topk(qi, w, n_entries - 1, codes, scales, n_entries, 1, k, blk=blk)
    got = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.csa2_indexer_score_topk_noalloc(
        _p(qi), _p(w), B, 1, n_entries - 1, _p(codes), _p(scales), n_entries, n_entries, 1,
        None, 0, blk, k, _p(got), None, stream)
    assert st == 0, lib.csa2_last_error_message()
    torch.cuda.synchronize()
    assert ops.last_device_status() == 0
    np.testing.assert_array_equal(got.cpu().numpy(), ref.cpu().numpy())


_CONTEXT_SCRIPT = r'''
import ctypes as C, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from compressed_sparse_attention_04_gb300 import _lib
lib = _lib.load()
cu = C.CDLL("libcuda.so.1")
def ok(r, what):
    assert r == 0, f"{what}: CUresult {r}"
ok(cu.cuInit(0), "cuInit")
dev = C.c_int()
ok(cu.cuDeviceGet(C.byref(dev), 0), "cuDeviceGet")

def alloc(nbytes):
    p = C.c_uint64()
    ok(cu.cuMemAlloc_v2(C.byref(p), C.c_size_t(nbytes)), "cuMemAlloc")
    return p.value

def upload(a):
    a = np.ascontiguousarray(a)
    p = alloc(a.nbytes)
    ok(cu.cuMemcpyHtoD_v2(C.c_uint64(p), a.ctypes.data_as(C.c_void_p), C.c_size_t(a.nbytes)), "HtoD")
    return p

def download(p, shape, dtype):
    a = np.empty(shape, dtype)
    ok(cu.cuMemcpyDtoH_v2(a.ctypes.data_as(C.c_void_p), C.c_uint64(p), C.c_size_t(a.nbytes)), "DtoH")
    return a

def one_context_case(seed):
    # inputs allocated in the current context; workspace entry point vs no-alloc, twice
    B, n, k, blk = 2, 5000, 64, 64
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((B, 1, 32, 128)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w = rng.standard_normal((B, 1, 32)).astype(np.float32)
    codes = rng.integers(0, 256, (B, n, 64), dtype=np.uint8)
    scales = rng.integers(0x18, 0x58, (B, n, 4), dtype=np.uint8)
    dq, dw, dc, ds = upload(q), upload(w), upload(codes), upload(scales)
    ws_bytes = lib.csa2_indexer_workspace_size(B, 1, n, 0, blk, 0)
    ws = alloc(ws_bytes + 256)
    ref_p, got_p = alloc(B * k * 4), alloc(B * k * 4)
    vp = C.c_void_p
    st = lib.csa2_indexer_score_topk(vp(dq), vp(dw), B, 1, n - 1, vp(dc), vp(ds), n, n, 1, None, 0,
                                     blk, k, vp(ref_p), None, None, vp(ws), ws_bytes + 256, None)
    assert st == 0, lib.csa2_last_error_message()
    ref = None
    for call in range(2):
        ok(cu.cuMemsetD8_v2(C.c_uint64(got_p), C.c_ubyte(0xA5), C.c_size_t(B * k * 4)), "memset")
        st = lib.csa2_indexer_score_topk_noalloc(vp(dq), vp(dw), B, 1, n - 1, vp(dc), vp(ds), n, n,
                                                 1, None, 0, blk, k, vp(got_p), None, None)
        assert st == 0, lib.csa2_last_error_message()
        assert lib.csa2_last_device_status(None) == 0
        ref = download(ref_p, (B, k), np.int32)
        got = download(got_p, (B, k), np.int32)
        assert (got == ref).all(), f"call {call}"
    assert (ref >= 0).all()
    for p in (dq, dw, dc, ds, ws, ref_p, got_p):
        ok(cu.cuMemFree_v2(C.c_uint64(p)), "cuMemFree")

# first the device's primary context, then a second context made current through the
# driver API: the array has another address there, which the entry point must look up
prim = C.c_void_p()
ok(cu.cuDevicePrimaryCtxRetain(C.byref(prim), dev), "cuDevicePrimaryCtxRetain")
ok(cu.cuCtxSetCurrent(prim), "cuCtxSetCurrent")
one_context_case(1)
ctx2 = C.c_void_p()
ok(cu.cuCtxCreate_v2(C.byref(ctx2), 0, dev), "cuCtxCreate")
one_context_case(2)
ok(cu.cuCtxDestroy_v2(ctx2), "cuCtxDestroy")
ok(cu.cuCtxSetCurrent(prim), "cuCtxSetCurrent")
one_context_case(3)
print("contexts ok")
'''


def test_noalloc_in_a_second_cuda_context(lib):
    # A caller that makes its own context current through the driver API gets that
    # context's copy of the array, not the one the primary context saw first.
    import subprocess
    import sys
    from conftest import ROOT
    r = subprocess.run([sys.executable, "-c", _CONTEXT_SCRIPT, ROOT], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "contexts ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
