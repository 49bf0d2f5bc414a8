"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad calls on the host before any launch (no compute call is made)."""

import ctypes as C
import os
import re

import pytest

from conftest import ROOT
import compressed_sparse_attention_04_gb300._lib as L
from compressed_sparse_attention_04_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build_all()
    return L.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"{n} has no ctypes signature"
    assert set(L.SIGNATURES) == set(names)


def test_struct_layouts_match_header():
    # csa2_layer_io: 21 pointers + 6 ints; csa2_step_params: 8 ints + 4 floats
    assert C.sizeof(L.LayerIO) == 21 * 8 + 6 * 4
    assert C.sizeof(L.StepParams) == 12 * 4


def test_status_strings(lib):
    assert lib.csa2_status_str(0) == b"CSA2_OK"
    assert lib.csa2_status_str(3) == b"CSA2_ERR_WORKSPACE"
    assert lib.csa2_version().startswith(b"csa2")


def _vp(x):
    return C.c_void_p(x)


FAKE = 0x10000   # never dereferenced: every call below fails validation first


def test_compress_validation(lib):
    f = lib.csa2_compress
    args = dict(x=_vp(FAKE), B=2, T=8, hidden=128, m=2, pos0=0, w_kv=_vp(FAKE), w_gate=_vp(FAKE),
                norm_w=_vp(FAKE), eps=1e-6, base=1e4, kv=_vp(FAKE), n_cap=4, kv_pre=_vp(FAKE),
                ws=_vp(FAKE), wsb=0, st=_vp(0))

    def call(**kw):
        a = dict(args, **kw)
        return f(*a.values())

    assert call(m=3) == L.ERR_UNSUPPORTED
    assert call(x=_vp(0)) == L.ERR_INVALID_ARG
    assert call(w_gate=_vp(0)) == L.ERR_INVALID_ARG          # m = 2 needs a gate
    assert call(m=1) == L.ERR_INVALID_ARG                    # m = 1 must not have one
    assert call(hidden=100) == L.ERR_INVALID_ARG
    assert call(pos0=1) == L.ERR_INVALID_ARG
    assert call(n_cap=3) == L.ERR_INVALID_ARG                # 4 entries do not fit
    assert call(x=_vp(FAKE + 4)) == L.ERR_INVALID_ARG        # misaligned
    assert call() == L.ERR_WORKSPACE                         # workspace too small
    assert b"workspace" in lib.csa2_last_error_message()


def test_indexer_and_hsi_validation(lib):
    f = lib.csa2_indexer_score_topk
    base = [_vp(FAKE), _vp(FAKE), 1, 1, 10, _vp(FAKE), _vp(FAKE), 64, 32, 1, _vp(0), 0, 64, 16,
            _vp(FAKE), _vp(0), _vp(0), _vp(0), 0, _vp(0)]

    def call(**over):
        a = list(base)
        for i, v in over.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a13=0) == L.ERR_INVALID_ARG                  # k = 0
    assert call(a13=4096) == L.ERR_INVALID_ARG               # k > 2048
    assert call(a7=16) == L.ERR_INVALID_ARG                  # n_cap < n_entries
    assert call(a10=_vp(FAKE), a11=4, a12=48) == L.ERR_UNSUPPORTED   # blk not a power of 2
    assert call(a10=_vp(FAKE), a11=0) == L.ERR_INVALID_ARG   # nb = 0
    assert call(a10=_vp(FAKE), a11=4, a15=_vp(FAKE)) == L.ERR_INVALID_ARG  # pool + blockmax
    assert call() == L.ERR_WORKSPACE
    # the bounded-wait diagnostic: decode-scorer shapes only, stall needs a limit; both
    # refused before any launch
    g = lib.csa2_indexer_score_topk_bounded

    def bounded(Tq=1, q_pos0=10, m=1, wait_limit=64, stall=1):
        return g(_vp(FAKE), _vp(FAKE), 1, Tq, q_pos0, _vp(FAKE), _vp(FAKE), 64, 32, m, 16,
                 _vp(FAKE), _vp(0), 0, wait_limit, stall, _vp(0))

    assert bounded(wait_limit=0) == L.ERR_INVALID_ARG                 # stall needs a limit
    assert bounded(Tq=64) == L.ERR_UNSUPPORTED                        # the prefill scorer's shape
    assert bounded(q_pos0=0, m=2) == L.ERR_UNSUPPORTED                # no visible entry
    assert bounded() == L.ERR_WORKSPACE
    h = lib.csa2_hsi_candidates
    assert h(_vp(0), 1, 1, 0, 10, 1, 64, 4, _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG
    assert h(_vp(FAKE), 1, 1, 0, 10, 1, 64, 0, _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG


def test_sparse_attn_validation(lib):
    f = lib.csa2_sparse_attn
    base = [_vp(FAKE), 1, 1, 4, 200, _vp(FAKE), 64, 32, _vp(FAKE), 8, _vp(FAKE), 128, 73, 128,
            _vp(0), 0.05, _vp(FAKE), _vp(0), _vp(0), 0, _vp(0)]

    def call(**over):
        a = list(base)
        for i, v in over.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a12=74) == L.ERR_INVALID_ARG    # window row 73 not in the window cache
    assert call(a11=127) == L.ERR_INVALID_ARG   # query row 200 not in it
    assert call(a8=_vp(0)) == L.ERR_INVALID_ARG  # k > 0 without top-k
    assert call(a3=0) == L.ERR_INVALID_ARG
    assert call(a13=0) == L.ERR_INVALID_ARG
    assert call(a15=0.0) == L.ERR_INVALID_ARG


def test_compress_chunk_validation(lib):
    f = lib.csa2_compress_chunk
    args = dict(x=_vp(FAKE), B=2, T=3, hidden=128, m=2, pos0=5, w_kv=_vp(FAKE), w_gate=_vp(FAKE),
                norm_w=_vp(FAKE), eps=1e-6, base=1e4, state=_vp(FAKE), kv=_vp(FAKE), n_cap=4,
                kv_pre=_vp(FAKE), ws=_vp(FAKE), wsb=0, st=_vp(0))

    def call(**kw):
        a = dict(args, **kw)
        return f(*a.values())

    assert call(state=_vp(0)) == L.ERR_INVALID_ARG                       # m = 2 needs state
    assert call(m=1, w_gate=_vp(0)) == L.ERR_INVALID_ARG                 # m = 1 carries none
    assert call(state=_vp(FAKE + 8)) == L.ERR_INVALID_ARG                # misaligned state
    assert call(pos0=7) == L.ERR_INVALID_ARG                             # completes entries 3, 4
    assert call(pos0=-1) == L.ERR_INVALID_ARG
    assert call() == L.ERR_WORKSPACE                                     # odd pos0 is fine
    assert call(m=1, w_gate=_vp(0), state=_vp(0), pos0=1) == L.ERR_WORKSPACE


def test_stored_format_quantiser_validation(lib):
    q8 = lib.csa2_swa_kv_quant_fp8
    assert q8(_vp(0), 2, 16, 0, 4, _vp(FAKE), _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG
    assert q8(_vp(FAKE), 2, 16, 10, 7, _vp(FAKE), _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG   # rows past S
    assert q8(_vp(FAKE), 2, 16, 0, 4, _vp(FAKE), _vp(FAKE + 4), _vp(0)) == L.ERR_INVALID_ARG
    assert q8(_vp(FAKE), 2, 16, 3, 0, _vp(FAKE), _vp(FAKE), _vp(0)) == L.OK   # nothing to do
    q4 = lib.csa2_main_kv_quant_fp4
    assert q4(_vp(FAKE), 2, 16, 10, 7, _vp(FAKE), _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG
    assert q4(_vp(FAKE), 0, 16, 0, 4, _vp(FAKE), _vp(FAKE), _vp(0)) == L.ERR_INVALID_ARG


def test_sparse_attn_ex_validation(lib):
    f = lib.csa2_sparse_attn_ex
    # 64 heads, FP4 entries and FP8 window rows
    base = [_vp(FAKE), 1, 1, 64, 200, _vp(0), _vp(FAKE), _vp(FAKE), 64, 32, _vp(FAKE), 8,
            _vp(0), _vp(FAKE), _vp(FAKE), 128, 73, 128, _vp(0), 0.05, _vp(FAKE), _vp(0), _vp(0), 0,
            _vp(0)]

    def call(**over):
        a = list(base)
        for i, v in over.items():
            a[int(i[1:])] = v
        return f(*a)

    assert call(a12=_vp(FAKE)) == L.ERR_INVALID_ARG                # window rows given twice
    assert call(a13=_vp(0), a14=_vp(0)) == L.ERR_INVALID_ARG       # ... and not at all
    assert call(a14=_vp(0)) == L.ERR_INVALID_ARG                   # codes without scales
    assert call(a5=_vp(FAKE)) == L.ERR_INVALID_ARG                 # entries given twice
    assert call(a3=12) == L.ERR_UNSUPPORTED                        # quantised rows: H a multiple of 8
    assert call(a3=72) == L.ERR_UNSUPPORTED                        # ... up to 64
    assert call(a14=_vp(FAKE + 8)) == L.ERR_INVALID_ARG            # misaligned scales
    assert call(a16=74) == L.ERR_INVALID_ARG                       # window row 73 missing


def _runner(lib, kv, idx, ratio, blk=64, nb=64):
    n = len(kv)
    arr = C.c_int32 * n
    h = C.c_void_p()
    st = lib.csa2_runner_create(n, arr(*kv), arr(*idx), arr(*ratio), blk, nb, C.byref(h))
    return st, h


def test_runner_modes_and_rejections(lib):
    import sys
    sys.path.insert(0, ROOT)
    from oracle import layers as Lr   # the oracle's table reader is the reference here
    kv, idx, ratio = Lr.v41_flash_tables()
    st, h = _runner(lib, kv, idx, ratio)
    assert st == L.OK
    modes = [lib.csa2_runner_layer_mode(h, l) for l in range(40)]
    names = {L.MODE_SWA: "swa", L.MODE_FULL: "full", L.MODE_REINDEX: "reindex", L.MODE_REUSE: "reuse"}
    assert [names[m] for m in modes] == Lr.layer_modes(kv, idx)
    assert lib.csa2_runner_layer_mode(h, 40) == -1
    p = L.StepParams(64, 1, 131071, 64, 4096, 512, 128, 0, 512 ** -0.5, 1e-6, 1e4, 0.0)
    assert lib.csa2_runner_workspace_size(h, C.byref(p), 2, 131072) > 64 * 131072 * 4
    lib.csa2_runner_destroy(h)
    for kv_, idx_ in ([[0, 1], [0, 0]], [[0, 2, 2], [0, 1, 2]], [[0, 1, 0], [0, 1, 1]],
                      [[-1, 0], [-1, 0]], [[-1], [0]]):
        st, h = _runner(lib, kv_, idx_, [1] * len(kv_))
        assert st == L.ERR_INVALID_ARG, (kv_, idx_)
    assert _runner(lib, [0], [0], [3])[0] == L.ERR_UNSUPPORTED
    assert _runner(lib, [0], [0], [1], blk=48)[0] == L.ERR_UNSUPPORTED


def _header_struct_fields(name):
    """Field names of typedef struct { ... } name; in include/csa2.h, in order."""
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    m = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        for part in decl.split(","):
            fields.append(re.findall(r"[A-Za-z_][A-Za-z0-9_]*", part)[-1])
    return fields


def test_struct_field_order_matches_header():
    assert [f for f, _ in L.LayerIO._fields_] == _header_struct_fields("csa2_layer_io")
    assert [f for f, _ in L.StepParams._fields_] == _header_struct_fields("csa2_step_params")


def _header_prototypes():
    """name -> list of parameter kinds ('ptr', 'int', 'float', 'size') from include/csa2.h."""
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(csa2_[a-z0-9_]+)\s*\(([^()]*)\)\s*;", src):
        params = m.group(2).strip()
        kinds = []
        if params and params != "void":
            for p in params.split(","):
                p = p.strip()
                if "*" in p:
                    kinds.append("ptr")
                elif re.search(r"\bsize_t\b", p):
                    kinds.append("size")
                elif re.search(r"\bfloat\b", p):
                    kinds.append("float")
                else:
                    assert re.search(r"\b(int|int32_t|unsigned)\b", p), p
                    kinds.append("int")
        out[m.group(1)] = kinds
    return out


def test_ctypes_signatures_match_header_prototypes():
    kind_of = {C.c_void_p: "ptr", C.c_int: "int", C.c_uint: "int", C.c_float: "float",
               C.c_size_t: "size"}
    protos = _header_prototypes()
    assert set(protos) == set(L.SIGNATURES)
    for name, (_, argtypes) in L.SIGNATURES.items():
        got = [kind_of.get(t, "ptr") for t in argtypes]   # POINTER(...) types are pointers
        assert got == protos[name], name


def test_library_exports_nothing_undeclared(lib):
    import shutil
    import subprocess
    if not shutil.which("nm"):
        pytest.skip("nm not available")
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {w for line in out.splitlines() for w in line.split()[-1:] if w.startswith("csa2_")}
    assert exported == set(_declared_functions())


def test_plain_c_program_links_and_calls_the_library(lib, tmp_path):
    """The boundary is usable from C: the header compiles as C99 and a C program linked
    against libcsa2.so runs its host-only calls (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    prog = tmp_path / "abi_check.c"
    prog.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "csa2.h"
int main(void) {
  if (strncmp(csa2_version(), "csa2", 4) != 0) return 1;
  if (strcmp(csa2_status_str(CSA2_ERR_WORKSPACE), "CSA2_ERR_WORKSPACE") != 0) return 2;
  /* host-side validation: m = 3 is refused before any launch */
  int st = csa2_compress((void*)16, 1, 2, 64, 3, 0, (void*)16, (void*)16, (float*)16, 1e-6f,
                         1e4f, (void*)16, 4, NULL, NULL, 0, NULL);
  if (st != CSA2_ERR_UNSUPPORTED) return 3;
  if (csa2_last_error_message()[0] == 0) return 4;
  printf("ok\n");
  return 0;
}
''')
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(L.LIB_PATH)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(prog), "-L", libdir, "-lcsa2", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stderr)


def _noalloc_limit_entries(lib, B, blk=64):
    """Largest decode row length (Tq = 1, Full) whose workspace fits the built-in array."""
    cap = lib.csa2_indexer_noalloc_max_scratch_bytes()
    ws = lambda n: lib.csa2_indexer_workspace_size(B, 1, n, 0, blk, 0)
    lo, hi = 1, 1 << 26
    assert ws(lo) <= cap < ws(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ws(mid) <= cap:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_refuses_one_entry_past_its_limit(lib):
    # The limit is the workspace size of the call, not a count of scores: one entry more
    # than the largest accepted row length is refused on the host, before any launch.
    f = lib.csa2_indexer_score_topk_noalloc
    cap = lib.csa2_indexer_noalloc_max_scratch_bytes()
    for B in (1, 4):
        n = _noalloc_limit_entries(lib, B)
        assert lib.csa2_indexer_workspace_size(B, 1, n, 0, 64, 0) <= cap
        assert lib.csa2_indexer_workspace_size(B, 1, n + 1, 0, 64, 0) > cap
        st = f(_vp(FAKE), _vp(FAKE), B, 1, n, _vp(FAKE), _vp(FAKE), n + 1, n + 1, 1, None, 0, 64,
               512, _vp(FAKE), None, _vp(0))
        assert st == L.ERR_UNSUPPORTED
        assert str(cap).encode() in lib.csa2_last_error_message()
    # a prefill call with short rows is counted with its FP4 query images (2176 B per row)
    Tq = cap // 2176 + 1
    st = f(_vp(FAKE), _vp(FAKE), 1, Tq, 0, _vp(FAKE), _vp(FAKE), 64, 64, 1, None, 0, 64, 16,
           _vp(FAKE), None, _vp(0))
    assert st == L.ERR_UNSUPPORTED
