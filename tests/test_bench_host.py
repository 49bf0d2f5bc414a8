"""bench.py's host-side pieces without a GPU: the config object both arms print, the
attention traffic record lookup, and the algorithmic bytes per stage for each workload."""

import json
import os
import sys

import pytest

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_both_arms_share_the_workload_config():
    for name, wl in bench.WORKLOADS.items():
        c = bench.workload_config(wl, 1)
        json.dumps(c)
        assert c["workload"].startswith(f"csa2_decode_40layer_b{wl['B']}_ctx{wl['C']}")
        assert c["parallelism"] == "single" and bench.workload_config(wl, 2)["parallelism"] == "replicas"
        assert ("_fp4kv_fp8swa" in c["workload"]) == bool(wl.get("stored"))
    assert bench.workload_config(bench.WORKLOADS["decode40"], 1)["workload"] == \
        "csa2_decode_40layer_b64_ctx131072"


def test_traffic_record_lookup():
    kv, idx, ratio = bench.layer_tables()
    modes = [0 if k == -1 else (1 if k == l else (2 if idx[l] == l else 3)) for l, k in enumerate(kv)]
    t = bench.attention_traffic(modes)
    assert t is None or t > 0
    src = open(os.path.join(ROOT, "compressed_sparse_attention_04_gb300", "csrc", "attention.cu"),
               encoding="utf-8").read()
    h = bench.attention_kernel_hash(src)
    assert len(h) == 16
    # a host-side edit after the first extern "C" block leaves the kernel hash unchanged
    i = src.index('\nextern "C" {')
    assert bench.attention_kernel_hash(src[:i] + src[i:] + "\n// host note\n") == h
    assert bench.attention_kernel_hash("// a comment\n" + src) == h          # comments ignored
    assert bench.attention_kernel_hash("static int edit;\n" + src) != h


class _FakeStack:
    stage_bytes = bench.Stack.stage_bytes

    def __init__(self, wl):
        self.wl = wl
        self.kv_src, self.idx_src, self.ratio = bench.layer_tables()
        self.modes = [0 if k == -1 else (1 if k == l else (2 if self.idx_src[l] == l else 3))
                      for l, k in enumerate(self.kv_src)]


@pytest.mark.parametrize("name", ["decode40", "decode40_stored"])
def test_attention_algorithmic_bytes(name):
    wl = bench.WORKLOADS[name]
    st = _FakeStack(wl)
    B, H, k, W = wl["B"], wl["H"], wl["k"], wl["window"]
    fixed = 2 * B * H * 512 * 2
    row = (288, 520) if wl.get("stored") else (1024, 1024)
    assert st.stage_bytes(0, 5) == B * W * row[1] + fixed                       # window-only layer
    assert st.stage_bytes(5, 5) == B * (k * row[0] + W * row[1]) + fixed + B * k * 4
    # a Full layer's scoring reads every key once (68 B each)
    assert st.stage_bytes(20, 2) == B * (wl["C"] // 1) * 68 + B * (32 * 128 * 2 + 32 * 4)


def test_layer_tables_are_the_pages_pattern():
    kv, idx, ratio = bench.layer_tables()
    assert sum(1 for l, k in enumerate(kv) if k == l) == 4          # Full layers
    assert sum(1 for l, k in enumerate(kv) if k not in (-1, l) and idx[l] == l) == 4   # Reindex
    assert kv[:2] == [-1, -1] and ratio[20] == 1 and ratio[2] == 2
