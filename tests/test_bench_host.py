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
        pat = bench.PATTERN_NAMES[wl.get("pattern", "stack40")]
        assert c["workload"].startswith(f"csa2_decode_{pat}_b{wl['B']}_ctx{wl['C']}")
        assert c["layers"] == len(bench.layer_tables(wl.get("pattern", "stack40"))[0])
        assert c["parallelism"] == "single" and bench.workload_config(wl, 2)["parallelism"] == "replicas"
        assert ("_fp4kv_fp8swa" in c["workload"]) == bool(wl.get("stored"))
    assert bench.workload_config(bench.WORKLOADS["decode40"], 1)["workload"] == \
        "csa2_decode_40layer_b64_ctx131072"
    assert bench.workload_config(bench.WORKLOADS["decoder_group"], 1)["workload"] == \
        "csa2_decode_decoder_group_b32_ctx65536"
    assert bench.workload_config(bench.WORKLOADS["long1m"], 1)["workload"] == \
        "csa2_decode_full_layer_b4_ctx1048576"


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
        self.kv_src, self.idx_src, self.ratio = bench.layer_tables(wl.get("pattern", "stack40"))
        n = len(self.kv_src)
        self.modes = [0 if k == -1 else (1 if k == l else (2 if self.idx_src[l] == l else 3))
                      for l, k in enumerate(self.kv_src)]
        self.builds_pool = [any(self.modes[j] == 2 and self.kv_src[j] == l for j in range(n))
                            for l in range(n)]


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


def test_decoder_group_and_long_context_patterns():
    # decoder group: Full (m = 1) -> Reindex -> 2 Reuse reading the Reindex layer's selection
    kv, idx, ratio = bench.layer_tables("decoder_group")
    assert (kv, idx, ratio) == ([0, 0, 0, 0], [0, 1, 1, 1], [1, 0, 0, 0])
    st = _FakeStack(bench.WORKLOADS["decoder_group"])
    assert st.modes == [1, 2, 3, 3] and st.builds_pool == [True, False, False, False]
    B, C, k, W, H = 32, 65536, 512, 128, 64
    # the Reindex layer scores its 64 x 64-entry pool, not the cache
    assert st.stage_bytes(1, 2) == B * 4096 * 68 + B * 64 * 4 + B * (32 * 128 * 2 + 32 * 4)
    assert st.stage_bytes(0, 4) == B * (C // 64) * 4 + B * 64 * 4
    # the configuration's algorithmic bytes: scoring + selection + pools + 4 attention layers
    hot = sum(st.stage_bytes(l, s) for l in range(4) for s in (2, 3, 4, 5))
    assert hot == (B * C * 68 + B * (32 * 128 * 2 + 32 * 4) + B * C * 4 + B * k * 4 +
                   B * (C // 64) * 4 + B * 64 * 4 +
                   B * 4096 * 68 + B * 64 * 4 + B * (32 * 128 * 2 + 32 * 4) + B * 4096 * 4 + B * k * 4 +
                   4 * (B * (k + W) * 1024 + 2 * B * H * 512 * 2 + B * k * 4))
    # one encoder Full layer: no Reindex layer reads its block maxima, so no pool is built
    st = _FakeStack(bench.WORKLOADS["long1m"])
    assert st.modes == [1] and st.builds_pool == [False] and st.stage_bytes(0, 4) == 0
    assert st.stage_bytes(0, 2) == 4 * 524288 * 68 + 4 * (32 * 128 * 2 + 32 * 4)
