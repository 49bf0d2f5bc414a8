#!/usr/bin/env python3
"""Decode throughput of the CSA2 global-attention hot path on one GB300.

Workload (default): the 40-layer attention-only stack of DeepSeek-V4.1-Flash, one
decode step for 64 sequences at 131072 tokens of context: layers 0-1 window only,
encoder Full layers 2/8/14 (m = 2, 65536 entries) with Reuse layers, decoder Full
layer 20 (m = 1, 131072 entries) building an HSI pool (top-64 blocks of 64),
Reindex layers 24/28/32/36 and Reuse layers; 64 heads x 512, top-512, window 128.
Inputs are seeded synthetic (generator module ``synth``); caches are built through
the library's own compressor before timing.  A step = one csa2_runner_step call
(every stage of the path for every layer).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle instead.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA2 decode tokens/s at 128K ctx (1 GB300); indexer+sparse-attn % HBM roofline"
STAGE_NAMES = ["compress", "index_k", "indexer_scores", "topk_select", "hsi_pool", "sparse_attn"]

WORKLOADS = {
    # the headline configuration
    "decode40": dict(B=64, C=131072, H=64, hidden=4096, k=512, window=128, blk=64, nb=64),
    # a small stand-in for quick checks (not a bench line)
    "small": dict(B=4, C=8192, H=64, hidden=4096, k=512, window=128, blk=64, nb=64),
    # the headline step with the HSI variant of 8-entry blocks, 2048 candidate blocks per
    # pool (16 384 entries); a measured variant, not the headline
    "decode40_hsi8": dict(B=64, C=131072, H=64, hidden=4096, k=512, window=128, blk=8, nb=2048),
    # the headline step with the pages' stored formats: FP4 main KV (the Full layers quantise
    # their new entries) and FP8 window rows; a measured variant, not the headline
    "decode40_stored": dict(B=64, C=131072, H=64, hidden=4096, k=512, window=128, blk=64, nb=64,
                            stored=True),
    # the headline batch at an 8K context: every attention launch has the headline shape
    # (64 rows x (512 + 128) rows x 64 heads) with a few GB of caches, small enough for a
    # full profiler capture (not a bench line)
    "b64_ctx8k": dict(B=64, C=8192, H=64, hidden=4096, k=512, window=128, blk=64, nb=64),
    # the decoder group alone: a Full layer (m = 1) building the HSI pool, one Reindex layer
    # rescoring it, two Reuse layers; 32 sequences at 65536 entries
    "decoder_group": dict(B=32, C=65536, H=64, hidden=4096, k=512, window=128, blk=64, nb=64,
                          pattern="decoder_group"),
    # one encoder Full layer (m = 2) at 1 048 576 tokens of context: 524 288 entries, 4 sequences
    "long1m": dict(B=4, C=1048576, H=64, hidden=4096, k=512, window=128, blk=64, nb=64,
                   pattern="encoder_full"),
}

# Layer patterns: (kv_source_layer_ids, index_source_layer_ids, m per layer, 0 for a layer
# that compresses nothing).
PATTERN_NAMES = {"stack40": "40layer", "decoder_group": "decoder_group", "encoder_full": "full_layer"}


NOMINAL_HBM_GBS = 8000.0   # the ~8 TB/s nominal HBM3e rate, reported beside the measured one


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def attention_kernel_hash(text):
    """16 hex digits of SHA-256 over the kernel code of attention.cu: everything before its
    first extern "C" block (the host entry points follow it), with #include lines, // comments
    and blank lines left out."""
    import hashlib
    head = text[:text.index('\nextern "C" {')]
    code = []
    for line in head.splitlines():
        if line.startswith("#include"):
            continue
        line = line.split("//", 1)[0].rstrip()
        if line:
            code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "attn_traffic.json")


def attention_traffic(modes):
    """DRAM bytes per attention launch, averaged over one step's layers, from the ncu traffic
    record (a JSON data file next to the profile summaries: bytes of a launch for a layer with
    a global branch at the headline shape, and of a window-only launch, plus the hash of the
    kernel code they were captured on).  None when the kernel code no longer matches the
    record or the record is missing."""
    try:
        with open(TRAFFIC_RECORD, encoding="utf-8") as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, "compressed_sparse_attention_04_gb300", "csrc", "attention.cu"),
                  encoding="utf-8") as f:
            h = attention_kernel_hash(f.read())
        if rec.get("attention_kernel_sha256_16") != h:
            return None
        full, win = int(rec["traffic_full_launch_bytes"]), int(rec["traffic_window_launch_bytes"])
        return sum(win if m == 0 else full for m in modes) / len(modes)
    except Exception:
        return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ----------------------------------------------------------------------------- GPU setup
def layer_tables(pattern="stack40"):
    """A workload's Full/Reindex/Reuse pattern (kv_source_layer_ids, index_source_layer_ids, m):
    the 40-layer stack, the decoder group (Full m = 1, Reindex, 2 Reuse) or one encoder Full
    layer (m = 2)."""
    if pattern == "decoder_group":
        return [0, 0, 0, 0], [0, 1, 1, 1], [1, 0, 0, 0]
    if pattern == "encoder_full":
        return [0], [0], [2]
    assert pattern == "stack40", pattern
    kv, idx, ratio = [], [], []
    cur_kv = cur_idx = -1
    for l in range(40):
        if l < 2:
            kv.append(-1); idx.append(-1); ratio.append(0)
            continue
        if l in (2, 8, 14, 20):
            cur_kv = cur_idx = l
            ratio.append(2 if l < 20 else 1)
        else:
            if l in (24, 28, 32, 36):
                cur_idx = l
            ratio.append(0)
        kv.append(cur_kv); idx.append(cur_idx)
    return kv, idx, ratio


class Stack:
    """Device-resident inputs, caches and outputs of the decode step."""

    def __init__(self, wl, device, seed_base=5000, log=print):
        import torch
        from compressed_sparse_attention_04_gb300 import ops
        from synth import gpu as sg
        self.wl = wl
        B, C, H, hid, W = wl["B"], wl["C"], wl["H"], wl["hidden"], wl["window"]
        self.t = C - 1
        self.kv_src, self.idx_src, self.ratio = layer_tables(wl.get("pattern", "stack40"))
        self.n_layers = len(self.kv_src)
        self.runner = ops.Runner(self.kv_src, self.idx_src, self.ratio, wl["blk"], wl["nb"])
        self.modes = [self.runner.mode(l) for l in range(self.n_layers)]
        # Full layers whose block maxima feed a Reindex layer's candidate pool
        self.builds_pool = [any(self.modes[j] == 2 and self.kv_src[j] == l for j in range(self.n_layers))
                            for l in range(self.n_layers)]
        self.params = ops.Runner.params(B, 1, self.t, H, hid, wl["k"], W)
        self.layers = []
        dev = device
        t0 = time.time()
        Tc = 2048
        xbuf = torch.empty(B * Tc * hid, dtype=torch.bfloat16, device=dev)
        gemm_ws = torch.empty(ops.L.load().csa2_compress_workspace_size(B, Tc, hid, 2) + 256,
                              dtype=torch.uint8, device=dev)
        pre_buf = torch.empty(B * Tc * 512, dtype=torch.float32, device=dev)
        for l in range(self.n_layers):
            s = seed_base + l
            md = self.modes[l]
            g = {}
            g["q"] = sg.fill_normal(torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev), s, 5, 0, 1.28)
            g["swa_kv"] = sg.fill_normal(torch.empty(B, W, 512, dtype=torch.bfloat16, device=dev), s, 8)
            g["swa_len"], g["swa_pos0"] = W, self.t - W + 1
            if wl.get("stored"):
                g["swa_codes"] = torch.empty(B, W, 512, dtype=torch.uint8, device=dev)
                g["swa_scales"] = torch.empty(B, W, 8, dtype=torch.uint8, device=dev)
                ops.swa_kv_quant_fp8(g["swa_kv"], 0, W, g["swa_codes"], g["swa_scales"])
            g["out"] = torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device=dev)
            if md in (1, 2):
                g["q_idx"] = sg.fill_normal(torch.empty(B, 1, 32, 128, dtype=torch.bfloat16, device=dev), s, 6, 0, 1.28)
                g["w_idx"] = sg.fill_normal(torch.empty(B, 1, 32, dtype=torch.float32, device=dev), s, 7, 0, 1.28)
            if md == 1:
                m = self.ratio[l]
                n_cap = C // m
                g["w_kv"] = sg.fill_normal(torch.empty(512, hid, dtype=torch.bfloat16, device=dev), s, 2, 0, 0.02)
                g["w_gate"] = (sg.fill_normal(torch.empty(512, hid, dtype=torch.bfloat16, device=dev), s, 3, 0, 0.02)
                               if m == 2 else None)
                g["w_ik"] = sg.fill_normal(torch.empty(128, 512, dtype=torch.bfloat16, device=dev), s, 4, 0, 0.02)
                g["norm_w"] = torch.ones(512, dtype=torch.float32, device=dev)
                g["kv_cache"] = torch.empty(B, n_cap, 512, dtype=torch.bfloat16, device=dev)
                g["idx_codes"] = torch.empty(B, n_cap, 64, dtype=torch.uint8, device=dev)
                g["idx_scales"] = torch.empty(B, n_cap, 4, dtype=torch.uint8, device=dev)
                g["n_cap"] = n_cap
                # prefix: tokens 0 .. C-m-1 through the library's compressor, in chunks
                n_prefix = C - m
                for p0 in range(0, n_prefix, Tc):
                    tc = min(Tc, n_prefix - p0)
                    x = xbuf[: B * tc * hid].view(B, tc, hid)
                    for b in range(B):
                        sg.fill_normal(x[b], s, 1, (b * C + p0) * hid)
                    pre = pre_buf[: B * (tc // m) * 512].view(B, tc // m, 512)
                    ops.compress(x, g["w_kv"], g["w_gate"], g["norm_w"], m, p0, g["kv_cache"],
                                 kv_pre=pre, workspace=gemm_ws)
                    ops.index_k_quant(pre, p0 // m, m, g["w_ik"], g["idx_codes"], g["idx_scales"])
                if wl.get("stored"):
                    g["kv_codes"] = torch.empty(B, n_cap, 256, dtype=torch.uint8, device=dev)
                    g["kv_scales"] = torch.empty(B, n_cap, 32, dtype=torch.uint8, device=dev)
                    ops.main_kv_quant_fp4(g["kv_cache"], 0, n_prefix // m, g["kv_codes"], g["kv_scales"])
                xs = torch.empty(B, m, hid, dtype=torch.bfloat16, device=dev)
                for b in range(B):
                    sg.fill_normal(xs[b], s, 1, (b * C + n_prefix) * hid)
                g["x"], g["x_tokens"], g["x_pos0"] = xs, m, n_prefix
            self.layers.append(g)
        torch.cuda.synchronize()
        del xbuf, gemm_ws, pre_buf
        log(f"[bench] caches built in {time.time() - t0:.1f}s")
        self.ios = [ops.layer_io(**g) for g in self.layers]
        max_n = max((g["x_pos0"] + g["x_tokens"]) // self.ratio[l]
                    for l, g in enumerate(self.layers) if "x" in g)
        nbytes = self.runner.workspace_size(self.params, 2, max_n)
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=dev)
        # a step that moves less than 4x the L2 (129 MB) could find the previous step's rows
        # there: such workloads overwrite a 512 MB buffer before every timed step, outside
        # the step's events
        self.step_bytes = sum(self.stage_bytes(l, s) for l in range(self.n_layers) for s in range(6))
        self.flush_buf = (torch.empty(512 << 20, dtype=torch.uint8, device=dev)
                          if self.step_bytes < 4 * 129e6 else None)

    def flush_l2(self, stream=None):
        if self.flush_buf is not None:
            import torch
            with torch.cuda.stream(stream or torch.cuda.current_stream()):
                self.flush_buf.fill_(1)

    def step(self, stream=None):
        self.runner.step(self.params, self.ios, self.ws, stream)

    def stage_bytes(self, l, stage):
        """Algorithmic HBM bytes of one stage launch (each byte the method must move once)."""
        wl = self.wl
        B, H, k, W, hid = wl["B"], wl["H"], wl["k"], wl["window"], wl["hidden"]
        md = self.modes[l]
        if stage == 5:
            if wl.get("stored"):   # FP4 entries (288 B), FP8 window rows (520 B)
                rows_bytes = (k * 288 if md != 0 else 0) + W * 520
            else:
                rows_bytes = ((k if md != 0 else 0) + W) * 1024
            return B * rows_bytes + 2 * B * H * 512 * 2 + (B * k * 4 if md != 0 else 0)
        if md == 1:
            m = self.ratio[l]
            N = wl["C"] // m
            if stage == 0:
                return ((512 * hid * 2) * (2 if m == 2 else 1) + B * m * hid * 2 + B * 1024 + B * 2048 +
                        (B * (1024 + 288) if wl.get("stored") else 0))
            if stage == 1:
                return 128 * 512 * 2 + B * 2048 + B * 68
            if stage == 2:
                return B * N * 68 + B * (32 * 128 * 2 + 32 * 4)
            if stage == 3:
                return B * N * 4 + B * k * 4
            if stage == 4:
                return B * (N // wl["blk"]) * 4 + B * wl["nb"] * 4 if self.builds_pool[l] else 0
        if md == 2:
            pool = wl["nb"] * wl["blk"]
            if stage == 2:
                return B * pool * 68 + B * wl["nb"] * 4 + B * (32 * 128 * 2 + 32 * 4)
            if stage == 3:
                return B * pool * 4 + B * k * 4
        return 0


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(wl, n_seq=1, seed=77):
    """Float64 oracle inputs for n_seq sequences of the workload (values from a fast
    NumPy generator: this leg only times the oracle)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    kv_src, idx_src, ratio = layer_tables(wl.get("pattern", "stack40"))
    C, H, hid, W = wl["C"], wl["H"], wl["hidden"], wl["window"]
    t = C - 1
    layers = []
    for l in range(len(kv_src)):
        d = {"q": rng.standard_normal((n_seq, 1, H, 512)) * 1.28,
             "swa": rng.standard_normal((n_seq, W, 512)), "swa_pos0": t - W + 1}
        if idx_src[l] == l:
            d["q_idx"] = rng.standard_normal((n_seq, 1, 32, 128)) * 1.28
            d["w_idx"] = rng.standard_normal((n_seq, 1, 32)) * 1.28
        if kv_src[l] == l:
            m = ratio[l]
            n0 = (C - m) // m
            d.update(x=rng.standard_normal((n_seq, m, hid)), x_pos0=C - m,
                     w_kv=rng.standard_normal((512, hid)) * 0.02,
                     w_gate=rng.standard_normal((512, hid)) * 0.02 if m == 2 else None,
                     gamma=np.ones(512), w_ik=rng.standard_normal((128, 512)) * 0.02,
                     prev_kv=rng.standard_normal((n_seq, n0, 512)),
                     prev_codes=rng.integers(0, 256, (n_seq, n0, 64), dtype=np.uint8),
                     prev_scales=rng.integers(0x18, 0x58, (n_seq, n0, 4), dtype=np.uint8))
        layers.append(d)
    return kv_src, idx_src, ratio, layers


def time_oracle(wl, budget_s=12.0, max_reps=4, sample=None):
    from oracle import layers as Lr
    kv_src, idx_src, ratio, layers = sample or oracle_sample(wl)
    t = wl["C"] - 1
    reps, total = 0, 0.0
    while reps < max_reps and (reps == 0 or total < budget_s):
        t0 = time.perf_counter()
        Lr.run_step(kv_src, idx_src, ratio, layers, 1, 1, t, wl["k"], hsi_blk=wl["blk"],
                    hsi_nb=wl["nb"], window=wl["window"])
        total += time.perf_counter() - t0
        reps += 1
    return reps, total


# ----------------------------------------------------------------------------- ranks
# Multi-GPU runs are independent replicas (decode sequences share nothing): each rank builds
# its own caches from its own seeds and times the same step; the job's time is the slowest
# rank's and its throughput counts every rank's batch.  No collective touches the data path.
def replica_seed_base(rank):
    return 5000 + 100 * rank


def max_over_ranks(ms, world, device=None):
    """The slowest rank's time; every rank returns it (an all-reduce of one number)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([float(ms)], device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch, world, ms):
    """Tokens per second of the whole job: every rank decodes `batch` sequences per step."""
    return batch * world / (ms * 1e-3)


# ----------------------------------------------------------------------------- main arms
def workload_config(wl, world):
    """The `config` object both arms print: the workload's name and shape."""
    n_layers = len(layer_tables(wl.get("pattern", "stack40"))[0])
    return {"workload": f"csa2_decode_{PATTERN_NAMES[wl.get('pattern', 'stack40')]}_b{wl['B']}_ctx{wl['C']}" +
                        (f"_hsi{wl['nb']}x{wl['blk']}" if wl["blk"] != 64 else "") +
                        ("_fp4kv_fp8swa" if wl.get("stored") else ""),
            "batch": wl["B"], "context": wl["C"], "layers": n_layers, "heads": wl["H"], "topk": wl["k"],
            "window": wl["window"], "hsi": f"{wl['nb']}x{wl['blk']}",
            "kv_format": "fp4 main kv, fp8 window rows" if wl.get("stored") else "bf16",
            "l2": "no flush: each step reads ~3.5 GB of caches (> 129 MB L2)",
            "parallelism": "replicas" if world > 1 else "single"}


def run_indexer_prefill(args):
    """The indexer of the 16384-token encoder prefill on its own: 16384 queries x 8192 FP4
    index keys (m = 2, causal), 32 heads x 128, top-512; W warm-up calls, then the median of
    K (at least 10) CUDA-event timed calls.  One JSON line; not the bench line."""
    import numpy as np
    import torch
    from compressed_sparse_attention_04_gb300 import build, ops
    from synth import gpu as sg
    build.build_all()
    Tq, N, m, k, seed = 16384, 8192, 2, 512, 9500
    codes = torch.empty(1, N, 64, dtype=torch.uint8, device="cuda")
    scales = torch.empty(1, N, 4, dtype=torch.uint8, device="cuda")
    r = torch.empty(N * 68, dtype=torch.int32, device="cuda")
    sg.fill_u32(r, seed, 3, 0)
    r = r.view(1, N, 68)
    codes[:] = (r[..., :64] & 0xFF).to(torch.uint8)
    scales[:] = (0x18 + (r[..., 64:] & 0x3F)).to(torch.uint8)
    qi = sg.fill_normal(torch.empty(1, Tq, 32, 128, dtype=torch.bfloat16, device="cuda"), seed, 1, 0, 1.28)
    w = sg.fill_normal(torch.empty(1, Tq, 32, dtype=torch.float32, device="cuda"), seed, 2, 0, 1.28)
    topk = torch.empty(1, Tq, k, dtype=torch.int32, device="cuda")
    call = lambda: ops.indexer_score_topk(qi, w, 0, codes, scales, N, m, k, topk_out=topk)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ts = []
    for _ in range(max(args.steps, 10)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    assert ops.last_device_status() == 0
    pairs = sum(min((i + 1) // m, N) for i in range(Tq))
    gflop = pairs * 32 * 128 * 2 / 1e9
    ms = float(np.median(ts))
    print(json.dumps({"metric": "indexer call (scores + top-k), 16384-token prefill", "ms_per_call": ms,
                      "causal_pairs": pairs, "fp4_gflop": gflop,
                      "note": "the scorer kernel's own time comes from the ncu launch list"}), flush=True)
    return 0


PREFILL = {
    # the 16384-token encoder macro-group: 1 Full (m = 2) + 5 Reuse layers, 64 heads, top-512
    "prefill16k": dict(B=1, T=16384, hidden=4096, m=2, k=512, H=64, window=128, n_reuse=5),
    # one Full layer over 1024 tokens, 16 heads, top-128
    "prefill1k": dict(B=1, T=1024, hidden=4096, m=2, k=128, H=16, window=128, n_reuse=0),
}


def prefill_flops(wl):
    """Algorithmic work of one prefill pass: the compressor's projections (bf16), the
    indexer's causal FP4 products, every layer's attention (S and P V, bf16)."""
    T, m, k, W, H, hid = wl["T"], wl["m"], wl["k"], wl["window"], wl["H"], wl["hidden"]
    N = T // m
    comp = 2.0 * wl["B"] * T * hid * 512 * (2 if m == 2 else 1)
    pairs = sum(min((t + 1) // m, N) for t in range(T)) * wl["B"]
    idx = pairs * 32 * 128 * 2.0
    rows = sum(min(k, min((t + 1) // m, N)) + min(W, t + 1) for t in range(T)) * wl["B"]
    attn = (1 + wl["n_reuse"]) * rows * 4.0 * H * 512
    return {"compress": comp, "indexer_scores": idx, "sparse_attn": attn, "causal_pairs": pairs}


def fp4_peak_tflops():
    """Dense FP4 rate of this GPU from the library's tensor-rate probe (M 128 x N 256)."""
    import ctypes as C
    from compressed_sparse_attention_04_gb300 import build
    lib = C.CDLL(os.path.join(os.path.dirname(build.__file__), "peak", "libcsa2_peak.so"))
    f = lib.csa2peak_mxf4
    f.argtypes = [C.c_int, C.c_int, C.c_int, C.POINTER(C.c_double), C.POINTER(C.c_double)]
    tf, ms = C.c_double(), C.c_double()
    rc = f(128, 256, 8192, C.byref(tf), C.byref(ms))
    return tf.value if rc == 0 else None


def run_gather_rate(args):
    """DRAM read rate of row gathers through 16-byte cp.async on this GPU (the library's
    gather probe: one CTA per SM, row indices staged in shared memory, 512 MB per launch after
    an L2-evicting write), random and contiguous rows of 256 B .. 4 KB.  One JSON line."""
    import ctypes as C
    from compressed_sparse_attention_04_gb300 import build
    build.build_all()
    lib = C.CDLL(os.path.join(os.path.dirname(build.__file__), "peak", "libcsa2_peak.so"))
    f = lib.csa2peak_gather
    f.argtypes = [C.c_int, C.c_int, C.POINTER(C.c_double), C.POINTER(C.c_double)]
    res = {}
    for rb in (256, 512, 1024, 2048, 4096):
        for rnd in (1, 0):
            g, ms = C.c_double(), C.c_double()
            rc = f(rb, rnd, C.byref(g), C.byref(ms))
            if rc != 0:
                raise RuntimeError(f"gather probe failed: CUDA error {rc}")
            res[f"{rb}B_{'random' if rnd else 'contiguous'}"] = round(g.value, 1)
    print(json.dumps({"metric": "row-gather DRAM read rate (cp.async, one CTA per SM, 192 KB in flight)",
                      "unit": "GB/s", "rates": res}), flush=True)
    return 0


def time_oracle_prefill(wl, n_sample=32, seed=78):
    """The float64 oracle on the same prefill, timed on a bounded sample: the Full layer's
    compressor and index keys over every token, then the indexer + top-k + attention of
    n_sample queries spread over the sequence, and one Reuse layer's attention for the same
    queries; per-query costs are scaled to all queries and all Reuse layers."""
    import numpy as np
    from oracle import csa2_ref as R
    rng = np.random.default_rng(seed)
    T, m, k, W, H, hid = wl["T"], wl["m"], wl["k"], wl["window"], wl["H"], wl["hidden"]
    x = rng.standard_normal((1, T, hid))
    w_kv, w_gate = rng.standard_normal((512, hid)) * 0.02, rng.standard_normal((512, hid)) * 0.02
    w_ik = rng.standard_normal((128, 512)) * 0.02
    t0 = time.perf_counter()
    kv, pre = R.compress(x, w_kv, w_gate if m == 2 else None, np.ones(512), m, 0)
    N = kv.shape[1]
    kq = R.index_k(pre, w_ik, np.broadcast_to(m * np.arange(N), (1, N)))
    codes, scales = R.index_k_quant(kq)
    k_hat = R.fp4.dequantize_rows(codes, scales)[0]
    kv_b = R.bf16_to_f64(R.f64_to_bf16_bits(kv))[0]
    t_build = time.perf_counter() - t0
    swa = rng.standard_normal((T, 512))
    qs = [int(v) for v in np.linspace(T // 8, T - 1, n_sample)]
    t_full = t_reuse = 0.0
    for t in qs:
        q_idx = rng.standard_normal((32, 128)) * 1.28
        w = rng.standard_normal(32) * 1.28
        q = rng.standard_normal((H, 512)) * 1.28
        t1 = time.perf_counter()
        nv = R.n_visible(t, m, N)
        sc = R.indexer_scores(R.quant_query(q_idx), w, k_hat[:nv])
        sel = R.topk(sc, np.ones(nv, dtype=bool), k)
        R.sparse_attention(q, R.attention_rows(kv_b, sel, swa, 0, t, W))
        t2 = time.perf_counter()
        R.sparse_attention(q, R.attention_rows(kv_b, sel, swa, 0, t, W))
        t3 = time.perf_counter()
        t_full += t2 - t1
        t_reuse += t3 - t2
    total = t_build + T / n_sample * (t_full + wl["n_reuse"] * t_reuse)
    return total, (f"Full layer compressor + index keys over all {T} tokens timed in full "
                   f"({t_build:.2f} s); indexer + top-k + attention of {n_sample} queries spread "
                   f"over the sequence and one Reuse layer's attention for them, scaled to {T} "
                   f"queries and {wl['n_reuse']} Reuse layers (extrapolated)")


def run_prefill(args):
    """One prefill pass through the runner (a Full layer and its Reuse layers): tokens/s,
    the per-stage times, and each contraction's rate against its tensor peak.  One JSON
    line; the decode step stays the bench line."""
    import numpy as np
    import torch
    import ctypes as C
    from compressed_sparse_attention_04_gb300 import build, ops
    from synth import gpu as sg
    build.build_all()
    wl = PREFILL[args.workload]
    B, T, hid, m, k, H, W, n_re = (wl[x] for x in ("B", "T", "hidden", "m", "k", "H", "window", "n_reuse"))
    n_layers = 1 + n_re
    dev = torch.device("cuda", 0)
    kv_src, idx_src, ratio = [0] * n_layers, [0] * n_layers, [m] + [0] * n_re
    runner = ops.Runner(kv_src, idx_src, ratio, 64, 64)
    params = ops.Runner.params(B, T, 0, H, hid, k, W)
    N = T // m
    gs = []
    for l in range(n_layers):
        s = 7000 + l
        g = dict(q=sg.fill_normal(torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=dev), s, 5, 0, 1.28),
                 swa_kv=sg.fill_normal(torch.empty(B, T, 512, dtype=torch.bfloat16, device=dev), s, 8),
                 swa_len=T, swa_pos0=0, out=torch.empty(B, T, H, 512, dtype=torch.bfloat16, device=dev))
        if l == 0:
            g.update(x=sg.fill_normal(torch.empty(B, T, hid, dtype=torch.bfloat16, device=dev), s, 1),
                     w_kv=sg.fill_normal(torch.empty(512, hid, dtype=torch.bfloat16, device=dev), s, 2, 0, 0.02),
                     w_gate=sg.fill_normal(torch.empty(512, hid, dtype=torch.bfloat16, device=dev), s, 3, 0, 0.02)
                     if m == 2 else None,
                     w_ik=sg.fill_normal(torch.empty(128, 512, dtype=torch.bfloat16, device=dev), s, 4, 0, 0.02),
                     norm_w=torch.ones(512, dtype=torch.float32, device=dev),
                     kv_cache=torch.empty(B, N, 512, dtype=torch.bfloat16, device=dev),
                     idx_codes=torch.empty(B, N, 64, dtype=torch.uint8, device=dev),
                     idx_scales=torch.empty(B, N, 4, dtype=torch.uint8, device=dev),
                     n_cap=N, x_tokens=T, x_pos0=0,
                     q_idx=sg.fill_normal(torch.empty(B, T, 32, 128, dtype=torch.bfloat16, device=dev), s, 6, 0, 1.28),
                     w_idx=sg.fill_normal(torch.empty(B, T, 32, dtype=torch.float32, device=dev), s, 7, 0, 1.28))
        gs.append(g)
    ios = [ops.layer_io(**g) for g in gs]
    ws = torch.empty(runner.workspace_size(params, T, N) + 256, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        runner.step(params, ios, ws)
    torch.cuda.synchronize()
    assert ops.last_device_status() == 0
    lib = ops.L.load()
    n_ev = n_layers * 6 * 2
    K = max(args.steps, 3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    for es in evs:
        for e in es:
            e.record(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    n0 = lib.csa2_kernel_launches()
    t0.record(stream)
    for _ in range(K):
        runner.step(params, ios, ws)
    t1.record(stream)
    torch.cuda.synchronize()
    ck = clocks.stop()
    launches = lib.csa2_kernel_launches() - n0
    ms = t0.elapsed_time(t1) / K
    stage_ms = [0.0] * 6
    for i in range(K):
        h = (C.c_void_p * n_ev)(*[e.cuda_event for e in evs[i]])
        ops.L.check(lib.csa2_runner_set_timing(runner._h, h, n_ev), "set_timing")
        runner.step(params, ios, ws)
    lib.csa2_runner_set_timing(runner._h, None, 0)
    torch.cuda.synchronize()
    assert ops.last_device_status() == 0
    for i in range(K):
        for l in range(n_layers):
            for st_ in range(6):
                a, b = evs[i][(l * 6 + st_) * 2], evs[i][(l * 6 + st_) * 2 + 1]
                if (l > 0 and st_ < 5):
                    continue
                stage_ms[st_] += a.elapsed_time(b) / K
    fl = prefill_flops(wl)
    bf16_peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16_peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        bf16_peak = 1900.0
    fp4_meas = fp4_peak_tflops()
    fp4_recipe = bf16_peak * 6.0

    def rate(name, flops, peak):
        t = stage_ms[STAGE_NAMES.index(name)]
        tf = flops / (t * 1e-3) / 1e12 if t > 0 else None
        return {"tflops": tf, "peak_tflops": peak, "frac": (tf / peak) if (tf and peak) else None,
                "ms": t, "gflop": flops / 1e9}

    tensor = {"compress": rate("compress", fl["compress"], bf16_peak),
              "indexer_scores": rate("indexer_scores", fl["indexer_scores"], fp4_meas),
              "sparse_attn": rate("sparse_attn", fl["sparse_attn"], bf16_peak)}
    tensor["indexer_scores"]["frac_of_recipe_peak"] = (
        tensor["indexer_scores"]["tflops"] / fp4_recipe if tensor["indexer_scores"]["tflops"] else None)
    # dominant kernel against its tensor peak: FLOPs per launch / mean launch time
    dom = max(tensor, key=lambda n: tensor[n]["ms"])
    n_launch = n_layers if dom == "sparse_attn" else 1
    roof = {"bound": "tensor", "kernel": dom, "achieved": tensor[dom]["tflops"],
            "peak": tensor[dom]["peak_tflops"], "peak_kind": "measured", "unit": "TFLOP/s",
            "frac": tensor[dom]["frac"], "traffic": None, "launches_per_step": n_launch,
            "flops_per_launch": tensor[dom]["gflop"] * 1e9 / n_launch}
    e2e = None
    if not args.no_e2e:
        e2e = prefill_e2e(runner, params, gs, ws, stream, args, B * T)
    cpu = None
    if not args.no_cpu_baseline:
        tot, desc = time_oracle_prefill(wl)
        cpu = {"value": B * T / tot, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": desc}
    line = {"metric": f"CSA2 prefill tokens/s ({T}-token group, 1 Full + {n_re} Reuse layers)",
            "value": B * T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"csa2_prefill_{n_layers}layer_T{T}", "batch": B, "tokens": T,
                       "hidden": hid, "m": m, "topk": k, "heads": H, "window": W,
                       "l2": f"no flush: a pass reads {6 * T * H * 512 * 2 / 1e9:.1f} GB of queries alone"},
            "stage_ms_per_step": {STAGE_NAMES[i]: stage_ms[i] for i in range(6)},
            "tensor": tensor, "fp4_peak_tflops": {"measured": fp4_meas, "recipe_bf16x6": fp4_recipe},
            "roofline": roof, "causal_pairs": fl["causal_pairs"], "gpu_launches": launches // K,
            "clocks": ck, "cpu_baseline": cpu, "e2e": e2e}
    print(json.dumps(line), flush=True)
    return 0


def prefill_e2e(runner, params, gs, ws, stream, args, tokens):
    """The prefill pass through the C ABI with host buffers: each step copies every layer's
    inputs (hidden states, queries, window rows, indexer queries and weights) from pinned host
    memory, runs the pass and reads the last layer's output back; copies and pass in order on
    one stream, all inside the timed region."""
    import torch
    from compressed_sparse_attention_04_gb300 import ops
    keys = ("x", "q", "swa_kv", "q_idx", "w_idx")
    pairs, h2d = [], 0
    for g in gs:
        for key in keys:
            if key in g and g[key] is not None:
                h = torch.empty_like(g[key], device="cpu").pin_memory()
                h.copy_(g[key])
                pairs.append((g[key], h))
                h2d += g[key].numel() * g[key].element_size()
    out_h = torch.empty_like(gs[-1]["out"], device="cpu").pin_memory()
    d2h = out_h.numel() * out_h.element_size()
    ios = [ops.layer_io(**g) for g in gs]

    def one():
        for d, h in pairs:
            d.copy_(h, non_blocking=True)
        runner.step(params, ios, ws, stream.cuda_stream)
        out_h.copy_(gs[-1]["out"], non_blocking=True)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    K = max(args.steps, 3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(K):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    assert ops.last_device_status() == 0
    ms = max(e0.elapsed_time(e1), wall * 1e3) / K
    return {"value": tokens / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "no: uploads, pass and read-back in order on one stream"}


def run_attention_formats(args):
    """The decode attention launch at the headline shape (64 rows x (512 entries + 128 window
    rows) x 64 heads, 64K-entry caches) with each stored format: bf16, FP8 window rows, FP4
    entries, both.  Per format: W warm-up launches, then the mean of 40 back-to-back launches
    (CUDA events).  One JSON line; not the bench line."""
    import torch
    from compressed_sparse_attention_04_gb300 import build, ops
    from synth import gpu as sg
    build.build_all()
    B, N, H, k, S = 64, 65536, 64, 512, 256
    t = 131071
    q = sg.fill_normal(torch.empty(B, 1, H, 512, dtype=torch.bfloat16, device="cuda"), 1, 1, 0, 1.28)
    kv = sg.fill_normal(torch.empty(B, N, 512, dtype=torch.bfloat16, device="cuda"), 1, 2)
    codes = torch.empty(B, N, 256, dtype=torch.uint8, device="cuda")
    scales = torch.empty(B, N, 32, dtype=torch.uint8, device="cuda")
    ops.main_kv_quant_fp4(kv, 0, N, codes, scales)
    swa = sg.fill_normal(torch.empty(B, S, 512, dtype=torch.bfloat16, device="cuda"), 1, 3)
    wc = torch.empty(B, S, 512, dtype=torch.uint8, device="cuda")
    wsc = torch.empty(B, S, 8, dtype=torch.uint8, device="cuda")
    ops.swa_kv_quant_fp8(swa, 0, S, wc, wsc)
    # 512 distinct ascending entries per row, spread over the cache
    base = (torch.arange(k, device="cuda", dtype=torch.int64) * N) // k
    off = (torch.arange(B, device="cuda", dtype=torch.int64) * 37) % (N // k)
    topk = (base[None, :] + off[:, None]).to(torch.int32).view(B, 1, k).contiguous()
    out = torch.empty(B, 1, H, 512, device="cuda", dtype=torch.bfloat16)
    runs = {"bf16": lambda: ops.sparse_attn(q, t, kv, N, topk, swa, t - S + 1, out=out),
            "fp8_window": lambda: ops.sparse_attn(q, t, kv, N, topk, None, t - S + 1, out=out,
                                                  swa_fp8=(wc, wsc)),
            "fp4_entries": lambda: ops.sparse_attn(q, t, None, N, topk, swa, t - S + 1, out=out,
                                                   kv_fp4=(codes, scales)),
            "fp4_entries_fp8_window": lambda: ops.sparse_attn(q, t, None, N, topk, None, t - S + 1,
                                                              out=out, kv_fp4=(codes, scales),
                                                              swa_fp8=(wc, wsc))}
    res = {}
    for name, f in runs.items():
        for _ in range(args.warmup):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(40):
            f()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) * 1000 / 40
    assert ops.last_device_status() == 0
    print(json.dumps({"metric": "decode attention launch, 64 x (512 + 128) rows x 64 heads",
                      "unit": "us per launch (back to back)", "per_format": res}), flush=True)
    return 0


def run_reference(args, wl, rank, world):
    if rank != 0:
        return 0
    sample = oracle_sample(wl)
    for _ in range(args.warmup):
        time_oracle(wl, budget_s=0, max_reps=1, sample=sample)
    reps, total = 0, 0.0
    for _ in range(args.steps):
        r, tt = time_oracle(wl, budget_s=0, max_reps=1, sample=sample)
        reps += r
        total += tt
    v = reps / total
    cores = os.cpu_count()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / reps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(wl, world),
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "one sequence of the decode step per timed step (B=1 of the "
                                       f"{wl['B']}-sequence batch, full-size caches)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, wl, rank, world, local_rank):
    import torch
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    from compressed_sparse_attention_04_gb300 import build
    if rank == 0:
        build.build_all()
    if world > 1:
        torch.distributed.barrier()
    log = (lambda *a: print(*a, file=sys.stderr, flush=True)) if rank == 0 else (lambda *a: None)
    st = Stack(wl, dev, seed_base=replica_seed_base(rank), log=log)
    stream = torch.cuda.current_stream(dev)
    B = wl["B"]
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    from compressed_sparse_attention_04_gb300 import ops  # noqa: F401
    assert ops.last_device_status() == 0, "device-side check fired during warm-up"

    # per-stage timing events, one array per timed step
    n_ev = st.n_layers * 6 * 2
    import ctypes as C
    lib = ops.L.load()
    ev_sets, handles = [], []
    for _ in range(args.steps):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
        for e in evs:
            e.record(stream)            # creates the CUDA event
        ev_sets.append(evs)
        handles.append((C.c_void_p * n_ev)(*[e.cuda_event for e in evs]))
    torch.cuda.synchronize()

    # Two timed passes of K steps each.  Pass A gives the headline: the runner records no
    # per-stage events.  Pass B repeats the K steps with one event pair per (layer, stage) on
    # the launching stream, for the per-stage times and the roofline of the dominant kernel.
    # With --graph every step of a pass is one CUDA graph of the runner's launches, captured
    # and uploaded before the timed region.
    def make_graphs(with_events):
        cap = torch.cuda.Stream(dev)
        gs = []
        n0 = lib.csa2_kernel_launches()
        for i in range(args.steps):
            if with_events:
                ops.L.check(lib.csa2_runner_set_timing(st.runner._h, handles[i], n_ev), "set_timing")
            else:
                lib.csa2_runner_set_timing(st.runner._h, None, 0)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                st.step(cap.cuda_stream)
            gs.append(g)
        per_step = (lib.csa2_kernel_launches() - n0) // args.steps
        lib.csa2_runner_set_timing(st.runner._h, None, 0)
        for g in gs:
            g.replay()
        torch.cuda.synchronize()
        assert ops.last_device_status() == 0, "device-side check fired in the graph upload"
        return gs, per_step

    def timed_pass(with_events, graphs):
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        flush = st.flush_buf is not None
        # back to back: one event pair around the K steps; with an L2 flush before every
        # step: one pair per step, the flush outside it
        n_pairs = args.steps if flush else 1
        t0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_pairs)]
        t1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_pairs)]
        n_launch0 = lib.csa2_kernel_launches()
        if not flush:
            t0[0].record(stream)
        for i in range(args.steps):
            if flush:
                st.flush_l2(stream)
                t0[i].record(stream)
            if graphs:
                graphs[0][i].replay()
            else:
                if with_events:
                    ops.L.check(lib.csa2_runner_set_timing(st.runner._h, handles[i], n_ev), "set_timing")
                st.step()
            if flush:
                t1[i].record(stream)
        if not flush:
            t1[0].record(stream)
        launches = graphs[1] * args.steps if graphs else lib.csa2_kernel_launches() - n_launch0
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        lib.csa2_runner_set_timing(st.runner._h, None, 0)
        total = sum(a.elapsed_time(b) for a, b in zip(t0, t1))
        ms_ = max_over_ranks(total / args.steps, world, dev)
        assert ops.last_device_status() == 0, "device-side check fired during the timed steps"
        return ms_, launches

    lib.csa2_runner_set_timing(st.runner._h, None, 0)
    graphs_a = make_graphs(False) if args.graph else None
    graphs_b = make_graphs(True) if args.graph else None
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.5)
    ms, n_launches = timed_pass(False, graphs_a)
    ck = clocks.stop()
    ms_b, _ = timed_pass(True, graphs_b)

    # per-stage totals over the timed steps
    stage_ms = [0.0] * 6
    stage_bytes = [0] * 6
    stage_launches = [0] * 6
    for i in range(args.steps):
        evs = ev_sets[i]
        for l in range(st.n_layers):
            for s in range(6):
                a, b = evs[(l * 6 + s) * 2], evs[(l * 6 + s) * 2 + 1]
                nb = st.stage_bytes(l, s)
                if nb == 0:
                    continue
                stage_ms[s] += a.elapsed_time(b)
                stage_bytes[s] += nb
                stage_launches[s] += 1
    dom = max(range(6), key=lambda s: stage_ms[s])
    peak, peak_kind = peaks()
    achieved = stage_bytes[dom] / (stage_ms[dom] * 1e-3) / 1e9
    hot = [2, 3, 4, 5]
    hot_ms = sum(stage_ms[s] for s in hot)
    hot_gbs = sum(stage_bytes[s] for s in hot) / (hot_ms * 1e-3) / 1e9

    # end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e and not wl.get("stored"):
        e2e = run_e2e(st, args, stream)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not wl.get("stored"):
        reps, total = time_oracle(wl)
        cpu = {"value": reps / total, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{reps} x one sequence of the decode step (all {st.n_layers} layers, full-size "
                         "caches, cache building excluded as on the GPU); NumPy float64, BLAS threads "
                         "= host cores"}
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": job_throughput(B, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(workload_config(wl, world),
                       l2=(f"no flush: each step moves {st.step_bytes / 1e9:.2f} GB (> 4 x the 129 MB L2)"
                           if st.flush_buf is None else
                           f"each step moves {st.step_bytes / 1e6:.0f} MB: a 512 MB buffer is written "
                           "before every timed step, outside its events"),
                       launch="cuda_graph" if args.graph else "direct",
                       timing="headline pass without per-stage events; stage times from a second pass"),
        "roofline": {"bound": "hbm", "kernel": STAGE_NAMES[dom], "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": attention_traffic(st.modes) if STAGE_NAMES[dom] == "sparse_attn" and
                                wl["C"] == 131072 and wl["B"] == 64 and not wl.get("stored") else None,
                     "launches_timed": stage_launches[dom]},
        "hot_path_roofline": {"stages": [STAGE_NAMES[s] for s in hot], "achieved": hot_gbs,
                              "frac": hot_gbs / peak, "frac_of_nominal_8tbs": hot_gbs / NOMINAL_HBM_GBS,
                              "unit": "GB/s"},
        "stage_ms_per_step": {STAGE_NAMES[s]: stage_ms[s] / args.steps for s in range(6)},
        "ms_per_step_with_stage_events": ms_b,
        "gpu_launches": n_launches,
        "clocks": ck,
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_e2e(st, args, stream):
    """Same step measured through the C ABI with host inputs and outputs: each step copies
    its inputs (every layer's queries, indexer queries/weights, new hidden states, newest window
    row) from pinned host memory and reads the step's result, the last layer's output, back
    (the other layers' outputs are what a model's next layers consume on the device).  As a server would, steps are
    pipelined over two device copies of the per-step inputs and outputs (caches and weights
    shared): step s + 1's inputs go up on one copy stream and step s - 1's outputs come down
    on another while step s computes; events keep each buffer's uses in order.  Every step's
    copies are inside the timed region."""
    import torch
    from compressed_sparse_attention_04_gb300 import ops
    dev = stream.device
    keys = ("q", "q_idx", "w_idx", "x", "swa_kv", "out")
    sets = [st.layers]
    second = []
    for g in st.layers:
        g2 = dict(g)
        for key in keys:
            if key in g and g[key] is not None:
                g2[key] = g[key].clone()
        second.append(g2)
    sets.append(second)
    ios = [st.ios, [ops.layer_io(**g) for g in second]]
    h2d, d2h, host_in, host_out = 0, 0, [], []
    for g in st.layers:
        for key in ("q", "q_idx", "w_idx", "x"):
            if key in g and g[key] is not None:
                h = torch.empty_like(g[key], device="cpu").pin_memory()
                h.copy_(g[key])
                host_in.append((key, h))
                h2d += g[key].numel() * g[key].element_size()
        row = g["swa_kv"][:, -1]
        h = torch.empty(row.shape, dtype=row.dtype).pin_memory()
        h.copy_(row)
        host_in.append(("swa_row", h))
        h2d += row.numel() * row.element_size()
    g = st.layers[-1]
    host_out.append(torch.empty_like(g["out"], device="cpu").pin_memory())
    d2h += g["out"].numel() * g["out"].element_size()

    def dev_inputs(si):
        out = []
        for g in sets[si]:
            for key in ("q", "q_idx", "w_idx", "x"):
                if key in g and g[key] is not None:
                    out.append(g[key])
            out.append(g["swa_kv"][:, -1])
        return out
    dst_in = [dev_inputs(0), dev_inputs(1)]
    # NC streams per direction, so that the copies can use more than one copy engine
    # (measured: 1 stream 2.44 ms per step, 2 2.17, 4 2.03, 8 2.52)
    NC = 4
    ups = [torch.cuda.Stream(dev) for _ in range(NC)]
    downs = [torch.cuda.Stream(dev) for _ in range(NC)]
    in_ready = [[torch.cuda.Event() for _ in range(NC)] for _ in range(2)]
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    out_read = [[torch.cuda.Event() for _ in range(NC)] for _ in range(2)]
    used = [False, False]

    def one(s):
        si = s & 1
        for u, up in enumerate(ups):
            with torch.cuda.stream(up):
                if used[si]:
                    up.wait_event(computed[si])      # step s - 2 has read these inputs
                for j, (d, (_, h)) in enumerate(zip(dst_in[si], host_in)):
                    if j % NC == u:
                        d.copy_(h, non_blocking=True)
                in_ready[si][u].record(up)
        for u in range(NC):
            stream.wait_event(in_ready[si][u])
            if used[si]:
                stream.wait_event(out_read[si][u])   # step s - 2's outputs are down
        st.runner.step(st.params, ios[si], st.ws, stream.cuda_stream)
        computed[si].record(stream)
        for u, down in enumerate(downs):
            with torch.cuda.stream(down):
                down.wait_event(computed[si])
                for j, (h, g) in enumerate(zip(host_out, sets[si][-1:])):
                    if j % NC == u:
                        h.copy_(g["out"], non_blocking=True)
                out_read[si][u].record(down)
        used[si] = True

    for s in range(args.warmup):
        one(s)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    e0.record(stream)
    for up in ups:
        up.wait_event(e0)
    for s in range(args.steps):
        one(args.warmup + s)
    for down in downs:
        stream.wait_stream(down)
    e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(e0.elapsed_time(e1), wall * 1e3) / args.steps
    return {"value": st.wl["B"] / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelined": "two device copies of the step's inputs/outputs; copies on their own streams",
            "d2h": "the step's result: the last layer's output"}


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + sorted(PREFILL), default="decode40")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--indexer-prefill", action="store_true",
                    help="time the indexer of the 16384-token prefill alone (one JSON line, not the bench line)")
    ap.add_argument("--gather-rate", action="store_true",
                    help="measure the row-gather DRAM read rate of this GPU (one JSON line)")
    ap.add_argument("--attention-formats", action="store_true",
                    help="time the decode attention launch with each stored format (one JSON line)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each timed step as a captured CUDA graph (measured 1.607 ms per step "
                         "against 1.587 ms for direct launches with programmatic dependent launch)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("[bench] warm-up raised to 3 steps (minimum)", file=sys.stderr)
        args.warmup = 3
    if args.indexer_prefill:
        return run_indexer_prefill(args)
    if args.attention_formats:
        return run_attention_formats(args)
    if args.gather_rate:
        return run_gather_rate(args)
    if args.workload in PREFILL:
        if int(os.environ.get("RANK", "0")) != 0:
            return 0   # one GPU: a prefill pass is not split over ranks
        return run_prefill(args)
    wl = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        return run_ours(args, wl, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
