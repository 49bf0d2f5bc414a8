"""Shared helpers for the GPU parity tests: seeded inputs (both sides get the same
bits from the generator module) and the comparison rules.

Comparison rules
  * FP4 codes / scales, top-k sets, candidate pools: bit-exact, except where the
    oracle's float64 value sits within a stated tolerance of a decision boundary
    (a rounding midpoint, or the k-th score): there a swap is allowed and counted.
  * top-k tie rule: an element of the symmetric difference must have an oracle
    score within 1e-6 * max(|I_k|, 1e-3 * max_s |I_s|) of the k-th score I_k.
  * attention outputs (bf16): max abs error <= 2e-2 and mean abs error <= 2e-3.
  * compressor (float32 kv_pre): |gpu - oracle| <= 1e-3 * max(|oracle|, rms(row)).
"""

import numpy as np
import torch

import synth
from oracle import csa2_ref as R
from oracle import fp4

TOPK_REL = 1e-6
ATTN_MAX_ABS, ATTN_MEAN_ABS = 2e-2, 2e-3
COMPRESS_REL = 1e-3


# ------------------------------------------------------------------ inputs
def bf16_input(seed, stream, shape, sigma=1.0, device="cuda"):
    """Return (cuda bf16 tensor, float64 numpy copy) of generator elements 0..n-1."""
    n = int(np.prod(shape))
    bits = synth.normal_bf16_bits(seed, stream, 0, n, sigma).reshape(shape)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return t, R.bf16_to_f64(bits)


def f32_input(seed, stream, shape, sigma=1.0, device="cuda"):
    n = int(np.prod(shape))
    v = synth.normal_f32(seed, stream, 0, n, sigma).reshape(shape)
    return torch.from_numpy(v.copy()).to(device), v.astype(np.float64)


def u32_input(seed, stream, n):
    return synth.uniform_u32(seed, stream, 0, n)


def to_dev(a, dtype, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def index_cache_input(seed, stream, B, n_cap, zero_scale_every=97):
    """Random FP4 codes and valid E4M3 scales (no NaN), some zero-scale rows.

    Scales span 2^-4 .. 2^4 (bytes 0x18..0x57)."""
    r = u32_input(seed, stream, B * n_cap * 68).reshape(B, n_cap, 68)
    codes = (r[..., :64] & 0xFF).astype(np.uint8)
    scales = (0x18 + (r[..., 64:] % 0x40)).astype(np.uint8)
    flat = scales.reshape(-1, 4)
    flat[::zero_scale_every] = 0
    return codes, scales


def main_kv_fp4_input(seed, stream, B, n_cap):
    """Random FP4 main-KV entries: every code equally likely, one E4M3 scale per 16
    channels in 0x28..0x37 (0.25 .. 0.94: entries of unit size, like the bf16 cache)."""
    r = np.ascontiguousarray(u32_input(seed, stream, B * n_cap * 72).reshape(B, n_cap, 72))
    codes = np.ascontiguousarray(r[..., :64]).view(np.uint8).reshape(B, n_cap, 256)
    sbytes = np.ascontiguousarray(r[..., 64:]).view(np.uint8).reshape(B, n_cap, 32)
    return codes.copy(), (0x28 + sbytes % 16).astype(np.uint8)


# ------------------------------------------------------------------ comparisons
def check_topk_row(gpu, scores, valid, k, what=""):
    """Compare one GPU top-k row against the oracle under the tie rule.

    Returns the number of tolerated swaps."""
    gpu = np.asarray(gpu)
    exp = R.topk(scores, valid, k)
    n_valid = int(np.count_nonzero(valid))
    n_sel = min(k, n_valid)
    assert np.all(gpu[n_sel:] == -1), f"{what}: padding"
    sel = gpu[:n_sel]
    assert np.all(sel >= 0) and np.all(np.diff(sel) > 0), f"{what}: not ascending/valid: {sel[:10]}"
    assert np.all(valid[sel]), f"{what}: selected an entry that does not compete"
    if np.array_equal(sel, exp[:n_sel]):
        return 0
    vs = np.sort(scores[valid])[::-1]
    kth = vs[n_sel - 1]
    tol = TOPK_REL * max(abs(kth), 1e-3 * np.max(np.abs(vs)))
    diff = np.setxor1d(sel, exp[:n_sel])
    bad = [int(s) for s in diff if abs(scores[s] - kth) > tol]
    assert not bad, (f"{what}: {len(diff)} differing entries, {len(bad)} outside the tie band; "
                     f"k-th={kth!r} tol={tol:.3g} e.g. entry {bad[0]} score {scores[bad[0]]!r}")
    return len(diff) // 2


def _e2m1_margin(u):
    """Distance of |u| to the nearest E2M1 rounding midpoint."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    return np.min(np.abs(np.abs(u)[..., None] - mids), axis=-1)


def check_codes(gpu_codes, gpu_scales, k_oracle, tol=2e-5):
    """FP4 codes of keys computed in float64 by the oracle vs the GPU's codes.

    The GPU forms the key in float32 (a 4096-long projection, then 512 -> 128), so its value
    carries a relative error of a few 1e-6; tol = 2e-5 admits that and no more.
    Blocks must match bit for bit unless the oracle value lies within `tol`
    (relative) of a scale midpoint, or (elementwise) within tol * 6 of an E2M1
    midpoint in units of the scale, or within tol * scale of zero (sign).
    Returns (#blocks with a tolerated scale flip, #tolerated code flips)."""
    kf = np.asarray(k_oracle, np.float64)
    oc, os_ = R.index_k_quant(kf)
    gc = np.asarray(gpu_codes)
    gs = np.asarray(gpu_scales)
    nblk = kf.shape[-1] // 32
    kb = kf.reshape(kf.shape[:-1] + (nblk, 32))
    amax6 = np.max(np.abs(kb), axis=-1) / 6.0
    grid = fp4._E4M3_GRID
    mids = (grid[1:] + grid[:-1]) / 2
    scale_margin = np.min(np.abs(amax6[..., None] - mids), axis=-1) / np.maximum(amax6, 1e-30)
    sflip = gs != os_
    assert np.all(scale_margin[sflip] <= tol), "scale mismatch away from a rounding midpoint"
    ucodes_g = fp4.unpack_codes(gc).reshape(kb.shape)
    ucodes_o = fp4.unpack_codes(oc).reshape(kb.shape)
    s = fp4.e4m3_value(os_)
    u = kb / np.where(s == 0, 1.0, s)[..., None]
    cflip = (ucodes_g != ucodes_o) & ~sflip[..., None]
    near = (_e2m1_margin(u) <= tol * 6) | (np.abs(u) <= tol * 6)
    assert np.all(near[cflip]), f"{int(np.count_nonzero(cflip & ~near))} code mismatches away from a midpoint"
    return int(np.count_nonzero(sflip)), int(np.count_nonzero(cflip))


def check_attention(gpu_out, oracle_out, what=""):
    g = np.asarray(gpu_out, np.float64)
    o = np.asarray(oracle_out, np.float64)
    err = np.abs(g - o)
    assert err.max() <= ATTN_MAX_ABS, f"{what}: max abs err {err.max():.4g}"
    assert err.mean() <= ATTN_MEAN_ABS, f"{what}: mean abs err {err.mean():.4g}"
    return float(err.max()), float(err.mean())


def check_compress_f32(gpu_pre, oracle_pre, what=""):
    g = np.asarray(gpu_pre, np.float64)
    o = np.asarray(oracle_pre, np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True))
    bound = COMPRESS_REL * np.maximum(np.abs(o), rms)
    bad = np.abs(g - o) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1e-3 relative"
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), rms)))


def bf16_of(t):
    """float64 numpy copy of a CUDA bf16 tensor."""
    return R.bf16_to_f64(t.detach().cpu().view(torch.int16).numpy().view(np.uint16))
