"""Shared helpers for the GPU parity tests: tolerances and comparisons."""
import math

import numpy as np
import torch

# Tolerances for fp16/bf16 inputs against the FP64 oracle (absolute).
O_MAX = 2e-2
O_MEAN = 2e-3
LSE_MAX = 1e-3
# FP32 inputs: max |dO| 1e-3 (the bound stated for FP32 inputs); mean one tenth of it,
# the same ratio as the 16-bit bounds; LSE as for 16-bit inputs.
O_MAX_F32 = 1e-3
O_MEAN_F32 = 1e-4


def to_np(t):
    return t.detach().float().cpu().double().numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what="", o_max=O_MAX, o_mean=O_MEAN):
    """Element-by-element comparison; -inf LSE must match exactly."""
    og = to_np(o_gpu).reshape(o_ref.shape)
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    err = np.abs(og - o_ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    assert mx <= o_max, f"{what}: max |dO| {mx:.3e} > {o_max}"
    assert mean <= o_mean, f"{what}: mean |dO| {mean:.3e} > {o_mean}"
    if lse_gpu is not None:
        lg = to_np(lse_gpu).reshape(lse_ref.shape)
        ninf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lg), ninf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~ninf_ref
        if fin.any():
            le = float(np.abs(lg[fin] - lse_ref[fin]).max())
            assert le <= LSE_MAX, f"{what}: max |dLSE| {le:.3e} > {LSE_MAX}"
    return mx, mean


def sample_rows(B, H, Sq, BM, n_random=256, extra=(), seed=0):
    """Flat row ids (b*H + h)*Sq + i: for every (b, h) the first and the last query
    block, the rows listed in `extra`, and n_random rows drawn with a seeded generator."""
    g = torch.Generator().manual_seed(seed)
    rows = []
    last0 = ((Sq - 1) // BM) * BM
    base = list(range(min(BM, Sq))) + list(range(last0, Sq)) + [i for i in extra if 0 <= i < Sq]
    for bh in range(B * H):
        r = set(base)
        if n_random:
            r.update(torch.randint(0, Sq, (n_random,), generator=g).tolist())
        rows.extend(bh * Sq + i for i in sorted(r))
    return np.array(rows, dtype=np.int64)


def pick_rows(t, rows, Sq):
    """Gather flat rows from a [B,H,Sq,...] tensor."""
    flat = t.reshape(-1, *t.shape[3:]) if t.dim() > 3 else t.reshape(-1)
    idx = torch.as_tensor(rows, device=t.device)
    return flat.index_select(0, idx)


def scale_for(d):
    return 1.0 / math.sqrt(d)
