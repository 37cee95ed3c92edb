"""Page append and chunked prefill into a paged KV cache, through the C ABI.

A sequence's cache is built chunk by chunk with fa_kv_append (pages from a random
permutation of a NaN-poisoned pool); fa_fwd_paged then runs the last chunk's queries
against every cached key. Checked against the FP64 oracle and, bit for bit, the cache
contents against the appended rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

from _util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_attention_06_gb300 import build
    build.build()
    fa.lib()


def build_cache(B, H, d, page, num_pages, ctx0, chunk, dtype, seed):
    """Two appends per sequence: ctx0[b] tokens from position 0, then `chunk` tokens."""
    g = torch.Generator().manual_seed(seed)
    total = [c + chunk for c in ctx0]
    npages = [-(-t // page) for t in total]
    max_pages = max(npages)
    perm = torch.randperm(num_pages, generator=g)
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        table[b, :npages[b]] = perm[off:off + npages[b]].to(torch.int32)
        off += npages[b]
    T0 = max(max(ctx0), 1)
    k0 = torch.randn(B, H, T0, d, generator=g).to(dtype)
    v0 = torch.randn(B, H, T0, d, generator=g).to(dtype)
    k1 = torch.randn(B, H, chunk, d, generator=g).to(dtype)
    v1 = torch.randn(B, H, chunk, d, generator=g).to(dtype)
    q = torch.randn(B, H, chunk, d, generator=g).to(dtype)
    dev = "cuda"
    kp = torch.full((num_pages, H, page, d), float("nan"), dtype=dtype, device=dev)
    vp = torch.full((num_pages, H, page, d), float("nan"), dtype=dtype, device=dev)
    tab = table.to(dev)
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    c0 = torch.tensor(ctx0, dtype=torch.int32, device=dev)
    fa.fa_kv_append(k0.to(dev), v0.to(dev), kp, vp, tab, zero, new_lens=c0)
    fa.fa_kv_append(k1.to(dev), v1.to(dev), kp, vp, tab, c0)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rows_k = [torch.cat([k0[b, :, :ctx0[b]], k1[b]], dim=1) for b in range(B)]
    rows_v = [torch.cat([v0[b, :, :ctx0[b]], v1[b]], dim=1) for b in range(B)]
    return q, kp, vp, table, total, rows_k, rows_v


def test_append_writes_rows_and_zero_tails_bit_exact():
    B, H, d, page = 5, 2, 64, 64
    ctx0 = [0, 1, 63, 64, 200]
    q, kp, vp, table, total, rows_k, rows_v = build_cache(B, H, d, page, 40, ctx0, 37,
                                                          torch.float16, seed=1)
    kc, vc = kp.cpu(), vp.cpu()
    used = set()
    for b in range(B):
        for t in range(total[b]):
            pg = int(table[b, t // page])
            used.add(pg)
            assert torch.equal(kc[pg, :, t % page].view(torch.int16),
                               rows_k[b][:, t].view(torch.int16))
            assert torch.equal(vc[pg, :, t % page].view(torch.int16),
                               rows_v[b][:, t].view(torch.int16))
        last = int(table[b, (total[b] - 1) // page])
        tail = total[b] % page
        if tail:
            assert torch.all(kc[last, :, tail:] == 0) and torch.all(vc[last, :, tail:] == 0)
    for pg in range(40):
        if pg not in used:
            assert torch.isnan(kc[pg].float()).all()


@pytest.mark.parametrize("page,d,dt", [(64, 64, torch.float16), (128, 128, torch.bfloat16),
                                       (256, 128, torch.float16)])
@pytest.mark.parametrize("mode,w,g", [(fa.FA_MASK_CAUSAL, 0, 0), (fa.FA_MASK_NONE, 0, 0),
                                      (fa.FA_MASK_CAUSAL_WINDOW, 300, 16),
                                      (fa.FA_MASK_BAND, 100, 0), (fa.FA_MASK_PREFIX_LM, 0, 450)])
def test_chunked_prefill_matches_oracle(page, d, dt, mode, w, g):
    B, H, chunk = 4, 3, 200
    ctx0 = [0, 57, 600, 1000]
    q, kp, vp, table, total, rows_k, rows_v = build_cache(B, H, d, page, 64, ctx0, chunk, dt,
                                                          seed=page + d)
    dev = "cuda"
    o = torch.empty(q.shape, dtype=dt, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ctx = torch.tensor(total, dtype=torch.int32)
    scale = 1 / math.sqrt(d)
    fa.fa_fwd_paged(q.to(dev), kp, vp, table.to(dev), ctx.to(dev), o, lse, scale, mode, w, g)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention_paged(q, kp.cpu(), vp.cpu(), table, ctx, scale, mode, w, g)
    compare(o, lse, ref_o, ref_l, f"paged page {page} mode {mode}")
    # the same rows through the contiguous kernel on gathered keys
    for b in range(B):
        ob = torch.empty_like(q[b:b + 1], device=dev)
        lb = torch.empty(1, H, chunk, dtype=torch.float32, device=dev)
        fa.fa_fwd(q[b:b + 1].to(dev), rows_k[b][None].to(dev).contiguous(),
                  rows_v[b][None].to(dev).contiguous(), ob, lb, scale, mode, w, g)
        torch.cuda.synchronize()
        assert (ob.float() - o[b:b + 1].float()).abs().max().item() <= 1.6e-2


def test_chunked_prefill_long_contexts():
    """32 heads of 128, 256-token pages, contexts up to 8k, 512-token chunks."""
    B, H, d, page, chunk = 4, 32, 128, 256, 512
    ctx0 = [0, 1500, 4096, 7680]
    q, kp, vp, table, total, _, _ = build_cache(B, H, d, page, 200, ctx0, chunk,
                                                torch.bfloat16, seed=7)
    dev = "cuda"
    o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ctx = torch.tensor(total, dtype=torch.int32)
    scale = 1 / math.sqrt(d)
    fa.fa_fwd_paged(q.to(dev), kp, vp, table.to(dev), ctx.to(dev), o, lse, scale,
                    fa.FA_MASK_CAUSAL)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention_paged(q, kp.cpu(), vp.cpu(), table, ctx, scale,
                                          oracle.MASK_CAUSAL)
    compare(o, lse, ref_o, ref_l, "paged long")


def test_paged_prefill_reports_bad_page():
    B, H, d, page, chunk = 2, 2, 64, 64, 64
    q, kp, vp, table, total, _, _ = build_cache(B, H, d, page, 20, [100, 10], chunk,
                                                torch.float16, seed=9)
    bad = table.clone()
    bad[0, 1] = 20  # out of range
    dev = "cuda"
    o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    fa.fa_fwd_paged(q.to(dev), kp, vp, bad.to(dev), torch.tensor(total, dtype=torch.int32,
                    device=dev), o, None, 0.125)
    assert fa.fa_get_device_status() == fa.FA_ERR_BAD_PAGE
    assert fa.fa_get_device_status() == fa.FA_OK


@pytest.mark.parametrize("mode,w,g,page,d,dt", [
    (fa.FA_MASK_CAUSAL, 0, 0, 256, 128, torch.bfloat16),
    (fa.FA_MASK_CAUSAL_WINDOW, 300, 7, 256, 128, torch.bfloat16),
    (fa.FA_MASK_CAUSAL, 0, 0, 64, 64, torch.float16)])
def test_host_lengths_plan_gives_the_same_output(mode, w, g, page, d, dt):
    """fa_fwd_paged_host_lens only changes which CTA runs which item: with the right host
    lengths, with wrong ones and with none, every output bit and LSE bit is the same (256-
    and 64-token pages, the latter read as 64-key tiles)."""
    B, H, chunk = 6, 4, 300
    ctx0 = [5000, 0, 1200, 3100, 77, 2600]
    q, kp, vp, table, total, _, _ = build_cache(B, H, d, page, (160 * 256) // page, ctx0, chunk,
                                                dt, seed=7)
    qd, tab = q.cuda(), table.cuda()
    ctx = torch.tensor(total, dtype=torch.int32, device="cuda")
    scale = 1 / math.sqrt(d)
    outs = []
    for host in (None, torch.tensor(total, dtype=torch.int32),
                 torch.tensor([1, 9000, 0, -5, 4000, 300], dtype=torch.int32)):
        o = torch.empty_like(qd)
        lse = torch.empty(qd.shape[:3], dtype=torch.float32, device="cuda")
        fa.fa_fwd_paged(qd, kp, vp, tab, ctx, o, lse, scale, mode, w, g, ctx_lens_host=host)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), outs[0][1].view(torch.int32))
    with pytest.raises(ValueError):
        fa.fa_fwd_paged(qd, kp, vp, tab, ctx, outs[0][0], None, scale,
                        ctx_lens_host=torch.tensor(total[:3], dtype=torch.int32))
