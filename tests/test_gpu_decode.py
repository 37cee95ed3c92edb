"""GPU parity of fa_decode_paged (through the C ABI) against the FP64 CPU oracle."""
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


def run_decode(di, scale, pages_per_split=0, traces=False):
    dev = "cuda"
    q, kp, vp = di.q.to(dev), di.k_pages.to(dev), di.v_pages.to(dev)
    bt, cl = di.block_table.to(dev), di.ctx_lens.to(dev)
    B, H, d = q.shape
    mp = bt.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, d, mp, di.page_size), dtype=torch.uint8,
                     device=dev)
    tp = ts = None
    if traces:
        pps = pages_per_split or fa.fa_decode_default_pages_per_split(B, H, mp)
        nsplit = -(-mp // pps)
        tp = torch.full((B * H * mp,), -1, dtype=torch.int32, device=dev)
        ts = torch.full((B * H * nsplit * 2,), -7, dtype=torch.int32, device=dev)
    fa.fa_decode_paged_ex(q, kp, vp, bt, cl, o, lse, scale, ws, pages_per_split, tp, ts)
    torch.cuda.synchronize()
    return o, lse, tp, ts


def test_paged_decode_config_full():
    """B=32, H=32, d=128, fp16, ctx ~ U[1,8192], 256-token pages scattered over a pool
    of 1200 by a random permutation table; every (sequence, head)."""
    di = inputs.decode_inputs(B=32, H=32, d=128, page_size=256, num_pages=1200, max_ctx=8192,
                              dtype=torch.float16, seed=0)
    scale = 1 / math.sqrt(128)
    o, lse, _, _ = run_decode(di, scale)
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                       scale)
    compare(o, lse, ref_o, ref_l, "paged decode config")


@pytest.mark.parametrize("page,d,dt", [(16, 64, torch.float16), (64, 128, torch.bfloat16),
                                       (256, 128, torch.float16), (32, 128, torch.bfloat16)])
@pytest.mark.parametrize("pps", [0, 1, 3])
def test_small_paged_cases(page, d, dt, pps):
    max_pages = 12
    ctx = [0, 1, page - 1, page, page + 1, 5 * page + 3, max_pages * page, 2]
    di = inputs.decode_inputs(B=len(ctx), H=3, d=d, page_size=page, num_pages=100,
                              max_ctx=max_pages * page, dtype=dt, seed=page + d, ctx_lens=ctx)
    scale = 1 / math.sqrt(d)
    o, lse, _, _ = run_decode(di, scale, pages_per_split=pps)
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                       scale)
    compare(o, lse, ref_o, ref_l, f"page {page} d {d} pps {pps}")
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))   # ctx = 0


@pytest.mark.parametrize("pps", [1, 2, 5])
def test_page_and_split_traces_are_bit_exact(pps):
    """The physical page read for every logical page equals the block-table lookup,
    and every split covers exactly the oracle planner's token range."""
    page, mp = 32, 10
    di = inputs.decode_inputs(B=6, H=2, d=64, page_size=page, num_pages=70, max_ctx=page * mp,
                              dtype=torch.float16, seed=11)
    o, lse, tp, ts = run_decode(di, 0.125, pages_per_split=pps, traces=True)
    B, H = 6, 2
    tp = tp.cpu().numpy().reshape(B, H, mp)
    nsplit = -(-mp // pps)
    ts = ts.cpu().numpy().reshape(B, H, nsplit, 2)
    for b in range(B):
        c = int(di.ctx_lens[b])
        npg = -(-c // page)
        for h in range(H):
            want = np.full(mp, -1)
            want[:npg] = di.block_table[b, :npg].numpy()
            assert np.array_equal(tp[b, h], want)
            for s in range(nsplit):
                assert tuple(ts[b, h, s]) == oracle.decode_split_tokens(c, page, pps, s)
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                       0.125)
    compare(o, lse, ref_o, ref_l, "trace case")


def test_out_of_range_page_is_reported_and_skipped():
    page = 16
    di = inputs.decode_inputs(B=3, H=2, d=64, page_size=page, num_pages=20, max_ctx=4 * page,
                              dtype=torch.float16, seed=13, ctx_lens=[40, 33, 17])
    bt = di.block_table.clone()
    bt[1, 1] = 20  # sequence 1, logical page 1: out of range
    good = inputs.DecodeInputs(di.q, di.k_pages, di.v_pages, bt, di.ctx_lens, page)
    o, lse, _, _ = run_decode(good, 0.125)
    assert fa.fa_get_device_status() == fa.FA_ERR_BAD_PAGE
    assert fa.fa_get_device_status() == fa.FA_OK  # reading clears it
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                       0.125, bh_list=[0, 1, 4, 5])
    compare(o[[0, 2]].reshape(-1, 64), lse[[0, 2]].reshape(-1), ref_o, ref_l, "good sequences")
    # the sequence with the bad page attends over the tokens of its valid pages only
    keep = [t for t in range(33) if t // page != 1]
    qd = di.q[1][None, :, None, :]
    ks = torch.stack([di.k_pages[int(di.block_table[1, t // page]), :, t % page] for t in keep], 1)
    vs = torch.stack([di.v_pages[int(di.block_table[1, t // page]), :, t % page] for t in keep], 1)
    r_o, r_l = oracle.attention(qd, ks[None], vs[None], 0.125)
    compare(o[1], lse[1], r_o[0, :, 0], r_l[0, :, 0], "sequence with a bad page")


def test_split_choice_does_not_matter():
    di = inputs.decode_inputs(B=8, H=4, d=128, page_size=64, num_pages=200, max_ctx=64 * 20,
                              dtype=torch.bfloat16, seed=17)
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                       0.09)
    for pps in (1, 2, 4, 7, 20):
        o, lse, _, _ = run_decode(di, 0.09, pages_per_split=pps)
        compare(o, lse, ref_o, ref_l, f"pps {pps}")


@pytest.mark.parametrize("d,dt", [(128, torch.float16), (64, torch.bfloat16)])
def test_pools_only_16_byte_aligned(d, dt):
    """The split kernel reads 32 bytes of K and V per lane when both pools are 32-byte
    aligned and 16 bytes per lane otherwise: the same pages read through pools that start
    16 bytes past a 32-byte boundary take the second path and must give the same results
    (and the oracle's)."""
    di = inputs.decode_inputs(B=6, H=4, d=d, page_size=64, num_pages=60, max_ctx=64 * 9,
                              dtype=dt, seed=23)
    scale = 1 / math.sqrt(d)
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table,
                                       di.ctx_lens, scale)
    dev = "cuda"
    shifted = []
    for pool in (di.k_pages, di.v_pages):
        flat = torch.empty(pool.numel() + 8, dtype=dt, device=dev)  # 8 elements = 16 bytes
        view = flat[8:].view(pool.shape)
        view.copy_(pool.to(dev))
        assert view.data_ptr() % 32 == 16
        shifted.append(view)
    q, bt, cl = di.q.to(dev), di.block_table.to(dev), di.ctx_lens.to(dev)
    B, H, _ = q.shape
    mp = bt.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty(B, H, dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, d, mp, di.page_size), dtype=torch.uint8,
                     device=dev)
    fa.fa_decode_paged_ex(q, shifted[0], shifted[1], bt, cl, o, lse, scale, ws)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    compare(o, lse, ref_o, ref_l, "16-byte aligned pools")
    o2, lse2, _, _ = run_decode(di, scale)  # 32-byte aligned pools
    compare(o2, lse2, ref_o, ref_l, "32-byte aligned pools")
