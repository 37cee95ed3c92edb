"""The lazy rescale of the prefill softmax, driven hard and counted.

The per-block (m, l, O) recurrence (zwxr.cn article on ops-transformer, section 3.1;
the running max and sum of the ops-transformer overview's tiled loop, section 二.1)
multiplies the partial output and sum by exp(m_old - m_new) when a key block raises a
row's running maximum. The kernels take that correction lazily, only when the maximum
has risen by more than 8 (log2 units) since it was last taken. With N(0,1) inputs the
branch almost never runs, so these tests use inputs whose scores climb along the key
axis (every later key tile lifts every row's maximum by about 12 log2 units) or are
simply wide (q, k ~ N(0,1) * 4), and a falling ramp as the control.

Each case is checked three ways, through the C ABI:
  * O and LSE against the FP64 oracle, element by element, at the usual tolerances;
  * the kernel's count of rescaled rows (fa_fwd_params.rescale_count) per 128-query
    tile against the oracle's count of the same decisions (oracle.rescale_events);
    the two may differ only where the oracle finds a decision within 1e-3 of the
    threshold, which FP32 arithmetic may take the other way;
  * the count is non-zero (both tiles of a 256-row item, when there are two), so the
    branch was reached; the falling ramp counts zero.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

from _util import O_MAX_F32, O_MEAN_F32, compare, pick_rows, sample_rows

pytestmark = pytest.mark.gpu

TAU = 8 * math.log(2)  # the kernels' threshold (8 log2 units) in natural-log units
RISE_LOG2 = 12.0        # score rise per key tile of the climbing inputs, log2 units
DT = {"f16": torch.float16, "bf16": torch.bfloat16}
MASKS = {"none": (fa.FA_MASK_NONE, 0, 0), "causal": (fa.FA_MASK_CAUSAL, 0, 0),
         "window": (fa.FA_MASK_CAUSAL_WINDOW, 300, 5), "band": (fa.FA_MASK_BAND, 150, 0),
         "prefix": (fa.FA_MASK_PREFIX_LM, 0, 70)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_attention_06_gb300 import build
    build.build()
    fa.lib()


def climbing(B, H, Sq, Sk, d, dtype, kind, scale, bn, seed):
    """'up': scores rise by RISE_LOG2 per bn-key tile; 'down': they fall as much; 'wide':
    q, k ~ N(0,1) * 4 and v ~ N(0,1) / 2. Such wide scores put nearly all of a row's
    weight on one key, so O is close to a single V row; with v ~ N(0,1) that row can
    exceed 4, where one bf16 rounding of O alone may cost 2^-6, and P's own rounding
    (2^-9 relative) comes on top. Halving V keeps that sum inside the 2e-2 bound the
    16-bit tests use, which still leaves any wrong rescale visible."""
    if kind == "wide":
        return inputs.climbing_inputs(B, H, Sq, Sk, d, dtype, step=0.0, wide=4.0, v_scale=0.5,
                                      seed=seed)
    step = RISE_LOG2 * math.log(2) / (scale * bn)  # raw q.k rise per key
    return inputs.climbing_inputs(B, H, Sq, Sk, d, dtype, step=step if kind == "up" else -step,
                                  seed=seed)


def run_counted(q, k, v, scale, mode, w, g, layout=None, **ex):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    B, H, Sq, _ = q.shape
    cnt = torch.zeros(B * H, -(-Sq // 128), dtype=torch.int32, device=dev)
    fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, mode, w, g, rescale_count=cnt,
                 block_layout=None if layout is None else layout.to(dev), **ex)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o, lse, cnt.cpu().numpy().astype(np.int64)


def check_counts(got, q, k, scale, bn, mode, w, g, what, layout=None, expect_some=True):
    """The kernel's per-tile counts equal the oracle's, up to the decisions the oracle
    finds within 1e-3 of the threshold (each may also move the reference for the rest of
    its row, so it may change the row's count by up to the row's number of key tiles)."""
    want, near = oracle.rescale_events(q, k, scale, bn, TAU, mode, w, g,
                                       layout=None if layout is None else layout.numpy())
    slack = near * (-(-k.shape[2] // bn))
    bad = np.abs(got - want) > slack
    assert not bad.any(), (f"{what}: rescale counts differ at {np.argwhere(bad)[:5].tolist()}: "
                           f"got {got[bad][:5].tolist()} want {want[bad][:5].tolist()}")
    if expect_some:
        assert got.sum() > 0, f"{what}: no row was rescaled"
    return want


SHAPES = [(384, 384), (257, 700)]


@pytest.mark.parametrize("Sq,Sk", SHAPES)
@pytest.mark.parametrize("d,dt", [(64, "f16"), (64, "bf16"), (128, "f16"), (128, "bf16")])
@pytest.mark.parametrize("mask", list(MASKS))
@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
@pytest.mark.parametrize("kind", ["up", "wide"])
def test_rescale_small(Sq, Sk, d, dt, mask, bn, bm, kind):
    scale = 1 / math.sqrt(d)
    q, k, v = climbing(2, 3, Sq, Sk, d, DT[dt], kind, scale, bn, seed=Sq + Sk + d)
    mode, w, g = MASKS[mask]
    what = f"{kind} {Sq}x{Sk} d{d} {dt} {mask} bn{bn} bm{bm}"
    o, lse, cnt = run_counted(q, k, v, scale, mode, w, g, block_n=bn, block_m=bm)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g)
    compare(o, lse, ref_o, ref_l, what)
    check_counts(cnt, q, k, scale, bn, mode, w, g, what)
    if kind == "up" and bm == 256:
        # both softmax warpgroups of the 256-row kernel (tiles A and B of an item) rescale
        assert cnt[:, 0::2].sum() > 0 and cnt[:, 1::2].sum() > 0, what


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
@pytest.mark.parametrize("mask", ["none", "causal", "window"])
def test_falling_scores_never_rescale(bn, bm, mask):
    """Control: when the first visited key tile holds every row's maximum, nothing is
    rescaled, and the count says so."""
    d, S = 128, 640
    scale = 1 / math.sqrt(d)
    q, k, v = climbing(2, 3, S, S, d, torch.bfloat16, "down", scale, bn, seed=5)
    mode, w, g = MASKS[mask]
    o, lse, cnt = run_counted(q, k, v, scale, mode, w, g, block_n=bn, block_m=bm)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g)
    compare(o, lse, ref_o, ref_l, f"down {mask}")
    want = check_counts(cnt, q, k, scale, bn, mode, w, g, f"down {mask}", expect_some=False)
    assert want.sum() == 0 and cnt.sum() == 0


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
@pytest.mark.parametrize("kind", ["up", "wide"])
def test_rescale_block_sparse(bn, bm, kind):
    d, Sq, Sk = 128, 520, 640
    scale = 1 / math.sqrt(d)
    q, k, v = climbing(2, 3, Sq, Sk, d, torch.bfloat16, kind, scale, bn, seed=7)
    gen = torch.Generator().manual_seed(8)
    lay = (torch.rand(3, -(-Sq // 128), -(-Sk // 128), generator=gen) < 0.6).to(torch.uint8)
    what = f"block-sparse {kind} bn{bn} bm{bm}"
    o, lse, cnt = run_counted(q, k, v, scale, fa.FA_MASK_BLOCK_SPARSE, 0, 0, layout=lay,
                              block_n=bn, block_m=bm)
    ref_o, ref_l = oracle.attention_layout(q, k, v, scale, lay.numpy())
    compare(o, lse, ref_o, ref_l, what)
    check_counts(cnt, q, k, scale, bn, oracle.MASK_NONE, 0, 0, what, layout=lay)


@pytest.mark.parametrize("page", [64, 128])
@pytest.mark.parametrize("mask", ["causal", "window", "prefix"])
def test_rescale_paged_prefill(page, mask):
    """Chunked prefill through a block table (fa_fwd_paged) on climbing keys: the paged
    kernels run the same softmax on the same scores as the contiguous call, whose counts
    show the rescales taken; the paged outputs equal the contiguous ones bit for bit and
    the oracle within tolerance."""
    B, H, d, Sq, ctx = 2, 4, 128, 300, 900
    bn = 128 if page % 128 == 0 else 64
    scale = 1 / math.sqrt(d)
    q, k, v = climbing(B, H, Sq, ctx, d, torch.float16, "up", scale, bn, seed=11)
    mode, w, g = MASKS[mask]
    dev = "cuda"
    npg = -(-ctx // page)
    num_pages = B * npg + 5
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(12))
    table = perm[:B * npg].view(B, npg).to(torch.int32).to(dev)
    kp = torch.full((num_pages, H, page, d), float("nan"), dtype=torch.float16, device=dev)
    vp = torch.full_like(kp, float("nan"))
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    fa.fa_kv_append(k.to(dev), v.to(dev), kp, vp, table, zero)
    lens = torch.full((B,), ctx, dtype=torch.int32, device=dev)
    o = torch.empty(B, H, Sq, d, dtype=torch.float16, device=dev)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
    fa.fa_fwd_paged(q.to(dev), kp, vp, table, lens, o, lse, scale, mode, w, g)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    o_c, lse_c, cnt = run_counted(q, k, v, scale, mode, w, g, block_n=bn,
                                  block_m=fa.fa_fwd_default_block_m(mode))
    check_counts(cnt, q, k, scale, bn, mode, w, g, f"paged {mask} page {page}")
    assert torch.equal(o, o_c) and torch.equal(lse, lse_c)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g)
    compare(o, lse, ref_o, ref_l, f"paged {mask} page {page}")


def test_rescale_f32_inputs():
    """FP32 inputs (split bf16 products) on climbing keys, at the FP32 bounds."""
    d, S = 64, 500
    scale = 1 / math.sqrt(d)
    step = RISE_LOG2 * math.log(2) / (scale * 64)
    q, k, v = inputs.climbing_inputs(2, 2, S, S, d, torch.float32, step=step, seed=13)
    for mode in (fa.FA_MASK_CAUSAL, fa.FA_MASK_NONE):
        o, lse, cnt = run_counted(q, k, v, scale, mode, 0, 0)
        ref_o, ref_l = oracle.attention(q, k, v, scale, mode)
        compare(o, lse, ref_o, ref_l, f"f32 mode {mode}", o_max=O_MAX_F32, o_mean=O_MEAN_F32)
        check_counts(cnt, q, k, scale, 64, mode, 0, 0, f"f32 mode {mode}")


@pytest.mark.parametrize("bm", [64, 128, 256])
@pytest.mark.parametrize("mode", [fa.FA_MASK_CAUSAL, fa.FA_MASK_NONE])
def test_rescale_4k_sampled(bm, mode):
    """4k keys (32 key tiles per row, every one a rescale for most rows, while the previous
    tiles' P.V products are still being issued): sampled rows against the oracle, every
    count against the oracle's."""
    B, H, S, d, bn = 2, 8, 4096, 128, 128
    scale = 1 / math.sqrt(d)
    q, k, v = climbing(B, H, S, S, d, torch.bfloat16, "up", scale, bn, seed=21)
    o, lse, cnt = run_counted(q, k, v, scale, mode, 0, 0, block_m=bm)
    rows = sample_rows(B, H, S, 128, n_random=128, seed=22)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, rows=rows)
    what = f"4k mode {mode} bm{bm}"
    compare(pick_rows(o, rows, S), pick_rows(lse, rows, S), ref_o, ref_l, what)
    want = check_counts(cnt, q, k, scale, bn, mode, 0, 0, what)
    assert want.sum() > B * H * S * 4  # several rescales per row on average
