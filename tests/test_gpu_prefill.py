"""GPU parity of fa_fwd (through the C ABI) against the FP64 CPU oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

from _util import compare, pick_rows, sample_rows

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}
MASKS = {"none": (fa.FA_MASK_NONE, 0, 0), "causal": (fa.FA_MASK_CAUSAL, 0, 0),
         "window": (fa.FA_MASK_CAUSAL_WINDOW, 50, 5), "band": (fa.FA_MASK_BAND, 40, 0),
         "prefix": (fa.FA_MASK_PREFIX_LM, 0, 70)}
MODES = {name: m[0] for name, m in MASKS.items()}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_attention_06_gb300 import build
    build.build()
    fa.lib()


def run_fwd(q, k, v, scale, mode, window=0, n_global=0, **ex):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    if ex:
        fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, mode, window, n_global, **ex)
    else:
        fa.fa_fwd(qd, kd, vd, o, lse, scale, mode, window, n_global)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o, lse


def test_tiny_noncausal_config():
    """B=1, H=2, Sq=Sk=128, d=64, fp16, N(0,1), scale 1/sqrt(d); O[1,2,128,64] plus LSE."""
    q, k, v = inputs.prefill_inputs(1, 2, 128, 128, 64, torch.float16, seed=0)
    o, lse = run_fwd(q, k, v, 1 / 8, fa.FA_MASK_NONE)
    assert o.shape == (1, 2, 128, 64)
    ref_o, ref_l = oracle.attention(q, k, v, 1 / 8, oracle.MASK_NONE)
    compare(o, lse, ref_o, ref_l, "tiny")


SHAPES = [(1, 1), (63, 63), (65, 65), (127, 129), (129, 127), (200, 333), (257, 64), (64, 257),
          (384, 384)]


@pytest.mark.parametrize("Sq,Sk", SHAPES)
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16"), (128, "f16")])
@pytest.mark.parametrize("mask", ["none", "causal", "window", "band", "prefix"])
@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
def test_small_shapes(Sq, Sk, d, dt, mask, bn, bm):
    q, k, v = inputs.prefill_inputs(2, 3, Sq, Sk, d, DT[dt], seed=Sq * 1000 + Sk)
    mode, w, g = MASKS[mask]
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, mode, w, g, block_n=bn, block_m=bm)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g)
    compare(o, lse, ref_o, ref_l, f"{Sq}x{Sk} d{d} {dt} {mask} bn{bn} bm{bm}")


@pytest.mark.parametrize("mask,w,g", [("causal", 0, 0), ("window", 200, 70), ("window", 1, 0),
                                      ("window", 129, 300), ("none", 0, 0), ("band", 0, 0),
                                      ("band", 150, 0), ("prefix", 0, 0), ("prefix", 0, 300)])
@pytest.mark.parametrize("Sq,Sk,bn", [(1000, 1000, 128), (700, 1100, 64), (1100, 700, 128)])
@pytest.mark.parametrize("bm", [64, 128, 256])
def test_tile_trace_is_bit_exact(mask, w, g, Sq, Sk, bn, bm):
    """The tiles the kernel visits, and the class it gives each, equal the oracle's
    brute-force tile classification; no tile is visited twice. The trace has one row per
    tensor-core tile of queries: 128 rows, 64 for 64-row items."""
    mode = MODES[mask]
    B, H, d = 1, 2, 64
    q, k, v = inputs.prefill_inputs(B, H, Sq, Sk, d, torch.float16, seed=3)
    BM = 64 if bm == 64 else fa.fa_fwd_block_m()
    nmb, nnb = -(-Sq // BM), -(-Sk // bn)
    trace = torch.zeros(B * H * nmb * nnb, dtype=torch.int32, device="cuda")
    o, lse = run_fwd(q, k, v, 0.125, mode, w, g, block_n=bn, block_m=bm, trace=trace)
    got = trace.cpu().numpy().reshape(B * H, nmb, nnb)
    want = np.zeros((nmb, nnb), dtype=np.int32)
    for mb in range(nmb):
        for nb in range(nnb):
            c = oracle.tile_class(mb, nb, BM, bn, Sq, Sk, mode, w, g)
            want[mb, nb] = 0 if c == oracle.TILE_EMPTY else 16 + c
    for bh in range(B * H):
        assert np.array_equal(got[bh], want), f"bh {bh}"
    ref_o, ref_l = oracle.attention(q, k, v, 0.125, mode, w, g)
    compare(o, lse, ref_o, ref_l, "trace case")


def test_guard_regions_untouched_and_outputs_finite():
    """Inputs and outputs live inside NaN-filled buffers; the call must read no NaN
    (outputs finite) and write nothing outside o and lse."""
    B, H, S, d = 2, 2, 300, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=5)
    G = 4096
    dev = "cuda"

    def guarded(t):
        buf = torch.full((t.numel() + 2 * G,), float("nan"), dtype=t.dtype, device=dev)
        buf[G:G + t.numel()] = t.reshape(-1).to(dev)
        return buf, buf[G:G + t.numel()].view(t.shape)

    (bq, qd), (bk, kd), (bv, vd) = guarded(q), guarded(k), guarded(v)
    bo = torch.full((q.numel() + 2 * G,), float("nan"), dtype=q.dtype, device=dev)
    od = bo[G:G + q.numel()].view(q.shape)
    bl = torch.full((B * H * S + 2 * G,), float("nan"), dtype=torch.float32, device=dev)
    ld = bl[G:G + B * H * S].view(B, H, S)
    for mode in (fa.FA_MASK_NONE, fa.FA_MASK_CAUSAL, fa.FA_MASK_CAUSAL_WINDOW, fa.FA_MASK_BAND,
                 fa.FA_MASK_PREFIX_LM):
        fa.fa_fwd(qd, kd, vd, od, ld, 1 / math.sqrt(d), mode, 77, 3)
        torch.cuda.synchronize()
        assert torch.isfinite(od.float()).all() and torch.isfinite(ld).all()
        for buf in (bo, bl):
            assert torch.isnan(buf[:G].float()).all() and torch.isnan(buf[-G:].float()).all()
        ref_o, ref_l = oracle.attention(q, k, v, 1 / math.sqrt(d), mode, 77, 3)
        compare(od, ld, ref_o, ref_l, f"guarded mode {mode}")


def test_empty_and_fully_masked():
    # Sk = 0: every row sees nothing
    q, k, v = inputs.prefill_inputs(1, 2, 70, 0, 64, torch.float16, seed=7)
    o, lse = run_fwd(q, k.reshape(1, 2, 0, 64), v.reshape(1, 2, 0, 64), 0.125, fa.FA_MASK_NONE)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    # Sq > Sk under a causal mask: the first Sq-Sk rows see nothing
    q, k, v = inputs.prefill_inputs(1, 2, 300, 100, 64, torch.float16, seed=8)
    o, lse = run_fwd(q, k, v, 0.125, fa.FA_MASK_CAUSAL)
    ref_o, ref_l = oracle.attention(q, k, v, 0.125, oracle.MASK_CAUSAL)
    compare(o, lse, ref_o, ref_l, "Sq>Sk causal")
    # Sq = 0: nothing to do, nothing written
    q = torch.empty(1, 2, 0, 64, dtype=torch.float16)
    k = torch.randn(1, 2, 5, 64).half()
    o, lse = run_fwd(q, k, k, 0.125, fa.FA_MASK_CAUSAL)
    assert o.numel() == 0


def test_schedule_does_not_change_results():
    """Every work item is computed the same way whatever CTA runs it: outputs are
    bit-identical for any persistent grid size and head grouping."""
    q, k, v = inputs.prefill_inputs(2, 5, 700, 700, 128, torch.bfloat16, seed=9)
    for bm in (64, 128, 256):
        o0, l0 = run_fwd(q, k, v, 0.088, fa.FA_MASK_CAUSAL, block_m=bm)
        for ctas, hg in [(1, 1), (7, 3), (37, 0), (1000, 10)]:
            o1, l1 = run_fwd(q, k, v, 0.088, fa.FA_MASK_CAUSAL, num_ctas=ctas, group_heads=hg,
                             block_m=bm)
            assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_causal_2k_fp16_full():
    """B=4, H=32, Sq=Sk=2048, d=128, fp16, causal, N(0,1)*0.5, scale 1/sqrt(128): every row."""
    q, k, v = inputs.prefill_inputs(4, 32, 2048, 2048, 128, torch.float16, factor=0.5, seed=0)
    scale = 1 / math.sqrt(128)
    o, lse = run_fwd(q, k, v, scale, fa.FA_MASK_CAUSAL)
    ref_o, ref_l = oracle.attention(q, k, v, scale, oracle.MASK_CAUSAL)
    compare(o, lse, ref_o, ref_l, "causal 2k")


@pytest.mark.parametrize("mode,w,g", [(fa.FA_MASK_CAUSAL, 0, 0), (fa.FA_MASK_NONE, 0, 0),
                                      (fa.FA_MASK_BAND, 512, 0), (fa.FA_MASK_PREFIX_LM, 0, 1024)])
def test_long_4k_bf16_sampled(mode, w, g):
    """B=4, H=32, Sq=Sk=4096, d=128, bf16, N(0,1): causal, non-causal and the bench's band
    (±512) and prefix-LM (1024-key prefix) configurations, each with its default kernel; the
    oracle checks the first and last query block of every head and 256 random rows."""
    B, H, S, d = 4, 32, 4096, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=0)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, mode, w, g)
    rows = sample_rows(B, H, S, fa.fa_fwd_block_m(), n_random=256, seed=1)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g, rows=rows)
    compare(pick_rows(o, rows, S), pick_rows(lse, rows, S), ref_o, ref_l, f"4k mode {mode}")


def test_sliding_window_32k_sampled():
    """B=1, H=32, S=32768, d=128, bf16, causal window 2048 + 64 global keys; sampled rows
    include the window and global-token edges."""
    B, H, S, d = 1, 32, 32768, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=0)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(q, k, v, scale, fa.FA_MASK_CAUSAL_WINDOW, 2048, 64)
    rows = sample_rows(B, H, S, fa.fa_fwd_block_m(), n_random=256, extra=range(2040, 2121),
                       seed=2)
    ref_o, ref_l = oracle.attention(q, k, v, scale, oracle.MASK_CAUSAL_WINDOW, 2048, 64,
                                    rows=rows)
    compare(pick_rows(o, rows, S), pick_rows(lse, rows, S), ref_o, ref_l, "window 32k")


# --------------------------------------------------------------------------- block-sparse
def _layout(H, Sq, Sk, seed, density=0.45):
    g = torch.Generator().manual_seed(seed)
    nq, nk = -(-Sq // fa.FA_LAYOUT_BLOCK), -(-Sk // fa.FA_LAYOUT_BLOCK)
    lay = (torch.rand(H, nq, nk, generator=g) < density).to(torch.uint8)
    lay[0, 0, :] = 0  # one query block of head 0 sees nothing
    return lay


def run_sparse(q, k, v, scale, lay, **ex):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, fa.FA_MASK_BLOCK_SPARSE,
                 block_layout=lay.to(dev), **ex)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o, lse


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (127, 129), (200, 333), (384, 384), (520, 257)])
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16")])
@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
def test_block_sparse_small(Sq, Sk, d, dt, bn, bm):
    q, k, v = inputs.prefill_inputs(2, 3, Sq, Sk, d, DT[dt], seed=Sq + 7 * Sk)
    lay = _layout(3, Sq, Sk, seed=Sq * Sk)
    scale = 1 / math.sqrt(d)
    o, lse = run_sparse(q, k, v, scale, lay, block_n=bn, block_m=bm)
    ref_o, ref_l = oracle.attention_layout(q, k, v, scale, lay.numpy())
    compare(o, lse, ref_o, ref_l, f"block-sparse {Sq}x{Sk} d{d} bn{bn} bm{bm}")


@pytest.mark.parametrize("bn", [64, 128])
@pytest.mark.parametrize("bm", [64, 128, 256])
def test_block_sparse_trace_is_bit_exact(bn, bm):
    """Tiles the kernel visits, with their classes, equal the oracle's brute-force
    classification under the layout; a 256-row item visits only its tiles' blocks."""
    B, H, Sq, Sk, d = 1, 2, 900, 1100, 64
    q, k, v = inputs.prefill_inputs(B, H, Sq, Sk, d, torch.float16, seed=5)
    lay = _layout(H, Sq, Sk, seed=11, density=0.35)
    BM = 64 if bm == 64 else fa.fa_fwd_block_m()
    nmb, nnb = -(-Sq // BM), -(-Sk // bn)
    trace = torch.zeros(B * H * nmb * nnb, dtype=torch.int32, device="cuda")
    o, lse = run_sparse(q, k, v, 0.125, lay, block_n=bn, block_m=bm, trace=trace)
    got = trace.cpu().numpy().reshape(B * H, nmb, nnb)
    for h in range(H):
        want = np.zeros((nmb, nnb), dtype=np.int32)
        for mb in range(nmb):
            for nb in range(nnb):
                c = oracle.tile_class_layout(h, mb, nb, BM, bn, Sq, Sk, lay.numpy())
                want[mb, nb] = 0 if c == oracle.TILE_EMPTY else 16 + c
        assert np.array_equal(got[h], want), f"head {h}"
    ref_o, ref_l = oracle.attention_layout(q, k, v, 0.125, lay.numpy())
    compare(o, lse, ref_o, ref_l, "block-sparse trace case")


@pytest.mark.parametrize("bm", [64, 128, 256])
def test_block_sparse_host_layout_plan_gives_the_same_output(bm):
    """block_layout_host only changes which CTA runs which item: with the right host copy,
    a wrong one and none, every output bit and LSE bit is the same."""
    B, H, Sq, Sk, d = 2, 3, 1100, 900, 128
    q, k, v = inputs.prefill_inputs(B, H, Sq, Sk, d, torch.bfloat16, seed=41)
    lay = _layout(H, Sq, Sk, seed=5, density=0.3)
    lay[1, 2, :] = 1  # one query block of head 1 sees every key block
    wrong = torch.flip(lay, dims=[1]).contiguous()
    outs = [run_sparse(q, k, v, 0.1, lay, block_m=bm, **ex)
            for ex in ({}, {"block_layout_host": lay}, {"block_layout_host": wrong})]
    for o, lse in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0][0].view(torch.int16))
        assert torch.equal(lse.view(torch.int32), outs[0][1].view(torch.int32))
    with pytest.raises(ValueError):
        run_sparse(q, k, v, 0.1, lay, block_layout_host=lay[:, :-1].contiguous())


def test_block_sparse_4k_bigbird_sampled():
    """The bench's block-sparse configuration: B=4, H=32, S=4096, d=128, bf16 with the
    seeded BigBird-shaped layout; sampled rows of every head."""
    B, H, S, d = 4, 32, 4096, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=0)
    lay = inputs.block_layout(H, S, S)
    scale = 1 / math.sqrt(d)
    o, lse = run_sparse(q, k, v, scale, lay, block_layout_host=lay)
    rows = sample_rows(B, H, S, fa.fa_fwd_block_m(), n_random=128, seed=3)
    ref_o, ref_l = oracle.attention_layout(q, k, v, scale, lay.numpy(), rows=rows)
    compare(pick_rows(o, rows, S), pick_rows(lse, rows, S), ref_o, ref_l, "block-sparse 4k")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_output_only_16_byte_aligned(dt):
    """The API asks O to be 16-byte aligned only; the epilogue's 32-byte stores must fall back
    when O sits 16 bytes past a 32-byte boundary."""
    B, H, S, d = 1, 3, 300, 128
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda")
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, dtype, seed=31)
    step = 16 // torch.empty(0, dtype=dtype).element_size()  # elements in 16 bytes
    buf = torch.full((q.numel() + 64,), float("nan"), dtype=dtype, device=dev)
    assert buf.data_ptr() % 32 == 0
    o = buf[step:step + q.numel()].view(q.shape)
    assert o.data_ptr() % 32 == 16
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    for mode in (fa.FA_MASK_CAUSAL, fa.FA_MASK_NONE):
        fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), o, lse, scale, mode)
        torch.cuda.synchronize()
        assert fa.fa_get_device_status() == fa.FA_OK
        ref_o, ref_l = oracle.attention(q, k, v, scale, mode)
        if dt == "f32":
            compare(o, lse, ref_o, ref_l, f"16-byte aligned O, mode {mode}", o_max=1e-3, o_mean=1e-4)
        else:
            compare(o, lse, ref_o, ref_l, f"16-byte aligned O, mode {mode}")
        assert torch.isnan(buf[:step].float()).all() and torch.isnan(buf[step + q.numel():].float()).all()
