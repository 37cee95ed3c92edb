"""GPU parity of the FP32-input forward (fa_fwd_ex with FA_F32, through the C ABI)
against the FP64 oracle: max |O - O_ref| <= 1e-3, mean <= 1e-4, |LSE - LSE_ref| <= 1e-3,
-inf LSE patterns equal. The kernel forms every product from bf16 high and low parts
(hi*hi + hi*lo + lo*hi); the resolution test uses inputs on which the high parts alone
miss the bound (shown on the CPU in test_f32_split_host.py)."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

from _util import O_MAX_F32, O_MEAN_F32, compare, pick_rows, sample_rows

pytestmark = pytest.mark.gpu

MASKS = {"none": (fa.FA_MASK_NONE, 0, 0), "causal": (fa.FA_MASK_CAUSAL, 0, 0),
         "window": (fa.FA_MASK_CAUSAL_WINDOW, 50, 5), "band": (fa.FA_MASK_BAND, 40, 0),
         "prefix": (fa.FA_MASK_PREFIX_LM, 0, 70)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_attention_06_gb300 import build
    build.build()
    fa.lib()


def run_fwd32(q, k, v, scale, mode, window=0, n_global=0, **ex):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=dev)
    fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, mode, window, n_global, **ex)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o, lse


def check32(o, lse, ref_o, ref_l, what):
    assert o.dtype == torch.float32
    return compare(o, lse, ref_o, ref_l, what, o_max=O_MAX_F32, o_mean=O_MEAN_F32)


SHAPES = [(1, 1), (63, 63), (65, 65), (127, 129), (129, 127), (200, 333), (257, 64), (64, 257),
          (384, 384)]


@pytest.mark.parametrize("Sq,Sk", SHAPES)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask", list(MASKS))
def test_f32_small_shapes(Sq, Sk, d, mask):
    q, k, v = inputs.prefill_inputs(2, 3, Sq, Sk, d, torch.float32, seed=Sq * 1000 + Sk)
    mode, w, g = MASKS[mask]
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd32(q, k, v, scale, mode, w, g)
    ref_o, ref_l = oracle.attention(q, k, v, scale, mode, w, g)
    check32(o, lse, ref_o, ref_l, f"{Sq}x{Sk} d{d} {mask}")


@pytest.mark.parametrize("mask", ["causal", "none", "prefix"])
def test_f32_resolution(mask):
    """Logits up to ~+-10 and V near 1 with small deviations: bf16 rounding of Q, K, V or
    P alone moves O by more than 1e-3 here, so only the products of both parts pass."""
    q, k, v = inputs.f32_resolution_inputs(2, 2, 300, 300, 64, seed=11)
    mode, w, g = MASKS[mask]
    o, lse = run_fwd32(q, k, v, 0.125, mode, w, g)
    ref_o, ref_l = oracle.attention(q, k, v, 0.125, mode, w, g)
    check32(o, lse, ref_o, ref_l, f"resolution {mask}")


def test_f32_block_sparse():
    B, H, S, d = 1, 2, 700, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.float32, seed=21)
    lay = inputs.block_layout(H, S, S, seed=4)
    o, lse = run_fwd32(q, k, v, 0.088, fa.FA_MASK_BLOCK_SPARSE, block_layout=lay.cuda())
    ref_o, ref_l = oracle.attention_layout(q, k, v, 0.088, lay.numpy())
    check32(o, lse, ref_o, ref_l, "block-sparse f32")


def test_f32_tile_trace_matches_oracle_classes():
    """The FP32 kernel visits exactly the tiles of the 16-bit kernels (64-key blocks)."""
    B, H, Sq, Sk, bn = 1, 2, 1000, 1000, 64
    q, k, v = inputs.prefill_inputs(B, H, Sq, Sk, 64, torch.float32, seed=3)
    BM = fa.fa_fwd_block_m()
    nmb, nnb = -(-Sq // BM), -(-Sk // bn)
    for mode, w, g in [MASKS["causal"], (fa.FA_MASK_CAUSAL_WINDOW, 200, 70), MASKS["band"]]:
        trace = torch.zeros(B * H * nmb * nnb, dtype=torch.int32, device="cuda")
        run_fwd32(q, k, v, 0.125, mode, w, g, trace=trace)
        got = trace.cpu().numpy().reshape(B * H, nmb, nnb)
        want = np.zeros((nmb, nnb), dtype=np.int32)
        for mb in range(nmb):
            for nb in range(nnb):
                c = oracle.tile_class(mb, nb, BM, bn, Sq, Sk, mode, w, g)
                want[mb, nb] = 0 if c == oracle.TILE_EMPTY else 16 + c
        for bh in range(B * H):
            assert np.array_equal(got[bh], want), f"mode {mode} bh {bh}"


def test_f32_empty_and_rows_without_keys():
    # Sq > Sk under a causal mask: the first Sq - Sk rows see no key (O = 0, LSE = -inf)
    q, k, v = inputs.prefill_inputs(1, 2, 300, 100, 128, torch.float32, seed=4)
    o, lse = run_fwd32(q, k, v, 0.088, fa.FA_MASK_CAUSAL)
    assert torch.all(o[:, :, :200] == 0) and torch.all(torch.isneginf(lse[:, :, :200]))
    ref_o, ref_l = oracle.attention(q, k, v, 0.088, oracle.MASK_CAUSAL)
    check32(o, lse, ref_o, ref_l, "Sq > Sk")
    # Sk = 0: every row sees no key
    q = torch.randn(1, 2, 70, 64)
    kv = torch.empty(1, 2, 0, 64)
    o, lse = run_fwd32(q, kv, kv, 0.125, fa.FA_MASK_NONE)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    # Sq = 0: nothing to do
    o, lse = run_fwd32(torch.empty(1, 2, 0, 64), q, q, 0.125, fa.FA_MASK_CAUSAL)
    assert o.numel() == 0


def test_f32_matches_plain_fa_fwd_binding():
    """fa_fwd on float32 tensors takes the same path (the binding supplies the workspace)
    and gives bit-identical results for any grid size."""
    q, k, v = inputs.prefill_inputs(2, 3, 500, 500, 128, torch.float32, seed=8)
    dev = torch.device("cuda")
    o1, l1 = run_fwd32(q, k, v, 0.088, fa.FA_MASK_CAUSAL)
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), o2, l2, 0.088, fa.FA_MASK_CAUSAL)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o3, l3 = run_fwd32(q, k, v, 0.088, fa.FA_MASK_CAUSAL, num_ctas=7, group_heads=2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_f32_causal_4k_sampled():
    """B=4, H=32, Sq=Sk=4096, d=128, FP32, causal, N(0,1): the launch the bench times; the
    oracle checks the first and last query block of every head and 128 random rows."""
    B, H, S, d = 4, 32, 4096, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.float32, seed=0)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd32(q, k, v, scale, fa.FA_MASK_CAUSAL)
    rows = sample_rows(B, H, S, fa.fa_fwd_block_m(), n_random=128, seed=1)
    ref_o, ref_l = oracle.attention(q, k, v, scale, oracle.MASK_CAUSAL, rows=rows)
    check32(pick_rows(o, rows, S), pick_rows(lse, rows, S), ref_o, ref_l, "4k f32 causal")
