"""GPU parity of fa_bwd (through the C ABI) against the FP64 oracle's backward.

Tolerance: P and dS are rounded to the 16-bit input type before their MMAs (relative error
2^-9 for bf16, 2^-12 for fp16) and dq, dk, dv once more on output, with FP32 accumulation;
errors of the summed terms are independent, so the error relative to the tensor's scale
stays near 2^-8. Checked: max |err| <= 2e-2 * max |ref| and mean |err| <= 4e-3 * mean |ref|
for every gradient tensor; exact zeros where no tile contributes (a key no query sees, a
query that sees no key), and |err| <= 1e-5 where the definition's zero is a cancellation
(one visible key: dP - D = dO.V - dO.O with O = V)."""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import inputs

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16}
MASKS = {"none": (fa.FA_MASK_NONE, 0, 0), "causal": (fa.FA_MASK_CAUSAL, 0, 0),
         "window": (fa.FA_MASK_CAUSAL_WINDOW, 50, 5), "band": (fa.FA_MASK_BAND, 40, 0),
         "prefix": (fa.FA_MASK_PREFIX_LM, 0, 70)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from tiled_attention_06_gb300 import build
    build.build()
    fa.lib()


def fwd_bwd(q, k, v, dout, scale, mode, w, g):
    dev = torch.device("cuda")
    qd, kd, vd, gd = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    fa.fa_fwd(qd, kd, vd, o, lse, scale, mode, w, g)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    B, H, Sq, _ = q.shape
    ws = torch.empty(max(fa.fa_bwd_workspace_size(B, H, Sq), 16), dtype=torch.uint8, device=dev)
    fa.fa_bwd(qd, kd, vd, o, gd, lse, dq, dk, dv, ws, scale, mode, w, g)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return dq.float().cpu().numpy(), dk.float().cpu().numpy(), dv.float().cpu().numpy()


def compare_grad(got, ref, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    err = np.abs(got - ref)
    scale = np.abs(ref)
    if scale.max() == 0:  # zero by cancellation (dP - D): FP32 rounding of the two terms
        assert err.max() <= 1e-5, f"{what}: want ~0, max |got| {err.max():.3e}"
        return
    assert err.max() <= 2e-2 * scale.max(), f"{what}: max err {err.max():.3e} vs {scale.max():.3e}"
    assert err.mean() <= 4e-3 * scale.mean(), \
        f"{what}: mean err {err.mean():.3e} vs mean |ref| {scale.mean():.3e}"


def check(q, k, v, dout, scale, mask, what):
    mode, w, g = MASKS[mask]
    dq, dk, dv = fwd_bwd(q, k, v, dout, scale, mode, w, g)
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, scale, mode, w, g)
    compare_grad(dq, rq, what + " dq")
    compare_grad(dk, rk, what + " dk")
    compare_grad(dv, rv, what + " dv")


SHAPES = [(1, 1), (64, 64), (127, 129), (129, 127), (200, 333), (333, 200), (384, 384)]


@pytest.mark.parametrize("Sq,Sk", SHAPES)
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16")])
@pytest.mark.parametrize("mask", list(MASKS))
def test_backward_small_shapes(Sq, Sk, d, dt, mask):
    q, k, v = inputs.prefill_inputs(2, 2, Sq, Sk, d, DT[dt], seed=Sq * 10 + Sk)
    dout = inputs.prefill_inputs(2, 2, Sq, Sq, d, DT[dt], seed=Sq + 99)[0]
    check(q, k, v, dout, 1 / math.sqrt(d), mask, f"{Sq}x{Sk} d{d} {dt} {mask}")


def test_backward_empty_sides():
    q, k, v = inputs.prefill_inputs(1, 2, 0, 130, 64, torch.float16, seed=1)
    dout = torch.zeros(1, 2, 0, 64, dtype=torch.float16)
    dq, dk, dv = fwd_bwd(q, k, v, dout, 0.125, fa.FA_MASK_NONE, 0, 0)
    assert np.all(dk == 0) and np.all(dv == 0)  # no query: every key's gradients are 0
    q, k, v = inputs.prefill_inputs(1, 2, 70, 0, 64, torch.float16, seed=2)
    dout = inputs.prefill_inputs(1, 2, 70, 70, 64, torch.float16, seed=3)[0]
    dq, dk, dv = fwd_bwd(q, k, v, dout, 0.125, fa.FA_MASK_NONE, 0, 0)
    assert np.all(dq == 0)


def test_backward_rows_without_keys():
    """Sq > Sk under a causal mask: the first Sq - Sk queries see no key."""
    q, k, v = inputs.prefill_inputs(1, 2, 300, 100, 128, torch.bfloat16, seed=4)
    dout = inputs.prefill_inputs(1, 2, 300, 300, 128, torch.bfloat16, seed=5)[0]
    dq, _, _ = fwd_bwd(q, k, v, dout, 0.088, fa.FA_MASK_CAUSAL, 0, 0)
    assert np.all(dq[:, :, :200] == 0)
    check(q, k, v, dout, 0.088, "causal", "Sq > Sk")


def test_backward_causal_2k_full():
    """B=1, H=2, S=2048, d=128, bf16, causal: every gradient element against the oracle."""
    q, k, v = inputs.prefill_inputs(1, 2, 2048, 2048, 128, torch.bfloat16, seed=0)
    dout = inputs.prefill_inputs(1, 2, 2048, 2048, 128, torch.bfloat16, seed=1)[0]
    check(q, k, v, dout, 1 / math.sqrt(128), "causal", "causal 2k")


@pytest.mark.parametrize("mask", ["causal", "band"])
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16")])
def test_backward_many_heads_launch_groups(mask, d, dt):
    """B=2, H=55, Sq=Sk=300: 110 heads of three key blocks, 330 CTAs of the dK/dV kernel. Its
    launch order takes heads in groups whose CTAs make about two waves (on 152 SMs, 102 heads
    of three CTAs) and, within a group, key block by key block, so here the last group is a
    partial one of 8 heads. Every gradient of every head against the oracle: a CTA mapped to
    the wrong (head, key block), or to one twice, leaves some dK and dV rows wrong."""
    q, k, v = inputs.prefill_inputs(2, 55, 300, 300, d, DT[dt], seed=d + 7)
    dout = inputs.prefill_inputs(2, 55, 300, 300, d, DT[dt], seed=d + 8)[0]
    check(q, k, v, dout, 1 / math.sqrt(d), mask, f"110 heads d{d} {dt} {mask}")


def _layout(H, Sq, Sk, seed, density=0.4):
    g = torch.Generator().manual_seed(seed)
    nq, nk = -(-Sq // fa.FA_LAYOUT_BLOCK), -(-Sk // fa.FA_LAYOUT_BLOCK)
    lay = (torch.rand(H, nq, nk, generator=g) < density).to(torch.uint8)
    lay[0, 0, :] = 0          # a query block of head 0 sees nothing
    lay[-1, -1, :] = 1        # a query block of the last head sees every key block but one:
    lay[-1, :, 0] = 0         # key block 0 of the last head, which no query sees
    return lay


@pytest.mark.parametrize("Sq,Sk", [(127, 129), (200, 333), (384, 384), (520, 257)])
@pytest.mark.parametrize("d,dt", [(64, "f16"), (128, "bf16")])
def test_backward_block_sparse(Sq, Sk, d, dt):
    """fa_bwd_block_sparse against the oracle's backward under the same layout; exact zeros
    for the query block that sees nothing and the key block no query sees."""
    B, H = 2, 3
    q, k, v = inputs.prefill_inputs(B, H, Sq, Sk, d, DT[dt], seed=Sq * 3 + Sk)
    dout = inputs.prefill_inputs(B, H, Sq, Sq, d, DT[dt], seed=Sq + 5)[0]
    lay = _layout(H, Sq, Sk, seed=Sq + Sk)
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda")
    qd, kd, vd, gd, ld = q.to(dev), k.to(dev), v.to(dev), dout.to(dev), lay.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, fa.FA_MASK_BLOCK_SPARSE, block_layout=ld)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, Sq), dtype=torch.uint8, device=dev)
    fa.fa_bwd_block_sparse(qd, kd, vd, o, gd, lse, dq, dk, dv, ws, scale, ld)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    rq, rk, rv = oracle.attention_backward_layout(q, k, v, dout, scale, lay.numpy())
    got = [t.float().cpu().numpy() for t in (dq, dk, dv)]
    what = f"block-sparse {Sq}x{Sk} d{d} {dt}"
    compare_grad(got[0], rq, what + " dq")
    compare_grad(got[1], rk, what + " dk")
    compare_grad(got[2], rv, what + " dv")
    assert np.all(got[0][:, 0, :min(128, Sq)] == 0)
    assert np.all(got[1][:, -1, :min(128, Sk)] == 0) and np.all(got[2][:, -1, :min(128, Sk)] == 0)
    with pytest.raises(fa.FaError):  # a layout mask without a layout is refused
        fa.fa_bwd(qd, kd, vd, o, gd, lse, dq, dk, dv, ws, scale, fa.FA_MASK_BLOCK_SPARSE)


@pytest.mark.parametrize("sparse", [False, True])
def test_backward_4k_bench_configuration_sampled_heads(sparse):
    """The bench's backward configurations at full size, B=4 H=32 S=4096 d=128 bf16 (causal,
    or the BigBird-shaped block layout of the block-sparse bench), run as the bench runs them;
    the gradients of two (batch, head) pairs checked element by element against the oracle on
    those heads alone (heads are independent)."""
    B, H, S, d = 4, 32, 4096, 128
    q, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=0)
    dout = inputs.prefill_inputs(B, H, S, S, d, torch.bfloat16, seed=1)[0]
    scale = 1 / math.sqrt(d)
    dev = torch.device("cuda")
    qd, kd, vd, gd = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    lay = inputs.block_layout(H, S, S) if sparse else None
    mode = fa.FA_MASK_BLOCK_SPARSE if sparse else fa.FA_MASK_CAUSAL
    if sparse:
        fa.fa_fwd_ex(qd, kd, vd, o, lse, scale, mode, block_layout=lay.to(dev))
    else:
        fa.fa_fwd(qd, kd, vd, o, lse, scale, mode)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, S), dtype=torch.uint8, device=dev)
    fa.fa_bwd(qd, kd, vd, o, gd, lse, dq, dk, dv, ws, scale, mode,
              block_layout=lay.to(dev) if sparse else None)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    for b, h in ((0, 0), (3, 29)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        args = (q[sl], k[sl], v[sl], dout[sl], scale)
        if sparse:
            ref = oracle.attention_backward_layout(*args, lay[h:h + 1].numpy())
        else:
            ref = oracle.attention_backward(*args, oracle.MASK_CAUSAL)
        for got, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            compare_grad(got[sl].float().cpu().numpy(), r, f"4k {'sparse' if sparse else 'causal'} "
                                                           f"b{b} h{h} {name}")
