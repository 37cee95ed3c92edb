"""FP32 inputs, checked on the CPU: the bf16 high/low split that the FP32 path stores its
inputs in holds every value to 2^-16 (with an exact residual), and the resolution inputs of
the GPU test really need both parts: the same inputs rounded to bf16, or P rounded to
bf16, move the oracle's O by more than the 1e-3 bound, while the split inputs move it by
far less."""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_06_gb300 import inputs


def split(x):
    hi = x.to(torch.bfloat16).to(torch.float32)
    lo = (x - hi).to(torch.bfloat16).to(torch.float32)
    return hi, lo


def test_split_residual_is_exact_and_pair_holds_value():
    g = torch.Generator().manual_seed(0)
    # magnitudes over 2^-60 .. 2^60, both signs, plus values next to powers of two
    x = torch.randn(200000, generator=g) * torch.exp2(torch.randint(-60, 61, (200000,),
                                                                    generator=g).float())
    edge = torch.tensor([1.0, 1.0 - 2 ** -24, 1.0 + 2 ** -23, 3.0 - 2 ** -22, -0.75, 2 ** -100])
    x = torch.cat([x, edge, -edge])
    hi, lo = split(x)
    x64, hi64, lo64 = x.double(), hi.double(), lo.double()
    # x - hi in float32 equals the exact difference
    assert torch.equal((x - hi).double(), x64 - hi64)
    rel = ((hi64 + lo64 - x64).abs() / x64.abs())
    assert rel.max().item() <= 2.0 ** -16
    # the dropped lo*lo term of a product is below 2^-16 of it as well
    assert (lo64.abs() <= 2.0 ** -8 * x64.abs()).all()


def _np_attention(q, k, v, scale, causal, round_p=None):
    """Plain FP64 attention of one head, optionally rounding the unnormalised P."""
    s = scale * (q @ k.T)
    if causal:
        Sq, Sk = s.shape
        i = np.arange(Sq)[:, None] + (Sk - Sq)
        s = np.where(np.arange(Sk)[None, :] <= i, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    if round_p is not None:
        p = round_p(p)
    return (p @ v) / l


@pytest.mark.parametrize("mask", [oracle.MASK_CAUSAL, oracle.MASK_NONE])
def test_resolution_inputs_need_both_parts(mask):
    q, k, v = inputs.f32_resolution_inputs(1, 2, 300, 300, 64, seed=11)
    ref, _ = oracle.attention(q, k, v, 0.125, mask)

    def rounded(t):
        return t.to(torch.bfloat16).to(torch.float32)

    def pair(t):
        hi, lo = split(t)
        return (hi.double() + lo.double()).float()

    # high parts only: Q and K, or V alone, each miss the bound
    o_qk, _ = oracle.attention(rounded(q), rounded(k), v, 0.125, mask)
    o_v, _ = oracle.attention(q, k, rounded(v), 0.125, mask)
    assert np.abs(o_qk - ref).max() > 1e-3
    assert np.abs(o_v - ref).max() > 1e-3
    # inputs replaced by their split pairs (hi + lo, within 2^-16 of x) move O by far less
    o_pair, _ = oracle.attention(pair(q), pair(k), pair(v), 0.125, mask)
    assert np.abs(o_pair - ref).max() <= 1e-4
    # P rounded to bf16 before P V (l from the unrounded P) misses the bound too
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    bf = lambda p: torch.from_numpy(p).float().to(torch.bfloat16).double().numpy()
    causal = mask == oracle.MASK_CAUSAL
    o_p = np.stack([_np_attention(qn[0, h], kn[0, h], vn[0, h], 0.125, causal, bf)
                    for h in range(2)])
    assert np.abs(o_p - ref[0]).max() > 1e-3
    o_np = np.stack([_np_attention(qn[0, h], kn[0, h], vn[0, h], 0.125, causal)
                     for h in range(2)])
    assert np.abs(o_np - ref[0]).max() <= 1e-9  # the emulation itself is the definition
