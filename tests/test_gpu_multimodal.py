"""Cross attention (Sq != Sk) and the multimodal three-call split, through the C ABI.

"ascend-transformer-boost 实战" (ai6s.net), scenario 4, splits a vision+text attention
into a vision-internal call, a text-internal causal call and a text-to-vision cross call,
with identical results. Here the text queries' part of that layer (all vision keys plus
causal text keys) is also a single causal call over the concatenated keys (queries
aligned to the last keys), so the three-call split merged by LSE must match both that
single call and the FP64 oracle. The whole layer, vision rows included, is also one
prefix-LM call over the concatenated tokens with the vision tokens as the prefix.
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


def fwd(q, k, v, scale, mode, n_global=0):
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    fa.fa_fwd(q.contiguous(), k.contiguous(), v.contiguous(), o, lse, scale, mode,
              n_global=n_global)
    return o, lse


@pytest.mark.parametrize("d,dt", [(64, torch.float16), (128, torch.bfloat16)])
@pytest.mark.parametrize("split", [1, 37, 128, 199])
def test_merge_of_key_ranges_equals_whole(d, dt, split):
    q, k, v = inputs.prefill_inputs(2, 3, 150, 200, d, dt, seed=split)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    oa, la = fwd(qd, kd[:, :, :split], vd[:, :, :split], scale, fa.FA_MASK_NONE)
    ob, lb = fwd(qd, kd[:, :, split:], vd[:, :, split:], scale, fa.FA_MASK_NONE)
    o = torch.empty_like(oa)
    lse = torch.empty_like(la)
    fa.fa_merge_partials(oa, la, ob, lb, o, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(q, k, v, scale, oracle.MASK_NONE)
    compare(o, lse, ref_o, ref_l, f"merge split {split}")


def test_merge_with_empty_part():
    """Rows whose causal part sees nothing (LSE = -inf) take the other part unchanged."""
    q, k, v = inputs.prefill_inputs(1, 2, 64, 16, 64, torch.float16, seed=3)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    oa, la = fwd(qd, kd, vd, 0.125, fa.FA_MASK_CAUSAL)   # rows 0..47 see no key
    ob, lb = fwd(qd, kd, vd, 0.125, fa.FA_MASK_NONE)
    o = torch.empty_like(oa)
    lse = torch.empty_like(la)
    fa.fa_merge_partials(oa, la, ob, lb, o, lse)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, :48], ob[:, :, :48])
    assert torch.equal(lse[:, :, :48], lb[:, :, :48])
    e = torch.full_like(la, -math.inf)
    fa.fa_merge_partials(oa, e, ob, e, o, lse)    # both empty
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("V,T,H", [(96, 300, 2), (576, 2048, 32)])
def test_multimodal_three_call_split(V, T, H):
    """Vision 576 (24x24 patches) + text 2048 tokens, 32 heads of 128 (the pages'
    LLaVA-1.5 example shape), and a small ragged case."""
    d, dt = 128, torch.bfloat16
    q, k, v = inputs.prefill_inputs(1, H, V + T, V + T, d, dt, seed=V + T)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    qv, qt = qd[:, :, :V], qd[:, :, V:]
    kv_, kt = kd[:, :, :V], kd[:, :, V:]
    vv, vt = vd[:, :, :V], vd[:, :, V:]
    # call 1: vision tokens attend to vision tokens (full)
    o_vis, l_vis = fwd(qv, kv_, vv, scale, fa.FA_MASK_NONE)
    # call 2: text tokens attend causally to text tokens
    o_tt, l_tt = fwd(qt, kt, vt, scale, fa.FA_MASK_CAUSAL)
    # call 3: text tokens attend to every vision token
    o_tv, l_tv = fwd(qt, kv_, vv, scale, fa.FA_MASK_NONE)
    o_txt = torch.empty_like(o_tt)
    l_txt = torch.empty_like(l_tt)
    fa.fa_merge_partials(o_tt, l_tt, o_tv, l_tv, o_txt, l_txt)
    # the same text rows as one causal call over [vision; text] keys
    o_one, l_one = fwd(qt, kd, vd, scale, fa.FA_MASK_CAUSAL)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention(q[:, :, V:], k, v, scale, oracle.MASK_CAUSAL)
    compare(o_txt, l_txt, ref_o, ref_l, "text rows, split + merge")
    compare(o_one, l_one, ref_o, ref_l, "text rows, one call")
    ref_o, ref_l = oracle.attention(q[:, :, :V], k[:, :, :V], v[:, :, :V], scale,
                                    oracle.MASK_NONE)
    compare(o_vis, l_vis, ref_o, ref_l, "vision rows")
    # split and single call agree with each other beyond the oracle tolerance
    diff = (o_txt.float() - o_one.float()).abs().max().item()
    assert diff <= 1.6e-2


@pytest.mark.parametrize("V,T,H", [(96, 300, 2), (576, 2048, 8)])
def test_multimodal_layer_is_one_prefix_lm_call(V, T, H):
    """The whole layer, vision and text rows together, as one prefix-LM call over the
    concatenated [vision; text] tokens with the V vision tokens as the prefix: a vision
    query sees every vision key (j < V), and no text key since j <= i < V; a text query
    sees every vision key and the text keys up to its own position. So the vision rows
    equal call 1 of the split and the text rows the merged calls 2 and 3."""
    d, dt = 128, torch.bfloat16
    S = V + T
    q, k, v = inputs.prefill_inputs(1, H, S, S, d, dt, seed=3 * S)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = 1 / math.sqrt(d)
    o_all, l_all = fwd(qd, kd, vd, scale, fa.FA_MASK_PREFIX_LM, n_global=V)
    o_vis, l_vis = fwd(qd[:, :, :V], kd[:, :, :V], vd[:, :, :V], scale, fa.FA_MASK_NONE)
    o_tt, l_tt = fwd(qd[:, :, V:], kd[:, :, V:], vd[:, :, V:], scale, fa.FA_MASK_CAUSAL)
    o_tv, l_tv = fwd(qd[:, :, V:], kd[:, :, :V], vd[:, :, :V], scale, fa.FA_MASK_NONE)
    o_txt, l_txt = torch.empty_like(o_tt), torch.empty_like(l_tt)
    fa.fa_merge_partials(o_tt, l_tt, o_tv, l_tv, o_txt, l_txt)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    ref_o, ref_l = oracle.attention(q, k, v, scale, oracle.MASK_PREFIX_LM, 0, V)
    compare(o_all, l_all, ref_o, ref_l, "prefix-LM over [vision; text]")
    # against the split, row block by row block
    for rows, (o_s, l_s) in ((slice(0, V), (o_vis, l_vis)), (slice(V, S), (o_txt, l_txt))):
        diff = (o_all[:, :, rows].float() - o_s.float()).abs().max().item()
        assert diff <= 1.6e-2
        ldiff = (l_all[:, :, rows] - l_s).abs().max().item()
        assert ldiff <= 1e-3
