"""Pins for the FP64 CPU oracle: each test ties it to something other than itself.

Closed forms (hand-worked examples, constant scores, one-hot scores, causal row 0,
pair counts), invariances (key permutation, affine values, splitting one attention
into calls over disjoint key sets), special cases (window >= Sk, window = 1, global
tokens covering everything, decode with one token, an identity page table) and a
library routine (torch's scaled_dot_product_attention in float64 with a boolean
mask built here from index ranges).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import MASK_BAND, MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_NONE, MASK_PREFIX_LM
from tiled_attention_06_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")
MASKS = {"none": MASK_NONE, "causal": MASK_CAUSAL, "causal_window": MASK_CAUSAL_WINDOW}


def _val(x):
    """Parse the small closed-form tokens used in the golden file."""
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln7": math.log(7),
             "ln13": math.log(13), "3ln2": 3 * math.log(2), "-inf": -math.inf, "nan": math.nan,
             "1": 1.0}
    if x in table:
        return table[x]
    a, b = x.split("/")
    return float(a) / float(b)


def _arr(x):
    return np.vectorize(_val, otypes=[np.float64])(np.array(x, dtype=object))


# --------------------------------------------------------------------------- #
# element decoding                                                            #
# --------------------------------------------------------------------------- #

def test_decode_every_half_pattern_matches_ieee():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    got = oracle.elem_values(bits.view(torch.float16))
    want = bits.numpy().view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_decode_every_bf16_pattern_matches_torch():
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = oracle.elem_values(t)
    want = t.to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


# --------------------------------------------------------------------------- #
# the mask                                                                    #
# --------------------------------------------------------------------------- #

def _mask_matrix(Sq, Sk, mode, window=0, n_global=0):
    return np.array([[oracle.visible(i, j, Sq, Sk, mode, window, n_global) for j in range(Sk)]
                     for i in range(Sq)], dtype=bool)


def _mask_by_ranges(Sq, Sk, mode, window=0, n_global=0):
    """The same masks, built independently from index ranges (torch.tril)."""
    delta = Sk - Sq
    ones = torch.ones(Sq, Sk, dtype=torch.bool)
    if mode == MASK_NONE:
        return ones
    if mode == MASK_BAND:   # |pos - j| <= window
        return torch.tril(ones, diagonal=delta + window) & torch.triu(ones, diagonal=delta - window)
    causal = torch.tril(ones, diagonal=delta)
    if mode == MASK_PREFIX_LM:
        prefix = torch.zeros(Sq, Sk, dtype=torch.bool)
        prefix[:, :min(n_global, Sk)] = True
        return causal | prefix
    if mode == MASK_CAUSAL:
        return causal
    too_far = torch.tril(ones, diagonal=delta - window)   # pos - j >= window
    glob = torch.zeros(Sq, Sk, dtype=torch.bool)
    glob[:, :min(n_global, Sk)] = True
    return causal & (~too_far | glob)


def test_mask_hand_enumerated():
    c = _mask_matrix(4, 4, MASK_CAUSAL)
    assert c.tolist() == [[1, 0, 0, 0], [1, 1, 0, 0], [1, 1, 1, 0], [1, 1, 1, 1]]
    w = _mask_matrix(5, 5, MASK_CAUSAL_WINDOW, window=2, n_global=1)
    assert w.astype(int).tolist() == [[1, 0, 0, 0, 0],
                                      [1, 1, 0, 0, 0],
                                      [1, 1, 1, 0, 0],
                                      [1, 0, 1, 1, 0],
                                      [1, 0, 0, 1, 1]]
    # bottom-right alignment when Sq < Sk and when Sq > Sk
    assert _mask_matrix(2, 4, MASK_CAUSAL).astype(int).tolist() == [[1, 1, 1, 0], [1, 1, 1, 1]]
    assert _mask_matrix(3, 2, MASK_CAUSAL).astype(int).tolist() == [[0, 0], [1, 0], [1, 1]]
    assert _mask_matrix(2, 3, MASK_NONE).all()


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (7, 7), (16, 9), (9, 16), (33, 65)])
@pytest.mark.parametrize("mode,window,n_global", [(MASK_NONE, 0, 0), (MASK_CAUSAL, 0, 0),
                                                  (MASK_CAUSAL_WINDOW, 1, 0),
                                                  (MASK_CAUSAL_WINDOW, 4, 3),
                                                  (MASK_CAUSAL_WINDOW, 100, 0),
                                                  (MASK_CAUSAL_WINDOW, 3, 100),
                                                  (MASK_BAND, 0, 0), (MASK_BAND, 3, 0),
                                                  (MASK_BAND, 100, 0), (MASK_PREFIX_LM, 0, 0),
                                                  (MASK_PREFIX_LM, 0, 5),
                                                  (MASK_PREFIX_LM, 0, 100)])
def test_mask_matches_range_construction(Sq, Sk, mode, window, n_global):
    got = _mask_matrix(Sq, Sk, mode, window, n_global)
    want = _mask_by_ranges(Sq, Sk, mode, window, n_global).numpy()
    assert np.array_equal(got, want)


def _window_pairs_closed_form(S, w, g):
    """Visible pairs for CAUSAL_WINDOW with Sq = Sk = S: the band holds
    min(i+1, w) keys; the global keys add those j < g that lie left of the band."""
    band = sum(min(i + 1, w) for i in range(S))
    extra = sum(max(0, min(g, i - w + 1)) for i in range(S))
    return band + extra


def test_pair_counts_closed_forms():
    for S in (1, 2, 5, 64, 129):
        assert oracle.count_visible(S, S, MASK_NONE) == S * S
        assert oracle.count_visible(S, S, MASK_CAUSAL) == S * (S + 1) // 2
    assert oracle.count_visible(3, 7, MASK_NONE) == 21
    # Sq < Sk causal: row i sees delta + i + 1 keys
    assert oracle.count_visible(3, 7, MASK_CAUSAL) == 5 + 6 + 7
    for S, w, g in [(50, 7, 3), (64, 64, 0), (100, 10, 20), (33, 1, 0)]:
        assert oracle.count_visible(S, S, MASK_CAUSAL_WINDOW, w, g) == _window_pairs_closed_form(S, w, g)
    # the long-context configuration: S=32768, window 2048, 64 global keys
    assert _window_pairs_closed_form(32768, 2048, 64) == 66_976_800


def test_band_and_prefix_masks_hand_enumerated():
    b = _mask_matrix(5, 5, MASK_BAND, window=1)
    assert b.astype(int).tolist() == [[1, 1, 0, 0, 0],
                                      [1, 1, 1, 0, 0],
                                      [0, 1, 1, 1, 0],
                                      [0, 0, 1, 1, 1],
                                      [0, 0, 0, 1, 1]]
    p = _mask_matrix(5, 5, MASK_PREFIX_LM, n_global=2)
    assert p.astype(int).tolist() == [[1, 1, 0, 0, 0],
                                      [1, 1, 0, 0, 0],
                                      [1, 1, 1, 0, 0],
                                      [1, 1, 1, 1, 0],
                                      [1, 1, 1, 1, 1]]
    # Sq < Sk: the queries sit at the last positions
    assert _mask_matrix(2, 4, MASK_BAND, window=1).astype(int).tolist() == [[0, 1, 1, 1],
                                                                            [0, 0, 1, 1]]


def test_band_and_prefix_pair_counts():
    for S, w in [(1, 0), (10, 0), (10, 3), (64, 20), (30, 100)]:
        want = sum(min(i + w, S - 1) - max(i - w, 0) + 1 for i in range(S))
        assert oracle.count_visible(S, S, MASK_BAND, w, 0) == want
    for S, g in [(1, 0), (10, 3), (64, 20), (30, 100)]:
        want = sum(max(i + 1, min(g, S)) for i in range(S))
        assert oracle.count_visible(S, S, MASK_PREFIX_LM, 0, g) == want


def test_band_and_prefix_special_cases():
    S = 29
    q, k, v = inputs.prefill_inputs(1, 2, S, S, 16, torch.float16, seed=101)
    on, ln = oracle.attention(q, k, v, 0.25, MASK_NONE)
    oc, lc = oracle.attention(q, k, v, 0.25, MASK_CAUSAL)
    ob, lb = oracle.attention(q, k, v, 0.25, MASK_BAND, S, 0)        # band covers all
    np.testing.assert_array_equal(ob, on)
    np.testing.assert_array_equal(lb, ln)
    o0, _ = oracle.attention(q, k, v, 0.25, MASK_BAND, 0, 0)         # only itself
    np.testing.assert_array_equal(o0, v.double().numpy())
    op, lp = oracle.attention(q, k, v, 0.25, MASK_PREFIX_LM, 0, 0)   # no prefix: causal
    np.testing.assert_array_equal(op, oc)
    np.testing.assert_array_equal(lp, lc)
    op, lp = oracle.attention(q, k, v, 0.25, MASK_PREFIX_LM, 0, S)   # all prefix: none
    np.testing.assert_array_equal(op, on)


@pytest.mark.slow
def test_pair_count_long_context_brute_force():
    assert oracle.count_visible(32768, 32768, MASK_CAUSAL_WINDOW, 2048, 64) == 66_976_800


# --------------------------------------------------------------------------- #
# tile classes                                                                #
# --------------------------------------------------------------------------- #

def test_tile_class_hand_classified():
    E, P, F = oracle.TILE_EMPTY, oracle.TILE_PARTIAL, oracle.TILE_FULL
    # S=8, 4x4 tiles, causal: diagonal partial, below full, above empty
    grid = [[oracle.tile_class(mb, nb, 4, 4, 8, 8, MASK_CAUSAL) for nb in range(2)] for mb in range(2)]
    assert grid == [[P, E], [F, P]]
    # ragged: S=6 -> the second row/column of tiles hangs over the end
    grid = [[oracle.tile_class(mb, nb, 4, 4, 6, 6, MASK_NONE) for nb in range(2)] for mb in range(2)]
    assert grid == [[F, P], [P, P]]
    # window 4, 1 global key, S=16, 4x4 tiles
    grid = [[oracle.tile_class(mb, nb, 4, 4, 16, 16, MASK_CAUSAL_WINDOW, 4, 1) for nb in range(4)]
            for mb in range(4)]
    assert grid == [[P, E, E, E],
                    [P, P, E, E],
                    [P, P, P, E],
                    [P, E, P, P]]
    # a tile entirely past the end of the keys is empty
    assert oracle.tile_class(0, 2, 4, 4, 8, 8, MASK_NONE) == E


def test_tile_class_agrees_with_mask_counts():
    for (Sq, Sk, BM, BN, mode, w, g) in [(37, 37, 8, 16, MASK_CAUSAL, 0, 0),
                                         (40, 29, 16, 8, MASK_CAUSAL, 0, 0),
                                         (64, 64, 8, 8, MASK_CAUSAL_WINDOW, 12, 5),
                                         (23, 41, 4, 8, MASK_NONE, 0, 0)]:
        m = _mask_by_ranges(Sq, Sk, mode, w, g).numpy()
        nmb, nnb = -(-Sq // BM), -(-Sk // BN) + 1
        for mb in range(nmb):
            for nb in range(nnb):
                blk = m[mb * BM:(mb + 1) * BM, nb * BN:(nb + 1) * BN]
                full_shape = blk.shape == (BM, BN)
                want = (oracle.TILE_EMPTY if not blk.any() else
                        oracle.TILE_FULL if (full_shape and blk.all()) else oracle.TILE_PARTIAL)
                assert oracle.tile_class(mb, nb, BM, BN, Sq, Sk, mode, w, g) == want


# --------------------------------------------------------------------------- #
# attention: hand-worked closed forms                                         #
# --------------------------------------------------------------------------- #

def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))


def test_golden_hand_examples():
    data = json.load(open(GOLDEN))
    for ex in data["examples"]:
        q = _t(_arr(ex["q"]))[None, None]
        k = _t(_arr(ex["k"]))[None, None]
        v = _t(_arr(ex["v"]))[None, None]
        o, lse = oracle.attention(q, k, v, _val(ex["scale"]), MASKS[ex["mask"]], ex["window"],
                                  ex["n_global"])
        np.testing.assert_allclose(o[0, 0], _arr(ex["o"]), rtol=0, atol=1e-12, err_msg=ex["name"])
        np.testing.assert_allclose(lse[0, 0], _arr(ex["lse"]), rtol=0, atol=1e-12, err_msg=ex["name"])


def test_golden_decode_example():
    data = json.load(open(GOLDEN))
    for ex in data["decode_examples"]:
        o, lse = oracle.decode_paged(_t(_arr(ex["q"])), _t(_arr(ex["k_pages"])),
                                     _t(_arr(ex["v_pages"])),
                                     torch.tensor(ex["block_table"], dtype=torch.int32),
                                     torch.tensor(ex["ctx_lens"], dtype=torch.int32),
                                     _val(ex["scale"]))
        np.testing.assert_allclose(o, _arr(ex["o"]), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, _arr(ex["lse"]), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- #
# attention: closed forms on random data                                      #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("mode,w,g", [(MASK_NONE, 0, 0), (MASK_CAUSAL, 0, 0),
                                      (MASK_CAUSAL_WINDOW, 5, 2)])
def test_constant_scores_give_mean_of_visible_values(mode, w, g):
    B, H, S, d = 1, 2, 23, 8
    q = torch.zeros(B, H, S, d, dtype=torch.float16)
    _, k, v = inputs.prefill_inputs(B, H, S, S, d, torch.float16, seed=3)
    o, lse = oracle.attention(q, k, v, 0.3, mode, w, g)
    vv = v.double().numpy()
    m = _mask_by_ranges(S, S, mode, w, g).numpy()
    for i in range(S):
        sel = np.nonzero(m[i])[0]
        np.testing.assert_allclose(o[:, :, i], vv[:, :, sel].mean(axis=2), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, :, i], math.log(sel.size), rtol=0, atol=1e-13)


def test_one_hot_scores_select_a_value_row():
    B, H, S, d = 1, 1, 40, 64
    t = 17
    q = torch.zeros(B, H, S, d, dtype=torch.float16)
    q[..., 0] = 240.0                      # exact in fp16; 240 * scale = 30
    k = torch.zeros(B, H, S, d, dtype=torch.float16)
    k[0, 0, t, 0] = 1.0
    _, _, v = inputs.prefill_inputs(B, H, S, S, d, torch.float16, seed=5)
    o, lse = oracle.attention(q, k, v, 0.125, MASK_NONE)
    vt = v[0, 0, t].double().numpy()
    bound = (S - 1) * math.exp(-30) * 2 * float(v.double().abs().max())
    for i in range(S):
        assert np.max(np.abs(o[0, 0, i] - vt)) <= bound
        assert abs(lse[0, 0, i] - (30 + math.log1p((S - 1) * math.exp(-30)))) < 1e-12


def test_causal_row_zero_is_first_value():
    q, k, v = inputs.prefill_inputs(2, 3, 50, 50, 16, torch.bfloat16, seed=7)
    o, lse = oracle.attention(q, k, v, 0.25, MASK_CAUSAL)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0].double().numpy())
    s00 = 0.25 * (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy()
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-13)


def test_probabilities_sum_to_one():
    q, k, v = inputs.prefill_inputs(1, 2, 70, 90, 32, torch.float16, seed=9)
    for mode in (MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW):
        _, _, err = oracle.attention(q, k, v, 0.2, mode, 9, 4, return_psum_err=True)
        assert err < 1e-12


# --------------------------------------------------------------------------- #
# attention: a library routine                                                #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("Sq,Sk", [(33, 33), (17, 49), (64, 64)])
@pytest.mark.parametrize("mode,w,g", [(MASK_NONE, 0, 0), (MASK_CAUSAL, 0, 0),
                                      (MASK_CAUSAL_WINDOW, 6, 3), (MASK_BAND, 5, 0),
                                      (MASK_PREFIX_LM, 0, 7)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_matches_torch_sdpa_float64(Sq, Sk, mode, w, g, dtype):
    q, k, v = inputs.prefill_inputs(2, 2, Sq, Sk, 32, dtype, seed=11)
    scale = 1 / math.sqrt(32)
    o, lse = oracle.attention(q, k, v, scale, mode, w, g)
    mask = _mask_by_ranges(Sq, Sk, mode, w, g)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(),
                                                           attn_mask=mask, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = torch.einsum("bhid,bhjd->bhij", q.double(), k.double()) * scale
    s = s.masked_fill(~mask, -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- #
# attention: invariances and special cases                                    #
# --------------------------------------------------------------------------- #

def test_key_permutation_invariance():
    q, k, v = inputs.prefill_inputs(1, 2, 20, 31, 16, torch.float16, seed=13)
    perm = torch.randperm(31, generator=torch.Generator().manual_seed(1))
    o1, l1 = oracle.attention(q, k, v, 0.25)
    o2, l2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.25)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_affine_values():
    q, k, v = inputs.prefill_inputs(1, 2, 25, 25, 16, torch.float64, seed=17)
    a, b = -2.5, 0.75
    for mode in (MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW):
        o1, _ = oracle.attention(q, k, v, 0.3, mode, 4, 2)
        o2, _ = oracle.attention(q, k, a * v + b, 0.3, mode, 4, 2)
        np.testing.assert_allclose(o2, a * o1 + b, rtol=0, atol=1e-12)


def test_split_into_key_ranges_and_merge_by_lse():
    """Splitting one attention into calls over disjoint key sets and merging by
    LSE is exact (ascend-transformer-boost scenario 4)."""
    q, k, v = inputs.prefill_inputs(1, 2, 12, 40, 16, torch.float16, seed=19)
    o, lse = oracle.attention(q, k, v, 0.25)
    parts = [(0, 9), (9, 10), (10, 33), (33, 40)]
    os_, ls_ = [], []
    for a, b in parts:
        oo, ll = oracle.attention(q, k[:, :, a:b], v[:, :, a:b], 0.25)
        os_.append(oo)
        ls_.append(ll)
    L = np.logaddexp.reduce(np.stack(ls_), axis=0)
    merged = sum(np.exp(l - L)[..., None] * oo for oo, l in zip(os_, ls_))
    np.testing.assert_allclose(merged, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L, lse, rtol=0, atol=1e-13)


def test_window_special_cases():
    S = 37
    q, k, v = inputs.prefill_inputs(1, 2, S, S, 16, torch.bfloat16, seed=23)
    oc, lc = oracle.attention(q, k, v, 0.25, MASK_CAUSAL)
    ow, lw = oracle.attention(q, k, v, 0.25, MASK_CAUSAL_WINDOW, S, 0)    # window covers all
    np.testing.assert_array_equal(ow, oc)
    np.testing.assert_array_equal(lw, lc)
    og, lg = oracle.attention(q, k, v, 0.25, MASK_CAUSAL_WINDOW, 3, S)    # all keys global
    np.testing.assert_array_equal(og, oc)
    o1, _ = oracle.attention(q, k, v, 0.25, MASK_CAUSAL_WINDOW, 1, 0)     # only itself
    np.testing.assert_array_equal(o1, v.double().numpy())


def test_ragged_and_empty_shapes():
    q, k, v = inputs.prefill_inputs(1, 1, 0, 5, 8, torch.float16, seed=29)
    o, lse = oracle.attention(q, k, v, 0.3, MASK_CAUSAL)
    assert o.shape == (1, 1, 0, 8)
    q, k, v = inputs.prefill_inputs(1, 1, 4, 0, 8, torch.float16, seed=29)
    o, lse = oracle.attention(q, k, v, 0.3, MASK_NONE)
    assert np.all(o == 0) and np.all(lse == -np.inf)
    q, k, v = inputs.prefill_inputs(1, 1, 5, 3, 8, torch.float16, seed=29)
    o, lse = oracle.attention(q, k, v, 0.3, MASK_CAUSAL)   # rows 0,1 see nothing
    assert np.all(o[0, 0, :2] == 0) and np.all(lse[0, 0, :2] == -np.inf)
    np.testing.assert_array_equal(o[0, 0, 2], v[0, 0, 0].double().numpy())


# --------------------------------------------------------------------------- #
# the blocked online recurrence                                               #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("block_n", [1, 3, 64])
@pytest.mark.parametrize("tau", [0.0, 8 * math.log(2)])
@pytest.mark.parametrize("mode", [MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW])
def test_online_recurrence_equals_full_softmax(block_n, tau, mode):
    q, k, v = inputs.prefill_inputs(1, 2, 30, 70, 16, torch.float16, factor=2.0, seed=31)
    o, lse = oracle.attention(q, k, v, 0.5, mode, 11, 3)
    o1, l1 = oracle.online_attention(q, k, v, 0.5, mode, 11, 3, block_n, tau,
                                     oracle.REC_UNNORMALISED)
    np.testing.assert_allclose(o1, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, lse, rtol=0, atol=1e-12)
    o2, l2 = oracle.online_attention(q, k, v, 0.5, mode, 11, 3, block_n, tau,
                                     oracle.REC_NORMALISED)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, lse, rtol=0, atol=1e-12)


def test_literal_page_two_update_is_not_softmax():
    """The per-block output update printed on the zwxr.cn page (section 3.1) drops
    the factor l on the old output; with more than one block it is wrong, which is
    why the corrected form is the one the implementation follows."""
    q, k, v = inputs.prefill_inputs(1, 1, 8, 64, 16, torch.float16, seed=37)
    o, _ = oracle.attention(q, k, v, 0.5)
    o3, _ = oracle.online_attention(q, k, v, 0.5, MASK_NONE, 0, 0, 16, 0.0,
                                    oracle.REC_LITERAL_P2)
    assert np.max(np.abs(o3 - o)) > 1e-2
    o1, _ = oracle.online_attention(q, k, v, 0.5, MASK_NONE, 0, 0, 64, 0.0,
                                    oracle.REC_LITERAL_P2)    # one block: agrees
    np.testing.assert_allclose(o1, o, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- #
# paged decode                                                                #
# --------------------------------------------------------------------------- #

def _contiguous_kv(di):
    """Gather each sequence's K/V rows into [H, ctx, d] by plain indexing."""
    out = []
    for b in range(di.B):
        c = int(di.ctx_lens[b])
        pages = [int(p) for p in di.block_table[b, :(c + di.page_size - 1) // di.page_size]]
        kk = torch.cat([di.k_pages[p] for p in pages], dim=1)[:, :c] if pages else di.k_pages[:0, :, :0].squeeze(0)
        vv = torch.cat([di.v_pages[p] for p in pages], dim=1)[:, :c] if pages else di.v_pages[:0, :, :0].squeeze(0)
        out.append((kk, vv))
    return out


def test_decode_equals_last_row_of_prefill():
    di = inputs.decode_inputs(B=5, H=3, d=16, page_size=8, num_pages=40, max_ctx=60,
                              dtype=torch.float16, seed=41)
    o, lse = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens, 0.25)
    for b, (kk, vv) in enumerate(_contiguous_kv(di)):
        for mode in (MASK_NONE, MASK_CAUSAL):   # the query is the last position: same result
            ob, lb = oracle.attention(di.q[b][:, None, :][None], kk[None], vv[None], 0.25, mode)
            np.testing.assert_allclose(o[b], ob[0, :, 0], rtol=0, atol=1e-13)
            np.testing.assert_allclose(lse[b], lb[0, :, 0], rtol=0, atol=1e-13)


def test_decode_single_token_and_identity_table():
    di = inputs.decode_inputs(B=3, H=2, d=8, page_size=4, num_pages=12, max_ctx=16,
                              dtype=torch.bfloat16, seed=43, ctx_lens=[1, 16, 5])
    o, _ = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens, 0.5)
    first_page = int(di.block_table[0, 0])
    np.testing.assert_array_equal(o[0], di.v_pages[first_page, :, 0].double().numpy())
    # identity table over a contiguous pool equals attention over the contiguous rows
    H, d, P = 2, 8, 4
    _, k, v = inputs.prefill_inputs(1, H, 1, 16, d, torch.float16, seed=47)
    kp = k[0].reshape(H, 4, P, d).permute(1, 0, 2, 3).contiguous()
    vp = v[0].reshape(H, 4, P, d).permute(1, 0, 2, 3).contiguous()
    q = inputs.prefill_inputs(1, H, 1, 1, d, torch.float16, seed=53)[0]
    o1, l1 = oracle.decode_paged(q[0, :, 0][None], kp, vp, torch.arange(4, dtype=torch.int32)[None],
                                 torch.tensor([16], dtype=torch.int32), 0.3)
    o2, l2 = oracle.attention(q, k, v, 0.3)
    np.testing.assert_allclose(o1[0], o2[0, :, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1[0], l2[0, :, 0], rtol=0, atol=1e-13)


def test_decode_empty_context():
    di = inputs.decode_inputs(B=2, H=2, d=8, page_size=4, num_pages=8, max_ctx=16,
                              dtype=torch.float16, seed=59, ctx_lens=[0, 3])
    o, lse = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens, 0.5)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(o[1]))


def test_decode_rejects_out_of_range_page():
    di = inputs.decode_inputs(B=1, H=1, d=8, page_size=4, num_pages=4, max_ctx=8,
                              dtype=torch.float16, seed=61, ctx_lens=[6])
    bt = di.block_table.clone()
    bt[0, 1] = 4
    with pytest.raises(ValueError):
        oracle.decode_paged(di.q, di.k_pages, di.v_pages, bt, di.ctx_lens, 0.5)


@pytest.mark.parametrize("pps", [1, 2, 3])
def test_split_partials_combine_to_unsplit(pps):
    """Decode split-K: softmax partials over any page-aligned partition merge
    exactly into the unsplit result."""
    di = inputs.decode_inputs(B=3, H=2, d=16, page_size=8, num_pages=30, max_ctx=70,
                              dtype=torch.float16, seed=67)
    o, lse = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens, 0.25)
    for b, (kk, vv) in enumerate(_contiguous_kv(di)):
        c = int(di.ctx_lens[b])
        nsplit = -(-c // (8 * pps))
        for h in range(2):
            qd = di.q[b, h].double().numpy()
            ms, ls, accs = [], [], []
            for s in range(nsplit):
                t0, t1 = oracle.decode_split_tokens(c, 8, pps, s)
                sc = 0.25 * (kk[h, t0:t1].double().numpy() @ qd)
                m = sc.max()
                p = np.exp(sc - m)
                ms.append(m)
                ls.append(p.sum())
                accs.append(p @ vv[h, t0:t1].double().numpy())
            oc, lc = oracle.combine_partials(ms, ls, np.stack(accs))
            np.testing.assert_allclose(oc, o[b, h], rtol=0, atol=1e-13)
            assert abs(lc - lse[b, h]) < 1e-13


def test_split_tokens_partition():
    for ctx in (0, 1, 255, 256, 257, 8192):
        for pps in (1, 2, 5):
            covered = []
            s = 0
            while True:
                a, b = oracle.decode_split_tokens(ctx, 256, pps, s)
                if a >= ctx:
                    break
                assert a == s * 256 * pps and b > a
                covered.extend(range(a, b))
                s += 1
            assert covered == list(range(ctx))
            assert s == -(-ctx // (256 * pps))


def test_combine_all_empty():
    o, lse = oracle.combine_partials([-np.inf, -np.inf], [0.0, 0.0], np.zeros((2, 4)))
    assert np.all(o == 0) and lse == -np.inf


# --------------------------------------------------------------------------- #
# brute force on tiny inputs                                                  #
# --------------------------------------------------------------------------- #

def test_brute_force_numpy_tiny():
    q, k, v = inputs.prefill_inputs(1, 1, 5, 6, 4, torch.float16, seed=71)
    o, lse = oracle.attention(q, k, v, 0.7, MASK_CAUSAL)
    Q, K, V = (x[0, 0].double().numpy() for x in (q, k, v))
    for i in range(5):
        js = [j for j in range(6) if j <= i + 1]
        s = np.array([0.7 * sum(Q[i, c] * K[j, c] for c in range(4)) for j in js])
        p = np.exp(s - s.max())
        np.testing.assert_allclose(o[0, 0, i], (p / p.sum()) @ V[js], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[0, 0, i], s.max() + math.log(p.sum()), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- #
# prefill against a paged cache                                               #
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("mode,w,g", [(MASK_NONE, 0, 0), (MASK_CAUSAL, 0, 0),
                                      (MASK_CAUSAL_WINDOW, 9, 2)])
def test_paged_prefill_equals_attention_on_gathered_keys(mode, w, g):
    """Each sequence's rows equal or_attention with Sk = its length over its keys
    gathered in position order (random permutation table)."""
    di = inputs.decode_inputs(B=4, H=2, d=16, page_size=8, num_pages=40, max_ctx=60,
                              dtype=torch.bfloat16, seed=73, ctx_lens=[5, 60, 23, 8])
    Sq = 5
    q = inputs.prefill_inputs(4, 2, Sq, 1, 16, torch.bfloat16, seed=79)[0]
    o, lse = oracle.attention_paged(q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens,
                                    0.3, mode, w, g)
    for b, (kk, vv) in enumerate(_contiguous_kv(di)):
        ob, lb = oracle.attention(q[b:b + 1], kk[None], vv[None], 0.3, mode, w, g)
        np.testing.assert_allclose(o[b], ob[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], lb[0], rtol=0, atol=1e-13)


def test_paged_prefill_identity_table_and_single_query():
    H, d, P, S = 2, 8, 4, 16
    _, k, v = inputs.prefill_inputs(1, H, 1, S, d, torch.float16, seed=83)
    kp = k[0].reshape(H, S // P, P, d).permute(1, 0, 2, 3).contiguous()
    vp = v[0].reshape(H, S // P, P, d).permute(1, 0, 2, 3).contiguous()
    table = torch.arange(S // P, dtype=torch.int32)[None]
    ctx = torch.tensor([S], dtype=torch.int32)
    q = inputs.prefill_inputs(1, H, 6, 1, d, torch.float16, seed=89)[0]
    o1, l1 = oracle.attention_paged(q, kp, vp, table, ctx, 0.4, MASK_CAUSAL)
    o2, l2 = oracle.attention(q, k, v, 0.4, MASK_CAUSAL)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)
    # one query per sequence is the decode step
    di = inputs.decode_inputs(B=3, H=2, d=8, page_size=4, num_pages=20, max_ctx=24,
                              dtype=torch.float16, seed=97)
    od, ld = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table, di.ctx_lens, 0.5)
    op, lp = oracle.attention_paged(di.q[:, :, None, :], di.k_pages, di.v_pages, di.block_table,
                                    di.ctx_lens, 0.5, MASK_CAUSAL)
    np.testing.assert_allclose(op[:, :, 0], od, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lp[:, :, 0], ld, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- #
# block-sparse layouts                                                        #
# --------------------------------------------------------------------------- #

def _rand_layout(H, Sq, Sk, blk, seed, density=0.5):
    rng = np.random.default_rng(seed)
    return (rng.random((H, -(-Sq // blk), -(-Sk // blk))) < density).astype(np.uint8)


def test_layout_all_ones_is_no_mask_and_tril_block1_is_causal():
    q, k, v = (torch.randn(2, 3, 37, 16, generator=torch.Generator().manual_seed(s))
               .to(torch.bfloat16) for s in (1, 2, 3))
    ones = np.ones((3, 2, 2), dtype=np.uint8)  # blk 32 over 37 rows / keys
    o, lse = oracle.attention_layout(q, k, v, 0.25, ones, blk=32)
    o2, lse2 = oracle.attention(q, k, v, 0.25, MASK_NONE)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    tril = np.broadcast_to(np.tril(np.ones((37, 37), dtype=np.uint8)), (3, 37, 37))
    o, lse = oracle.attention_layout(q, k, v, 0.25, tril, blk=1)
    o2, lse2 = oracle.attention(q, k, v, 0.25, MASK_CAUSAL)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("Sq,Sk,blk", [(40, 40, 8), (33, 70, 16), (70, 33, 16), (5, 9, 4)])
def test_layout_matches_sdpa_with_expanded_mask(Sq, Sk, blk):
    H = 3
    g = torch.Generator().manual_seed(Sq * 100 + Sk)
    q = torch.randn(2, H, Sq, 16, generator=g).to(torch.float16)
    k = torch.randn(2, H, Sk, 16, generator=g).to(torch.float16)
    v = torch.randn(2, H, Sk, 16, generator=g).to(torch.float16)
    lay = _rand_layout(H, Sq, Sk, blk, seed=Sq + Sk)
    lay[0, 0, :] = 0  # head 0's first query block sees nothing
    o, lse = oracle.attention_layout(q, k, v, 0.3, lay, blk=blk)
    # the layout blown up to one flag per (query, key), built here with np.kron
    full = np.stack([np.kron(lay[h], np.ones((blk, blk), dtype=np.uint8))[:Sq, :Sk]
                     for h in range(H)]).astype(bool)
    mask = torch.from_numpy(full)[None].expand(2, H, Sq, Sk)
    seen = mask.any(-1)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double(),
                                                           attn_mask=mask, scale=0.3)
    rows = seen.numpy()
    np.testing.assert_allclose(o[rows], ref.numpy()[rows], rtol=0, atol=1e-12)
    assert np.all(o[~rows] == 0) and np.all(np.isneginf(lse[~rows]))
    s = torch.einsum("bhid,bhjd->bhij", q.double(), k.double()) * 0.3
    want = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1).numpy()
    np.testing.assert_allclose(lse[rows], want[rows], rtol=0, atol=1e-12)
    assert oracle.count_visible_layout(H, Sq, Sk, lay, blk) == int(full.sum())


def test_layout_key_block_permutation_invariance():
    H, S, blk = 2, 48, 16
    g = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn(1, H, S, 8, generator=g).to(torch.bfloat16) for _ in range(3))
    lay = _rand_layout(H, S, S, blk, seed=3, density=0.6)
    perm = [2, 0, 1]  # move whole key blocks, and the layout's columns with them
    idx = torch.cat([torch.arange(p * blk, (p + 1) * blk) for p in perm])
    o1, l1 = oracle.attention_layout(q, k, v, 0.5, lay, blk=blk)
    o2, l2 = oracle.attention_layout(q, k[:, :, idx], v[:, :, idx], 0.5, lay[:, :, perm],
                                     blk=blk)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_layout_counts_and_tile_classes():
    lay = np.array([[[1, 0], [1, 1]]], dtype=np.uint8)  # one head, 2 x 2 blocks of 4
    # query rows 0-3 see keys 0-3; rows 4-6 (Sq = 7) see keys 0-5 (Sk = 6)
    assert oracle.count_visible_layout(1, 7, 6, lay, 4) == 4 * 4 + 3 * 6
    # 4x4 tiles: (0,0) full, (0,1) empty, (1,0) partial (3 of 4 rows), (1,1) partial
    classes = [[oracle.tile_class_layout(0, mb, nb, 4, 4, 7, 6, lay, 4) for nb in range(2)]
               for mb in range(2)]
    assert classes == [[oracle.TILE_FULL, oracle.TILE_EMPTY],
                       [oracle.TILE_PARTIAL, oracle.TILE_PARTIAL]]


# --------------------------------------------------------------------------- #
# backward                                                                    #
# --------------------------------------------------------------------------- #

def _explicit_mask(Sq, Sk, mode, w, g):
    """Visibility built here from index arithmetic (query i at key position i + Sk - Sq)."""
    i = torch.arange(Sq)[:, None] + (Sk - Sq)
    j = torch.arange(Sk)[None, :]
    if mode == MASK_NONE:
        return torch.ones(Sq, Sk, dtype=torch.bool)
    if mode == MASK_CAUSAL:
        return j <= i
    if mode == MASK_CAUSAL_WINDOW:
        return (j <= i) & ((i - j < w) | (j < g))
    if mode == MASK_BAND:
        return (j - i).abs() <= w
    return (j <= i) | (j < g)  # prefix-LM


@pytest.mark.parametrize("mode,w,g", [(MASK_NONE, 0, 0), (MASK_CAUSAL, 0, 0),
                                      (MASK_CAUSAL_WINDOW, 5, 2), (MASK_BAND, 3, 0),
                                      (MASK_PREFIX_LM, 0, 4)])
@pytest.mark.parametrize("Sq,Sk", [(17, 17), (9, 23), (23, 9)])
def test_backward_matches_autograd(mode, w, g, Sq, Sk):
    gen = torch.Generator().manual_seed(Sq * 31 + Sk + mode)
    q, k, v, do = (torch.randn(2, 3, n, 16, generator=gen).to(torch.bfloat16)
                   for n in (Sq, Sk, Sk, Sq))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, 0.3, mode, w, g)
    mask = _explicit_mask(Sq, Sk, mode, w, g)
    seen = mask.any(-1)
    qq, kk, vv = (t.double().requires_grad_() for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=0.3)
    # rows that see no key give NaN in SDPA and contribute nothing by definition
    o = torch.where(seen[None, None, :, None], o, torch.zeros_like(o))
    o.backward(do.double())
    for got, ref in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        ref = torch.nan_to_num(ref, nan=0.0).numpy()
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_backward_central_differences():
    """dL/dx for L = sum(G * O) by central differences of the FP64 forward."""
    gen = torch.Generator().manual_seed(5)
    q, k, v, G = (torch.randn(1, 2, n, 4, generator=gen, dtype=torch.float64)
                  for n in (6, 7, 7, 6))
    dq, dk, dv = oracle.attention_backward(q, k, v, G, 0.7, MASK_CAUSAL)
    eps = 1e-6

    def loss(qx, kx, vx):
        o, _ = oracle.attention(qx, kx, vx, 0.7, MASK_CAUSAL)
        return float((o * G.numpy()).sum())

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for idx in [(0, 0, 0, 0), (0, 1, 3, 2), (0, 1, 5, 3)]:
            plus = [t.clone() for t in (q, k, v)]
            minus = [t.clone() for t in (q, k, v)]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert abs(fd - grad[idx]) < 1e-7, (which, idx, fd, grad[idx])


def test_backward_closed_forms():
    gen = torch.Generator().manual_seed(9)
    q, k, v, do = (torch.randn(1, 2, 8, 8, generator=gen).to(torch.float16) for _ in range(4))
    # zero queries: every score is 0, dK = scale * sum_i dS_ij Q_i = 0
    _, dk, _ = oracle.attention_backward(torch.zeros_like(q), k, v, do, 0.5, MASK_NONE)
    assert np.all(dk == 0)
    # one visible key (causal row 0): P = 1, dS = 0, so dQ_0 = 0 and dV_0 gets dO_0 from it
    dq, _, dv = oracle.attention_backward(q, k, v, do, 0.5, MASK_CAUSAL)
    assert np.all(dq[:, :, 0] == 0)
    # identical keys: dQ_i = scale * K * sum_j dS_ij = 0 because each row of dS sums to 0
    kc = k[:, :, :1].expand(-1, -1, 8, -1).contiguous()
    dq, _, _ = oracle.attention_backward(q, kc, v, do, 0.5, MASK_NONE)
    np.testing.assert_allclose(dq, 0.0, atol=1e-13)
    # a row's dV contributions sum to dO_i: sum_j dV_j = sum_i dO_i (P rows sum to 1)
    _, _, dv = oracle.attention_backward(q, k, v, do, 0.5, MASK_NONE)
    np.testing.assert_allclose(dv.sum(axis=2), do.double().numpy().sum(axis=2), atol=1e-12)


# --------------------------------------------------------------------------- #
# rescale events of the lazy recurrence                                       #
# --------------------------------------------------------------------------- #

TAU = 8 * math.log(2)  # the kernels' threshold, 8 in log2 units, here in natural-log units


def _lazy_count_closed_form(rises, tau):
    """Rescales of a row whose visible blocks have maxima rising by rises[t] over the
    previous block: the reference moves only when the rise accumulated since it was last
    moved exceeds tau."""
    acc, n = 0.0, 0
    for r in rises:
        acc += r
        if acc > tau:
            n, acc = n + 1, 0.0
    return n


@pytest.mark.parametrize("block_n", [64, 128, 48])
@pytest.mark.parametrize("scale", [1 / 8, 1 / 512])
def test_rescale_events_closed_form_on_a_noiseless_ramp(block_n, scale):
    """q = 1, k_j = j / 8 (exact in fp16): s_j = scale * d * j / 8 rises by the same
    amount per key, so a row's block maxima sit at the block's last visible key. Each row's
    count follows from those rises in closed form: every block after the first when a
    block's rise exceeds tau (scale 1/8), only every ceil(tau / rise)-th block when it does
    not (scale 1/512: the lazy threshold, not an eager max update)."""
    d, S = 64, 700
    q = torch.ones(1, 1, S, d, dtype=torch.float16)
    k = (torch.arange(S, dtype=torch.float32)[:, None] / 8).expand(S, d).reshape(1, 1, S, d)
    k = k.to(torch.float16)
    assert torch.equal(k.float()[0, 0, :, 0] * 8, torch.arange(S, dtype=torch.float32))
    delta = scale * d / 8  # score rise per key
    for mode in (MASK_NONE, MASK_CAUSAL):
        counts, near = oracle.rescale_events(q, k, scale, block_n, TAU, mode, tile_rows=1)
        assert near.sum() == 0
        for i in range(S):
            last = S - 1 if mode == MASK_NONE else i  # last visible key of row i
            ends = [min(t + block_n, last + 1) - 1 for t in range(0, last + 1, block_n)]
            rises = [(ends[t] - ends[t - 1]) * delta for t in range(1, len(ends))]
            assert counts[0, i] == _lazy_count_closed_form(rises, TAU), (mode, i)
    # the same keys in descending order: the first block holds every row's maximum
    kd = k.flip(2).contiguous()
    counts, _ = oracle.rescale_events(q, kd, scale, block_n, TAU, MASK_NONE)
    assert counts.sum() == 0


def _brute_rescales(q, k, scale, block_n, tau, vis):
    """Rescale count of every row by a plain Python walk over the blocks."""
    qd, kd = q.double().numpy()[0, 0], k.double().numpy()[0, 0]
    out = []
    for i in range(qd.shape[0]):
        m, n = None, 0
        for j0 in range(0, kd.shape[0], block_n):
            js = [j for j in range(j0, min(j0 + block_n, kd.shape[0])) if vis(i, j)]
            if not js:
                continue
            b = max(scale * float(qd[i] @ kd[j]) for j in js)
            if m is None:
                m = b
            elif b - m > tau:
                m, n = b, n + 1
        out.append(n)
    return np.array(out)


@pytest.mark.parametrize("mask,w,g", [("none", 0, 0), ("causal", 0, 0), ("window", 40, 5),
                                      ("band", 30, 0), ("prefix", 0, 50), ("layout", 0, 0)])
def test_rescale_events_match_brute_force(mask, w, g):
    """Random wide scores (q, k ~ N(0,1) * 3): the per-row counts equal a plain Python walk
    of the blocks, for every mask and a block layout."""
    Sq, Sk, d, bn = 150, 260, 32, 16
    q, k, _ = inputs.prefill_inputs(1, 1, Sq, Sk, d, torch.bfloat16, factor=3.0, seed=17)
    scale = 1 / math.sqrt(d)
    mode = {"none": MASK_NONE, "causal": MASK_CAUSAL, "window": MASK_CAUSAL_WINDOW,
            "band": MASK_BAND, "prefix": MASK_PREFIX_LM, "layout": MASK_NONE}[mask]
    if mask == "layout":
        lay = inputs.block_layout(1, Sq, Sk, block=64, local=0, n_global=0, n_random=2, seed=3)
        def vis(i, j):
            return bool(lay[0, i // 64, j // 64])
        counts, near = oracle.rescale_events(q, k, scale, bn, TAU, layout=lay.numpy(), blk=64,
                                             tile_rows=1)
    else:
        def vis(i, j):
            return oracle.visible(i, j, Sq, Sk, mode, w, g)
        counts, near = oracle.rescale_events(q, k, scale, bn, TAU, mode, w, g, tile_rows=1)
    want = _brute_rescales(q, k, scale, bn, TAU, vis)
    assert want.sum() > 20  # the inputs do reach the rescale step
    assert np.array_equal(counts[0], want)
    # per-tile sums are the row counts added up
    c128, _ = oracle.rescale_events(q, k, scale, bn, TAU, mode, w, g, tile_rows=128,
                                    layout=lay.numpy() if mask == "layout" else None, blk=64)
    assert c128[0].tolist() == [int(want[:128].sum()), int(want[128:].sum())]


def test_rescale_events_threshold_limits():
    """A threshold above every rise gives no rescale; tau must be positive."""
    q, k, _ = inputs.prefill_inputs(1, 2, 64, 300, 64, torch.float16, factor=2.0, seed=4)
    counts, _ = oracle.rescale_events(q, k, 0.125, 32, 1e9)
    assert counts.sum() == 0
    with pytest.raises(ValueError):
        oracle.rescale_events(q, k, 0.125, 32, 0.0)


@pytest.mark.parametrize("Sq,Sk,blk", [(40, 40, 8), (33, 70, 16), (70, 33, 16)])
def test_backward_layout_matches_autograd_with_expanded_mask(Sq, Sk, blk):
    """Block-sparse gradients against torch autograd on float64 SDPA with the layout blown up
    into one flag per (query, key); the heads have different layouts and one query block of
    head 0 sees nothing."""
    H = 3
    gen = torch.Generator().manual_seed(Sq * 7 + Sk)
    q, k, v, do = (torch.randn(2, H, n, 16, generator=gen).to(torch.float16)
                   for n in (Sq, Sk, Sk, Sq))
    lay = _rand_layout(H, Sq, Sk, blk, seed=Sq * Sk, density=0.5)
    lay[0, 0, :] = 0
    dq, dk, dv = oracle.attention_backward_layout(q, k, v, do, 0.3, lay, blk=blk)
    full = np.stack([np.kron(lay[h], np.ones((blk, blk), dtype=np.uint8))[:Sq, :Sk]
                     for h in range(H)]).astype(bool)
    mask = torch.from_numpy(full)[None].expand(2, H, Sq, Sk)
    seen = mask.any(-1)
    qq, kk, vv = (t.double().requires_grad_() for t in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=0.3)
    o = torch.where(seen[..., None], o, torch.zeros_like(o))
    o.backward(do.double())
    for got, ref in ((dq, qq.grad), (dk, kk.grad), (dv, vv.grad)):
        ref = torch.nan_to_num(ref, nan=0.0).numpy()
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    assert np.all(dq[:, 0, :blk] == 0)  # the query block that sees nothing


def test_backward_layout_block1_tril_is_causal_per_head():
    """Block 1: a lower-triangular layout gives the causal gradients and an all-ones layout
    the unmasked ones, each for its own head."""
    S, H = 12, 2
    gen = torch.Generator().manual_seed(3)
    q, k, v, do = (torch.randn(1, H, S, 8, generator=gen).to(torch.bfloat16) for _ in range(4))
    lay = np.stack([np.ones((S, S), dtype=np.uint8), np.tril(np.ones((S, S), dtype=np.uint8))])
    got = oracle.attention_backward_layout(q, k, v, do, 0.5, lay, blk=1)
    dense = oracle.attention_backward(q, k, v, do, 0.5, MASK_NONE)
    causal = oracle.attention_backward(q, k, v, do, 0.5, MASK_CAUSAL)
    for g_, d_, c_ in zip(got, dense, causal):
        assert np.array_equal(g_[:, 0], d_[:, 0]) and np.array_equal(g_[:, 1], c_[:, 1])
