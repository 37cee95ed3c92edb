"""fa_decode_paged_noalloc: paged decode for callers that cannot allocate device memory.

Some users of this library cannot hand it a workspace: their device memory is fixed
when they start (a serving loop with a set budget), or a host program owns every
device allocation and gives its plug-ins no allocator. This entry point keeps the
decode's split partials in a scratch array built into the library instead. These
tests check, through the C ABI, that it gives the results of fa_decode_paged with a
caller workspace and of the FP64 oracle on two calls in a row (the second call reuses
whatever the first left in the shared array), that it serves the largest problem its
scratch holds, and that it refuses the next size up.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import build, inputs

from _util import compare

SCRATCH = 16 << 20  # bytes of the library's scratch array


def _run_both(di, scale):
    dev = "cuda"
    q, kp, vp = di.q.to(dev), di.k_pages.to(dev), di.v_pages.to(dev)
    bt, cl = di.block_table.to(dev), di.ctx_lens.to(dev)
    B, H, d = q.shape
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, d, bt.shape[1], di.page_size),
                     dtype=torch.uint8, device=dev)
    o_ws, l_ws = torch.empty_like(q), torch.empty(B, H, dtype=torch.float32, device=dev)
    fa.fa_decode_paged(q, kp, vp, bt, cl, o_ws, l_ws, scale, ws)
    o_na, l_na = torch.empty_like(q), torch.empty(B, H, dtype=torch.float32, device=dev)
    fa.fa_decode_paged_noalloc(q, kp, vp, bt, cl, o_na, l_na, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_status() == fa.FA_OK
    return o_ws, l_ws, o_na, l_na


def _check(di, scale, what):
    o_ws, l_ws, o_na, l_na = _run_both(di, scale)
    compare(o_na, l_na, o_ws.double().cpu().numpy(), l_ws.double().cpu().numpy(),
            f"{what}: against the workspace call")
    ref_o, ref_l = oracle.decode_paged(di.q, di.k_pages, di.v_pages, di.block_table,
                                       di.ctx_lens, scale)
    compare(o_na, l_na, ref_o, ref_l, f"{what}: against the oracle")


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_two_calls_in_a_row():
    build.build()
    scale = 1 / math.sqrt(128)
    # call 1: the paged-decode configuration (32 sequences, 32 heads, 256-token pages)
    first = inputs.decode_inputs(B=32, H=32, d=128, page_size=256, num_pages=1200, max_ctx=8192,
                                 dtype=torch.float16, seed=0)
    # call 2: other sequences, other lengths, other dtype; same shared scratch
    second = inputs.decode_inputs(B=16, H=32, d=128, page_size=256, num_pages=600, max_ctx=8192,
                                  dtype=torch.bfloat16, seed=1)
    for n, di in enumerate((first, second)):
        _check(di, scale, f"no-alloc call {n + 1}")


@pytest.mark.gpu
def test_noalloc_decode_at_the_scratch_limit():
    """B*H = 32263 sequence-heads at d = 128: one split per sequence needs
    32263 * 130 * 4 = 16,776,760 bytes, just under the 16 MiB scratch."""
    build.build()
    B, H, d = 4609, 7, 128
    assert B * H * (d + 2) * 4 <= SCRATCH < (B * H + 1) * (d + 2) * 4
    di = inputs.decode_inputs(B=B, H=H, d=d, page_size=16, num_pages=2 * B, max_ctx=32,
                              dtype=torch.float16, seed=3)
    assert fa.fa_decode_default_pages_per_split(B, H, di.block_table.shape[1]) == \
        di.block_table.shape[1]  # one split per sequence
    _check(di, 1 / math.sqrt(d), "no-alloc at the limit")


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    """One sequence-head more than the limit (B*H*(d+2)*4 bytes above 16 MiB), and a
    much larger case: refused on the host before anything is launched."""
    build.build()
    L = fa.lib()
    A = 0x10000  # aligned placeholder; the size check comes before any device access
    for B, H in ((4033, 8), (1024, 64)):
        assert B * H * 130 * 4 > SCRATCH
        rc = L.fa_decode_paged_noalloc(A, A, A, A, A, A, None, B, H, 128, 16, 2, 8, 0.1,
                                       fa.FA_F16, None)
        assert rc == fa.FA_ERR_INVALID_ARG
        assert "scratch" in fa.fa_last_error_string()
