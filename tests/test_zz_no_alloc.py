"""fa_decode_paged_noalloc: paged decode for callers that cannot allocate device memory.

Some users of this library cannot hand it a workspace: their device memory is fixed
when they start (a serving loop with a set budget), or a host program owns every
device allocation and gives its plug-ins no allocator. This entry point keeps the
decode's split partials in a scratch array built into the library instead. These
tests check, through the C ABI, that it gives the same results as fa_decode_paged
with a caller workspace on two calls in a row (the second call reuses whatever the
first left in the shared array), and that it refuses sizes its scratch cannot hold.
"""
import math

import pytest
import torch

import tiled_attention_06_gb300 as fa
from tiled_attention_06_gb300 import build, inputs

from _util import compare


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
        o_ws, l_ws, o_na, l_na = _run_both(di, scale)
        compare(o_na, l_na, o_ws.double().cpu().numpy(), l_ws.double().cpu().numpy(),
                f"no-alloc call {n + 1}")


def test_noalloc_decode_rejects_sizes_beyond_its_scratch():
    """B*H*(d+2)*4 bytes of partials (one split per sequence) above 16 MiB: refused on
    the host before anything is launched."""
    build.build()
    L = fa.lib()
    A = 0x10000  # aligned placeholder; the size check comes before any device access
    rc = L.fa_decode_paged_noalloc(A, A, A, A, A, A, None, 1024, 64, 128, 256, 4, 8, 0.1,
                                   fa.FA_F16, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    assert "scratch" in fa.fa_last_error_string()
