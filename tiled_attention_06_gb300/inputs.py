"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both take their
inputs from it without sharing any of the method.

All draws use a CPU ``torch.Generator`` seeded explicitly, in a fixed order, so
that the same bytes can be handed to the GPU and to the oracle.
"""
from dataclasses import dataclass

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def prefill_inputs(B, H, Sq, Sk, d, dtype=torch.float16, factor=1.0, seed=0):
    """q [B,H,Sq,d], k and v [B,H,Sk,d]: i.i.d. N(0,1) * factor in float32, then cast.

    Draw order: q, k, v.
    """
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, H, Sq, d, generator=g) * factor).to(dtype)
    k = (torch.randn(B, H, Sk, d, generator=g) * factor).to(dtype)
    v = (torch.randn(B, H, Sk, d, generator=g) * factor).to(dtype)
    return q, k, v


def f32_resolution_inputs(B, H, Sq, Sk, d, seed=0):
    """float32 q, k ~ N(0,1) * 2 and v ~ 1 + N(0,1) / 4: with scale 1/8 and d = 64 the
    logits spread over about +-10, and V's values sit near 1, where bf16's step is 2^-7.

    Draw order: q, k, v.
    """
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, d, generator=g) * 2.0
    k = torch.randn(B, H, Sk, d, generator=g) * 2.0
    v = 1.0 + torch.randn(B, H, Sk, d, generator=g) / 4.0
    return q, k, v


def climbing_inputs(B, H, Sq, Sk, d, dtype=torch.float16, step=0.0, wide=1.0, v_scale=1.0,
                    seed=0):
    """q, k, v whose scores climb (step > 0) or fall (step < 0) along the key axis.

    q = N(0,1) * wide + 1 and k_j = N(0,1) * wide + a_j with a_j = step * j / d (step > 0)
    or step * (j - Sk + 1) / d (step < 0), every component of a row shifted alike; then
    q . k_j = |step| * j + (a zero-mean part), so the raw dot product rises by about |step|
    per key for ascending keys (falls for step < 0) whatever the query.
    v ~ N(0,1) * v_scale. With step = 0 and wide > 1 the scores are only wider
    (N(0, wide^4)-like). The values are drawn in float32 and cast to `dtype`.

    Draw order: q, k, v.
    """
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Sq, d, generator=g) * wide + (1.0 if step != 0 else 0.0)
    k = torch.randn(B, H, Sk, d, generator=g) * wide
    v = torch.randn(B, H, Sk, d, generator=g) * v_scale
    if step != 0:
        j = torch.arange(Sk, dtype=torch.float32)
        a = (step * j if step > 0 else step * (j - (Sk - 1))) / d
        k = k + a[:, None]
    return q.to(dtype), k.to(dtype), v.to(dtype)


@dataclass
class DecodeInputs:
    q: torch.Tensor            # [B,H,d]
    k_pages: torch.Tensor      # [num_pages,H,page_size,d]
    v_pages: torch.Tensor      # [num_pages,H,page_size,d]
    block_table: torch.Tensor  # int32 [B,max_pages_per_seq], unused entries -1
    ctx_lens: torch.Tensor     # int32 [B]
    page_size: int

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def H(self):
        return self.q.shape[1]

    @property
    def d(self):
        return self.q.shape[2]


def decode_inputs(B=32, H=32, d=128, page_size=256, num_pages=1200, max_ctx=8192,
                  dtype=torch.float16, seed=0, ctx_lens=None, poison=True):
    """A paged KV cache with randomly scattered pages.

    Draw order: ctx_lens ~ U{1..max_ctx} (unless given), perm = randperm(num_pages),
    q, then for every referenced page in table order (sequence b ascending, page
    index ascending) its K block [H,page_size,d] then its V block.
    Sequence b takes the next ceil(ctx_b / page_size) entries of perm.
    Unused table entries are -1. With poison=True, unreferenced pages and the
    slots past ctx_b in a sequence's last page hold NaN, so that any read of a
    token the query may not see shows up in the output.
    """
    g = torch.Generator().manual_seed(seed)
    max_pages = (max_ctx + page_size - 1) // page_size
    if ctx_lens is None:
        ctx = torch.randint(1, max_ctx + 1, (B,), generator=g, dtype=torch.int64)
    else:
        ctx = torch.as_tensor(ctx_lens, dtype=torch.int64).clone()
        if ctx.numel() != B or (B > 0 and (int(ctx.max()) > max_ctx or int(ctx.min()) < 0)):
            raise ValueError("ctx_lens must have B entries, each in [0, max_ctx]")
    perm = torch.randperm(num_pages, generator=g)
    npages = [(int(c) + page_size - 1) // page_size for c in ctx]
    if sum(npages) > num_pages:
        raise ValueError("the pool is too small for these context lengths")
    table = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(B):
        table[b, :npages[b]] = perm[off:off + npages[b]].to(torch.int32)
        off += npages[b]
    q = torch.randn(B, H, d, generator=g).to(dtype)
    fill = float("nan") if poison else 0.0
    kp = torch.full((num_pages, H, page_size, d), fill, dtype=dtype)
    vp = torch.full((num_pages, H, page_size, d), fill, dtype=dtype)
    for b in range(B):
        for p in range(npages[b]):
            pg = int(table[b, p])
            kp[pg] = torch.randn(H, page_size, d, generator=g).to(dtype)
            vp[pg] = torch.randn(H, page_size, d, generator=g).to(dtype)
        tail = int(ctx[b]) - (npages[b] - 1) * page_size
        if poison and npages[b] > 0 and tail < page_size:
            pg = int(table[b, npages[b] - 1])
            kp[pg, :, tail:, :] = float("nan")
            vp[pg, :, tail:, :] = float("nan")
    return DecodeInputs(q, kp, vp, table, ctx.to(torch.int32), page_size)


def block_layout(H, Sq, Sk, block=128, local=1, n_global=1, n_random=2, seed=0):
    """Seeded block-sparse layout uint8 [H, ceil(Sq/block), ceil(Sk/block)] with the
    BigBird shape: per head, block (i, j) is on when |i - j| <= local, when i or j is one
    of the first n_global blocks, or when j is one of n_random blocks drawn for row i."""
    nq, nk = -(-Sq // block), -(-Sk // block)
    g = torch.Generator().manual_seed(seed)
    i = torch.arange(nq)[:, None]
    j = torch.arange(nk)[None, :]
    base = ((i - j).abs() <= local) | (i < n_global) | (j < n_global)
    lay = base.expand(H, nq, nk).clone()
    if n_random > 0 and nk > 0:
        pick = torch.rand(H, nq, nk, generator=g).argsort(dim=-1)[..., :min(n_random, nk)]
        lay.scatter_(-1, pick, True)
    return lay.to(torch.uint8)
