"""FP64 CPU oracle for FlashAttention forward (TEST INFRASTRUCTURE ONLY).

Only the test suite, the smoke check and the benchmark's CPU-baseline / reference
legs may import this package. The product library never loads it.

Thin ctypes wrapper over oracle/liboracle.so (built from fa_oracle.c). Inputs are
CPU torch tensors in float16 / bfloat16 / float32 / float64; the C code decodes
their exact stored bits into doubles. Outputs are float64 numpy arrays.
"""
import ctypes
import os

import numpy as np
import torch

from . import build as _build

MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_WINDOW, MASK_BAND, MASK_PREFIX_LM = 0, 1, 2, 3, 4
TILE_EMPTY, TILE_PARTIAL, TILE_FULL = 0, 1, 2
REC_UNNORMALISED, REC_NORMALISED, REC_LITERAL_P2 = 0, 1, 2

_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2, torch.float64: 3}

_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_dp = ctypes.POINTER(ctypes.c_double)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.or_elem.restype = ctypes.c_double
        L.or_elem.argtypes = [_vp, _i64, ctypes.c_int]
        L.or_visible.restype = ctypes.c_int
        L.or_visible.argtypes = [_i64, _i64, _i64, _i64, ctypes.c_int, _i64, _i64]
        L.or_count_visible.restype = _i64
        L.or_count_visible.argtypes = [_i64, _i64, ctypes.c_int, _i64, _i64]
        L.or_tile_class.restype = ctypes.c_int
        L.or_tile_class.argtypes = [_i64] * 6 + [ctypes.c_int, _i64, _i64]
        L.or_attention.restype = ctypes.c_int
        L.or_attention.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _i64, _i64, _i64,
                                   _i64, _i64, ctypes.c_double, ctypes.c_int, _i64, _i64,
                                   _vp, _i64, _dp, ctypes.c_int]
        L.or_online_attention.restype = ctypes.c_int
        L.or_online_attention.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _i64, _i64,
                                          _i64, _i64, _i64, ctypes.c_double, ctypes.c_int,
                                          _i64, _i64, _i64, ctypes.c_double, ctypes.c_int]
        L.or_decode_paged.restype = ctypes.c_int
        L.or_decode_paged.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _i64,
                                      _i64, _i64, _i64, _i64, _i64, ctypes.c_double, _vp,
                                      _i64, ctypes.c_int]
        L.or_attention_paged.restype = ctypes.c_int
        L.or_attention_paged.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _i64,
                                         _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                                         ctypes.c_int, _i64, _i64, ctypes.c_int]
        L.or_combine_partials.restype = None
        L.or_combine_partials.argtypes = [_vp, _vp, _vp, _i64, _i64, _vp, _vp]
        L.or_attention_layout.restype = ctypes.c_int
        L.or_attention_layout.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _i64, _i64,
                                          _i64, _i64, _i64, ctypes.c_double, _vp, _i64, _vp,
                                          _i64, ctypes.c_int]
        L.or_count_visible_layout.restype = _i64
        L.or_count_visible_layout.argtypes = [_i64, _i64, _i64, _vp, _i64]
        L.or_tile_class_layout.restype = ctypes.c_int
        L.or_tile_class_layout.argtypes = [_i64] * 7 + [_vp, _i64]
        L.or_rescale_events.restype = ctypes.c_int
        L.or_rescale_events.argtypes = [_vp, _vp, ctypes.c_int] + [_i64] * 5 + [
            ctypes.c_double, ctypes.c_int, _i64, _i64, _vp, _i64, _i64, ctypes.c_double, _i64,
            ctypes.c_double, _vp, _vp, ctypes.c_int]
        L.or_attention_backward.restype = ctypes.c_int
        L.or_attention_backward.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp,
                                            _i64, _i64, _i64, _i64, _i64, ctypes.c_double,
                                            ctypes.c_int, _i64, _i64, ctypes.c_int]
        L.or_attention_backward_layout.restype = ctypes.c_int
        L.or_attention_backward_layout.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, _vp, _vp,
                                                   _vp, _i64, _i64, _i64, _i64, _i64,
                                                   ctypes.c_double, _vp, _i64, ctypes.c_int]
        L.or_decode_split_tokens.restype = None
        L.or_decode_split_tokens.argtypes = [_i64, _i64, _i64, _i64,
                                             ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
        _lib = L
    return _lib


def _cpu(t):
    t = t.detach()
    if t.device.type != "cpu":
        raise ValueError("oracle inputs must be CPU tensors")
    return t.contiguous()


def _dtype_code(*ts):
    codes = {_DT[t.dtype] for t in ts}
    if len(codes) != 1:
        raise ValueError("q, k, v must share one dtype")
    return codes.pop()


def elem_values(t):
    """Exact values of a tensor's stored elements, decoded by the oracle's C code."""
    t = _cpu(t)
    out = np.empty(t.numel(), dtype=np.float64)
    L = lib()
    code = _DT[t.dtype]
    for i in range(t.numel()):
        out[i] = L.or_elem(ctypes.c_void_p(t.data_ptr()), i, code)
    return out.reshape(tuple(t.shape))


def visible(i, j, Sq, Sk, mask_mode, window=0, n_global=0):
    return bool(lib().or_visible(i, j, Sq, Sk, mask_mode, window, n_global))


def count_visible(Sq, Sk, mask_mode, window=0, n_global=0):
    return int(lib().or_count_visible(Sq, Sk, mask_mode, window, n_global))


def tile_class(mb, nb, BM, BN, Sq, Sk, mask_mode, window=0, n_global=0):
    return int(lib().or_tile_class(mb, nb, BM, BN, Sq, Sk, mask_mode, window, n_global))


def attention(q, k, v, scale, mask_mode=MASK_NONE, window=0, n_global=0, rows=None,
              nthreads=0, return_psum_err=False):
    """q [B,H,Sq,d], k/v [B,H,Sk,d] -> (o float64, lse float64).

    rows: optional 1-D int array of flat row ids (b*H + h)*Sq + i; then o is
    [len(rows), d] and lse [len(rows)].
    """
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    if rows is None:
        o = np.zeros((B, H, Sq, d))
        lse = np.zeros((B, H, Sq))
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.zeros((rows.size, d))
        lse = np.zeros(rows.size)
        rp, nr = rows.ctypes.data, rows.size
    err = ctypes.c_double(0.0)
    rc = lib().or_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), _dtype_code(q, k, v),
                            o.ctypes.data, lse.ctypes.data, B, H, Sq, Sk, d, float(scale),
                            mask_mode, window, n_global, rp, nr, ctypes.byref(err), nthreads)
    if rc != 0:
        raise ValueError("or_attention rejected its arguments")
    if return_psum_err:
        return o, lse, err.value
    return o, lse


def online_attention(q, k, v, scale, mask_mode=MASK_NONE, window=0, n_global=0,
                     block_n=64, tau=0.0, variant=REC_UNNORMALISED):
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    o = np.zeros((B, H, Sq, d))
    lse = np.zeros((B, H, Sq))
    rc = lib().or_online_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   _dtype_code(q, k, v), o.ctypes.data, lse.ctypes.data, B, H,
                                   Sq, Sk, d, float(scale), mask_mode, window, n_global, block_n,
                                   float(tau), variant)
    if rc != 0:
        raise ValueError("or_online_attention rejected its arguments")
    return o, lse


def rescale_events(q, k, scale, block_n, tau, mask_mode=MASK_NONE, window=0, n_global=0,
                   layout=None, blk=128, tile_rows=128, eps=1e-3, nthreads=0):
    """Rescales of the lazy online recurrence (threshold tau in natural-log units, key
    blocks of block_n in ascending order), summed per tile of tile_rows query rows:
    (counts, near) int64 [B*H, ceil(Sq/tile_rows)], near = decisions within eps of the
    threshold. layout: block-sparse visibility instead of mask_mode."""
    q, k = _cpu(q), _cpu(k)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    nt = -(-Sq // tile_rows)
    counts = np.zeros((B * H, nt), dtype=np.int64)
    near = np.zeros((B * H, nt), dtype=np.int64)
    lay = None if layout is None else _layout(layout, H, Sq, Sk, blk)
    rc = lib().or_rescale_events(q.data_ptr(), k.data_ptr(), _dtype_code(q, k), B, H, Sq, Sk,
                                 d, float(scale), mask_mode, window, n_global,
                                 None if lay is None else lay.ctypes.data, blk, block_n,
                                 float(tau), tile_rows, float(eps), counts.ctypes.data,
                                 near.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("or_rescale_events rejected its arguments")
    return counts, near


def decode_paged(q, k_pages, v_pages, block_table, ctx_lens, scale, bh_list=None, nthreads=0):
    """q [B,H,d]; pools [P,H,page,d]; block_table int32 [B,max_pages]; ctx_lens int32 [B]."""
    q, k_pages, v_pages = _cpu(q), _cpu(k_pages), _cpu(v_pages)
    bt = _cpu(block_table).to(torch.int32)
    cl = _cpu(ctx_lens).to(torch.int32)
    B, H, d = q.shape
    P, _, page, _ = k_pages.shape
    if bh_list is None:
        o = np.zeros((B, H, d))
        lse = np.zeros((B, H))
        bp, nb = None, 0
    else:
        bh_list = np.ascontiguousarray(np.asarray(bh_list, dtype=np.int64))
        o = np.zeros((bh_list.size, d))
        lse = np.zeros(bh_list.size)
        bp, nb = bh_list.ctypes.data, bh_list.size
    rc = lib().or_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                               _dtype_code(q, k_pages, v_pages), bt.data_ptr(), cl.data_ptr(),
                               o.ctypes.data, lse.ctypes.data, B, H, d, page, bt.shape[1], P,
                               float(scale), bp, nb, nthreads)
    if rc != 0:
        raise ValueError("or_decode_paged rejected its arguments")
    return o, lse


def attention_paged(q, k_pages, v_pages, block_table, ctx_lens, scale, mask_mode=MASK_NONE,
                    window=0, n_global=0, nthreads=0):
    """q [B,H,Sq,d] (the last Sq tokens of each sequence); pools [P,H,page,d]."""
    q, k_pages, v_pages = _cpu(q), _cpu(k_pages), _cpu(v_pages)
    bt = _cpu(block_table).to(torch.int32)
    cl = _cpu(ctx_lens).to(torch.int32)
    B, H, Sq, d = q.shape
    P, _, page, _ = k_pages.shape
    o = np.zeros((B, H, Sq, d))
    lse = np.zeros((B, H, Sq))
    rc = lib().or_attention_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                  _dtype_code(q, k_pages, v_pages), bt.data_ptr(), cl.data_ptr(),
                                  o.ctypes.data, lse.ctypes.data, B, H, Sq, d, page, bt.shape[1],
                                  P, float(scale), mask_mode, window, n_global, nthreads)
    if rc != 0:
        raise ValueError("or_attention_paged rejected its arguments")
    return o, lse


def combine_partials(m, l, acc):
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    ns, d = acc.shape
    o = np.zeros(d)
    lse = np.zeros(1)
    lib().or_combine_partials(m.ctypes.data, l.ctypes.data, acc.ctypes.data, ns, d,
                              o.ctypes.data, lse.ctypes.data)
    return o, float(lse[0])


def decode_split_tokens(ctx_len, page_size, pages_per_split, split):
    a, b = _i64(0), _i64(0)
    lib().or_decode_split_tokens(ctx_len, page_size, pages_per_split, split,
                                 ctypes.byref(a), ctypes.byref(b))
    return int(a.value), int(b.value)


def threads_used(nthreads=0):
    """How many OpenMP threads the oracle will use when nthreads <= 0."""
    if nthreads > 0:
        return nthreads
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def _layout(layout, H, Sq, Sk, blk):
    lay = np.ascontiguousarray(np.asarray(layout, dtype=np.uint8))
    want = (H, -(-Sq // blk), -(-Sk // blk))
    if lay.shape != want:
        raise ValueError(f"layout shape {lay.shape}, want {want}")
    return lay


def attention_layout(q, k, v, scale, layout, blk=128, rows=None, nthreads=0):
    """Block-sparse attention: query i of head h sees key j iff
    layout[h, i // blk, j // blk] != 0 (layout uint8 [H, ceil(Sq/blk), ceil(Sk/blk)], the
    same for every batch entry). Returns (o, lse) as attention()."""
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    lay = _layout(layout, H, Sq, Sk, blk)
    if rows is None:
        o = np.zeros((B, H, Sq, d))
        lse = np.zeros((B, H, Sq))
        rp, nr = None, 0
    else:
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        o = np.zeros((rows.size, d))
        lse = np.zeros(rows.size)
        rp, nr = rows.ctypes.data, rows.size
    rc = lib().or_attention_layout(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   _dtype_code(q, k, v), o.ctypes.data, lse.ctypes.data, B, H,
                                   Sq, Sk, d, float(scale), lay.ctypes.data, blk, rp, nr,
                                   nthreads)
    if rc != 0:
        raise ValueError("or_attention_layout rejected its arguments")
    return o, lse


def count_visible_layout(H, Sq, Sk, layout, blk=128):
    lay = _layout(layout, H, Sq, Sk, blk)
    return int(lib().or_count_visible_layout(H, Sq, Sk, lay.ctypes.data, blk))


def tile_class_layout(h, mb, nb, BM, BN, Sq, Sk, layout, blk=128):
    lay = _layout(layout, layout.shape[0], Sq, Sk, blk)
    return int(lib().or_tile_class_layout(h, mb, nb, BM, BN, Sq, Sk, lay.ctypes.data, blk))


def attention_backward_layout(q, k, v, dout, scale, layout, blk=128, nthreads=0):
    """Gradients (dq, dk, dv) in float64 of block-sparse attention (layout as in
    attention_layout) for the upstream gradient dout."""
    q, k, v, dout = _cpu(q), _cpu(k), _cpu(v), _cpu(dout)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    lay = _layout(layout, H, Sq, Sk, blk)
    dq = np.zeros((B, H, Sq, d))
    dk = np.zeros((B, H, Sk, d))
    dv = np.zeros((B, H, Sk, d))
    rc = lib().or_attention_backward_layout(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            dout.data_ptr(), _dtype_code(q, k, v, dout),
                                            dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, B, H,
                                            Sq, Sk, d, float(scale), lay.ctypes.data, blk,
                                            nthreads)
    if rc != 0:
        raise ValueError("or_attention_backward_layout rejected its arguments")
    return dq, dk, dv


def attention_backward(q, k, v, dout, scale, mask_mode=MASK_NONE, window=0, n_global=0,
                       nthreads=0):
    """Gradients (dq, dk, dv) in float64 of attention for the upstream gradient dout."""
    q, k, v, dout = _cpu(q), _cpu(k), _cpu(v), _cpu(dout)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    dq = np.zeros((B, H, Sq, d))
    dk = np.zeros((B, H, Sk, d))
    dv = np.zeros((B, H, Sk, d))
    rc = lib().or_attention_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                     _dtype_code(q, k, v, dout), dq.ctypes.data, dk.ctypes.data,
                                     dv.ctypes.data, B, H, Sq, Sk, d, float(scale), mask_mode,
                                     window, n_global, nthreads)
    if rc != 0:
        raise ValueError("or_attention_backward rejected its arguments")
    return dq, dk, dv
