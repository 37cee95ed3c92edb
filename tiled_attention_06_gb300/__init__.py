"""FlashAttention forward (prefill + paged decode) for one NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C-ABI library ``libfa.so`` (declared in
``include/fa.h``). The functions keep the C names; they only marshal torch
tensors into pointers, sizes and the current CUDA stream. Every step of the
computation runs in the library's CUDA kernels: there is no fallback, and a
missing library raises ``FaError``.
"""
import ctypes
import os

import torch

__all__ = [
    "FaError", "lib", "fa_fwd", "fa_fwd_ex", "fa_decode_paged", "fa_decode_paged_ex",
    "fa_decode_paged_noalloc", "fa_merge_partials", "fa_fwd_paged", "fa_fwd_paged_host_lens",
    "fa_kv_append",
    "fa_decode_workspace_size", "fa_decode_default_pages_per_split",
    "fa_get_device_status",
    "fa_selftest_timeout", "fa_last_error_string", "fa_version", "fa_fwd_block_m",
    "fa_fwd_default_block_m", "fa_bwd", "fa_bwd_block_sparse", "fa_bwd_workspace_size", "fa_fwd_workspace_size",
    "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
    "FA_ERR_BAD_PAGE", "FA_F16", "FA_BF16", "FA_F32", "FA_MASK_NONE", "FA_MASK_CAUSAL",
    "FA_MASK_CAUSAL_WINDOW", "FA_MASK_BAND", "FA_MASK_PREFIX_LM", "FA_MASK_BLOCK_SPARSE",
    "FA_LAYOUT_BLOCK",
]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_BAD_PAGE = range(6)
FA_F16, FA_BF16, FA_F32 = 0, 1, 2
FA_MASK_NONE, FA_MASK_CAUSAL, FA_MASK_CAUSAL_WINDOW, FA_MASK_BAND, FA_MASK_PREFIX_LM = 0, 1, 2, 3, 4
FA_MASK_BLOCK_SPARSE = 5
FA_LAYOUT_BLOCK = 128

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_u32 = ctypes.c_uint32
_sz = ctypes.c_size_t


class FaError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"fa status {status}: {msg}")
        self.status = status


class FwdParams(ctypes.Structure):
    _fields_ = [("q", _vp), ("k", _vp), ("v", _vp), ("o", _vp), ("lse", _vp),
                ("B", _i), ("H", _i), ("Sq", _i), ("Sk", _i), ("d", _i), ("scale", _f),
                ("mask_mode", _i), ("window", _i), ("n_global", _i), ("dtype", _i),
                ("block_n", _i), ("block_m", _i), ("num_ctas", _i), ("group_heads", _i),
                ("timeout_us", _u32),
                ("trace", _vp), ("block_layout", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("rescale_count", _vp), ("block_layout_host", _vp)]


class DecodeParams(ctypes.Structure):
    _fields_ = [("q", _vp), ("k_pages", _vp), ("v_pages", _vp), ("block_table", _vp),
                ("ctx_lens", _vp), ("o", _vp), ("lse", _vp), ("B", _i), ("H", _i), ("d", _i),
                ("page_size", _i), ("max_pages_per_seq", _i), ("num_pages", _i), ("scale", _f),
                ("dtype", _i), ("workspace", _vp), ("workspace_bytes", _sz),
                ("pages_per_split", _i), ("trace_pages", _vp), ("trace_splits", _vp)]


_lib = None


def lib():
    """The loaded libfa.so (raises FaError when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise FaError(FA_ERR_CUDA, f"{LIB_PATH} is missing: build it with "
                          "tiled_attention_06_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        L.fa_fwd.restype = _i
        L.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _i, _i, _i, _vp]
        L.fa_fwd_ex.restype = _i
        L.fa_fwd_ex.argtypes = [ctypes.POINTER(FwdParams), _vp]
        L.fa_fwd_block_m.restype = _i
        L.fa_fwd_block_m.argtypes = []
        L.fa_fwd_default_block_m.restype = _i
        L.fa_fwd_default_block_m.argtypes = [_i]
        L.fa_fwd_workspace_size.restype = _sz
        L.fa_fwd_workspace_size.argtypes = [_i] * 6
        L.fa_bwd_workspace_size.restype = _sz
        L.fa_bwd_workspace_size.argtypes = [_i, _i, _i]
        L.fa_bwd.restype = _i
        L.fa_bwd.argtypes = [_vp] * 10 + [_sz] + [_i] * 5 + [_f] + [_i] * 4 + [_vp]
        L.fa_bwd_block_sparse.restype = _i
        L.fa_bwd_block_sparse.argtypes = [_vp] * 10 + [_sz] + [_i] * 5 + [_f, _vp, _i, _vp]
        L.fa_decode_paged.restype = _i
        L.fa_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i,
                                      _f, _i, _vp, _sz, _vp]
        L.fa_decode_paged_ex.restype = _i
        L.fa_decode_paged_ex.argtypes = [ctypes.POINTER(DecodeParams), _vp]
        L.fa_decode_paged_noalloc.restype = _i
        L.fa_decode_paged_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i,
                                              _i, _i, _f, _i, _vp]
        L.fa_fwd_paged.restype = _i
        L.fa_fwd_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                   _f, _i, _i, _i, _i, _vp]
        L.fa_fwd_paged_host_lens.restype = _i
        L.fa_fwd_paged_host_lens.argtypes = [_vp] * 8 + [_i] * 7 + [_f] + [_i] * 4 + [_vp]
        L.fa_kv_append.restype = _i
        L.fa_kv_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                   _i, _vp]
        L.fa_merge_partials.restype = _i
        L.fa_merge_partials.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _i, _i, _vp]
        L.fa_decode_workspace_size.restype = _sz
        L.fa_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i]
        L.fa_decode_default_pages_per_split.restype = _i
        L.fa_decode_default_pages_per_split.argtypes = [_i, _i, _i]
        L.fa_get_device_status.restype = _i
        L.fa_get_device_status.argtypes = [_vp]
        L.fa_selftest_timeout.restype = _i
        L.fa_selftest_timeout.argtypes = [_u32, _vp]
        L.fa_last_error_string.restype = ctypes.c_char_p
        L.fa_last_error_string.argtypes = []
        L.fa_version.restype = _i
        L.fa_version.argtypes = []
        _lib = L
    return _lib


def _check(status):
    if status != FA_OK:
        raise FaError(status, fa_last_error_string())


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dtype_code(t):
    if t.dtype == torch.float16:
        return FA_F16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float32:  # fa_fwd / fa_fwd_ex only; the other calls refuse it
        return FA_F32
    raise FaError(FA_ERR_UNSUPPORTED, f"dtype {t.dtype} (float16, bfloat16 or float32)")


def _need_cuda_contig(**ts):
    for name, t in ts.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be contiguous")


def fa_last_error_string():
    return lib().fa_last_error_string().decode()


def fa_version():
    return lib().fa_version()


def fa_fwd_block_m():
    return lib().fa_fwd_block_m()


def fa_fwd_default_block_m(mask_mode):
    return lib().fa_fwd_default_block_m(mask_mode)


def fa_fwd_workspace_size(B, H, Sq, Sk, d, dtype):
    return lib().fa_fwd_workspace_size(B, H, Sq, Sk, d, dtype)


def fa_bwd_workspace_size(B, H, Sq):
    return lib().fa_bwd_workspace_size(B, H, Sq)


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, mask_mode=FA_MASK_NONE,
           window=0, n_global=0, stream=None, block_layout=None):
    """Gradients dq, dk, dv of fa_fwd for the upstream gradient dout (all [B,H,S,d]
    CUDA tensors of one 16-bit dtype; lse the float32 [B,H,Sq] fa_fwd returned; workspace
    a CUDA byte tensor of fa_bwd_workspace_size(B, H, Sq) bytes). FA_MASK_BLOCK_SPARSE takes
    block_layout, the uint8 CUDA layout of the forward call (fa_bwd_block_sparse)."""
    _need_cuda_contig(q=q, k=k, v=v, o=o, dout=dout, lse=lse, dq=dq, dk=dk, dv=dv,
                      workspace=workspace, block_layout=block_layout)
    B, H, Sq, d = q.shape
    if mask_mode == FA_MASK_BLOCK_SPARSE:
        _check(lib().fa_bwd_block_sparse(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), B, H, Sq, k.shape[2], d, float(scale),
            _ptr(block_layout), _dtype_code(q), _stream(stream)))
        return
    _check(lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                        lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(), B,
                        H, Sq, k.shape[2], d, float(scale), mask_mode, window, n_global,
                        _dtype_code(q), _stream(stream)))


def fa_bwd_block_sparse(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, block_layout,
                        stream=None):
    """fa_bwd under FA_MASK_BLOCK_SPARSE with the forward call's device layout."""
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, scale, FA_MASK_BLOCK_SPARSE,
           stream=stream, block_layout=block_layout)


def fa_fwd(q, k, v, o, lse, scale, mask_mode=FA_MASK_NONE, window=0, n_global=0, stream=None):
    """O = softmax(scale Q K^T + mask) V into `o` (and LSE into `lse`, may be None).

    q [B,H,Sq,d], k/v [B,H,Sk,d], o like q, lse float32 [B,H,Sq]; CUDA, contiguous.
    float32 inputs go through fa_fwd_ex, which needs a workspace (allocated here).
    """
    if q.dtype == torch.float32:
        return fa_fwd_ex(q, k, v, o, lse, scale, mask_mode, window, n_global, stream=stream)
    _need_cuda_contig(q=q, k=k, v=v, o=o, lse=lse)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    _check(lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _ptr(lse), B, H,
                        Sq, Sk, d, float(scale), mask_mode, window, n_global, _dtype_code(q),
                        _stream(stream)))


def fa_fwd_ex(q, k, v, o, lse, scale, mask_mode=FA_MASK_NONE, window=0, n_global=0,
              block_n=0, block_m=0, num_ctas=0, group_heads=0, timeout_us=0, trace=None,
              block_layout=None, workspace=None, rescale_count=None, stream=None,
              block_layout_host=None):
    """fa_fwd with the tuning and debug fields of fa_fwd_params. block_layout: uint8 CUDA
    tensor [H, ceil(Sq/128), ceil(Sk/128)] for FA_MASK_BLOCK_SPARSE; block_layout_host:
    the same layout as a contiguous CPU uint8 tensor, for the work plan. workspace: CUDA byte
    tensor of fa_fwd_workspace_size(...) bytes for float32 inputs (allocated here when
    None). rescale_count: zeroed int32 CUDA tensor [B*H, ceil(Sq/128)] that counts the
    rows whose output was rescaled, per 128-query tile."""
    _need_cuda_contig(q=q, k=k, v=v, o=o, lse=lse, trace=trace, block_layout=block_layout,
                      workspace=workspace, rescale_count=rescale_count)
    B, H, Sq, d = q.shape
    dt = _dtype_code(q)
    if workspace is None and dt == FA_F32:
        workspace = torch.empty(max(fa_fwd_workspace_size(B, H, Sq, k.shape[2], d, dt), 16),
                                dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if block_layout_host is not None:
        want = (H, -(-Sq // 128), -(-k.shape[2] // 128))
        if (block_layout_host.device.type != "cpu" or block_layout_host.dtype != torch.uint8
                or not block_layout_host.is_contiguous()
                or tuple(block_layout_host.shape) != want):
            raise ValueError(f"block_layout_host must be a contiguous CPU uint8 tensor {want}")
    p = FwdParams(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), _ptr(lse), B, H, Sq,
                  k.shape[2], d, float(scale), mask_mode, window, n_global, dt,
                  block_n, block_m, num_ctas, group_heads, timeout_us, _ptr(trace),
                  _ptr(block_layout), _ptr(workspace), ws_bytes, _ptr(rescale_count),
                  None if block_layout_host is None else block_layout_host.data_ptr())
    _check(lib().fa_fwd_ex(ctypes.byref(p), _stream(stream)))


def fa_decode_workspace_size(B, H, d, max_pages_per_seq, page_size):
    return lib().fa_decode_workspace_size(B, H, d, max_pages_per_seq, page_size)


def fa_decode_default_pages_per_split(B, H, max_pages_per_seq):
    return lib().fa_decode_default_pages_per_split(B, H, max_pages_per_seq)


def fa_decode_paged(q, k_pages, v_pages, block_table, ctx_lens, o, lse, scale, workspace,
                    stream=None):
    """One query token per sequence against a paged KV cache.

    q/o [B,H,d]; pools [num_pages,H,page_size,d]; block_table int32 [B,max_pages];
    ctx_lens int32 [B]; lse float32 [B,H] or None; workspace a CUDA byte tensor.
    """
    _need_cuda_contig(q=q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                      ctx_lens=ctx_lens, o=o, lse=lse, workspace=workspace)
    B, H, d = q.shape
    P, _, page, _ = k_pages.shape
    _check(lib().fa_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                 block_table.data_ptr(), ctx_lens.data_ptr(), o.data_ptr(),
                                 _ptr(lse), B, H, d, page, block_table.shape[1], P, float(scale),
                                 _dtype_code(q), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def fa_decode_paged_ex(q, k_pages, v_pages, block_table, ctx_lens, o, lse, scale, workspace,
                       pages_per_split=0, trace_pages=None, trace_splits=None, stream=None):
    _need_cuda_contig(q=q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                      ctx_lens=ctx_lens, o=o, lse=lse, workspace=workspace,
                      trace_pages=trace_pages, trace_splits=trace_splits)
    B, H, d = q.shape
    P, _, page, _ = k_pages.shape
    p = DecodeParams(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                     ctx_lens.data_ptr(), o.data_ptr(), _ptr(lse), B, H, d, page,
                     block_table.shape[1], P, float(scale), _dtype_code(q), workspace.data_ptr(),
                     workspace.numel() * workspace.element_size(), pages_per_split,
                     _ptr(trace_pages), _ptr(trace_splits))
    _check(lib().fa_decode_paged_ex(ctypes.byref(p), _stream(stream)))


def fa_decode_paged_noalloc(q, k_pages, v_pages, block_table, ctx_lens, o, lse, scale,
                            stream=None):
    """fa_decode_paged for callers that cannot allocate a workspace: the split partials
    go to a fixed 16 MiB scratch array inside the library (one per GPU). Calls that
    overlap on the GPU share that array and race; the first call on a device should
    come before any stream capture."""
    _need_cuda_contig(q=q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                      ctx_lens=ctx_lens, o=o, lse=lse)
    B, H, d = q.shape
    P, _, page, _ = k_pages.shape
    _check(lib().fa_decode_paged_noalloc(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                         block_table.data_ptr(), ctx_lens.data_ptr(),
                                         o.data_ptr(), _ptr(lse), B, H, d, page,
                                         block_table.shape[1], P, float(scale), _dtype_code(q),
                                         _stream(stream)))


def fa_fwd_paged(q, k_pages, v_pages, block_table, ctx_lens, o, lse, scale,
                 mask_mode=FA_MASK_CAUSAL, window=0, n_global=0, stream=None,
                 ctx_lens_host=None):
    """Chunked prefill against a paged cache: q/o [B,H,Sq,d] are the last Sq tokens of
    each sequence; pools [num_pages,H,page,d]; block_table int32 [B,max_pages];
    ctx_lens int32 [B] (cached tokens, the chunk included). ctx_lens_host: the same
    lengths as a CPU int32 tensor, for the work plan (fa_fwd_paged_host_lens)."""
    _need_cuda_contig(q=q, k_pages=k_pages, v_pages=v_pages, block_table=block_table,
                      ctx_lens=ctx_lens, o=o, lse=lse)
    B, H, Sq, d = q.shape
    P, _, page, _ = k_pages.shape
    if ctx_lens_host is None:
        _check(lib().fa_fwd_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                  block_table.data_ptr(), ctx_lens.data_ptr(), o.data_ptr(),
                                  _ptr(lse), B, H, Sq, d, page, block_table.shape[1], P,
                                  float(scale), mask_mode, window, n_global, _dtype_code(q),
                                  _stream(stream)))
        return
    if (ctx_lens_host.device.type != "cpu" or ctx_lens_host.dtype != torch.int32
            or not ctx_lens_host.is_contiguous() or ctx_lens_host.numel() != B):
        raise ValueError("ctx_lens_host must be a contiguous CPU int32 tensor of B entries")
    _check(lib().fa_fwd_paged_host_lens(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                        block_table.data_ptr(), ctx_lens.data_ptr(),
                                        ctx_lens_host.data_ptr(), o.data_ptr(), _ptr(lse), B, H,
                                        Sq, d, page, block_table.shape[1], P, float(scale),
                                        mask_mode, window, n_global, _dtype_code(q),
                                        _stream(stream)))


def fa_fwd_paged_host_lens(q, k_pages, v_pages, block_table, ctx_lens, ctx_lens_host, o, lse,
                           scale, mask_mode=FA_MASK_CAUSAL, window=0, n_global=0, stream=None):
    """fa_fwd_paged with the lengths also in host memory (a CPU int32 tensor) for the plan."""
    fa_fwd_paged(q, k_pages, v_pages, block_table, ctx_lens, o, lse, scale, mask_mode, window,
                 n_global, stream, ctx_lens_host=ctx_lens_host)


def fa_kv_append(k_new, v_new, k_pages, v_pages, block_table, ctx_lens, new_lens=None,
                 stream=None):
    """Write k_new/v_new [B,H,T,d] at positions ctx_lens[b] + t of the paged cache
    (t < new_lens[b], or all T); zero-fill the rest of each chunk's last page."""
    _need_cuda_contig(k_new=k_new, v_new=v_new, k_pages=k_pages, v_pages=v_pages,
                      block_table=block_table, ctx_lens=ctx_lens, new_lens=new_lens)
    B, H, T, d = k_new.shape
    P, _, page, _ = k_pages.shape
    _check(lib().fa_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_pages.data_ptr(),
                              v_pages.data_ptr(), block_table.data_ptr(), ctx_lens.data_ptr(),
                              _ptr(new_lens), B, H, T, d, page, block_table.shape[1], P,
                              _dtype_code(k_new), _stream(stream)))


def fa_merge_partials(o_a, lse_a, o_b, lse_b, o, lse=None, stream=None):
    """Combine two attention results over disjoint key sets of the same queries by LSE.

    o_* [..., d] (same shape, fp16/bf16), lse_* float32 with the leading shape of o.
    """
    _need_cuda_contig(o_a=o_a, lse_a=lse_a, o_b=o_b, lse_b=lse_b, o=o, lse=lse)
    d = o_a.shape[-1]
    rows = o_a.numel() // d
    _check(lib().fa_merge_partials(o_a.data_ptr(), lse_a.data_ptr(), o_b.data_ptr(),
                                   lse_b.data_ptr(), o.data_ptr(), _ptr(lse), rows, d,
                                   _dtype_code(o_a), _stream(stream)))


def fa_get_device_status(stream=None):
    """Synchronise the stream, read and clear the device status word; returns the code."""
    return lib().fa_get_device_status(_stream(stream))


def fa_selftest_timeout(timeout_us, stream=None):
    _check(lib().fa_selftest_timeout(timeout_us, _stream(stream)))
