"""ctypes binding of libattn_gqa.so (declared in include/attn_gqa.h).

Argument marshalling only: each function takes CUDA tensors (or raw device
addresses as ints) and passes their addresses, sizes and the CUDA stream to
the C entry point of the same name.  Every step of the computation runs in
the library's CUDA kernels; there is no fallback.  If the library has not
been built, loading fails with an error that says so.
"""
import ctypes
import os

ATTN_CAUSAL, ATTN_FULL, ATTN_CROSS = 0, 1, 2
ATTN_FP32, ATTN_TF32, ATTN_BF16 = 0, 1, 2
ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = 0, 1, 2, 3, 4

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_gqa.so")

_lib = None
_u32 = ctypes.c_uint32
_vp = ctypes.c_void_p


class AttnError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, attn_status_string(code), code))


def load_library(path=None):
    """Load libattn_gqa.so (once).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError("libattn_gqa.so is not built (%s): run "
                           "`python -m attention_gqa_online_gb300.build`" % p)
    lib = ctypes.CDLL(p)
    lib.attn_forward.restype = ctypes.c_int
    lib.attn_forward.argtypes = [_vp, _vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _u32,
                                 ctypes.c_int, ctypes.c_int, _vp]
    lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_decode_workspace_bytes.argtypes = [_u32, _u32, _u32, _u32]
    lib.attn_decode_cached.restype = ctypes.c_int
    lib.attn_decode_cached.argtypes = [_vp, _vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32,
                                       _vp, ctypes.c_size_t, _vp]
    lib.attn_prefill.restype = ctypes.c_int
    lib.attn_prefill.argtypes = [_vp, _vp, _vp, _vp] + [_u32] * 6 + [ctypes.c_float] + \
        [_u32] * 4 + [ctypes.c_int, _vp]
    lib.attn_forward_window.restype = ctypes.c_int
    lib.attn_forward_window.argtypes = lib.attn_forward.argtypes[:-1] + [_u32, _vp]
    lib.attn_decode_cached_window.restype = ctypes.c_int
    lib.attn_decode_cached_window.argtypes = lib.attn_decode_cached.argtypes[:-1] + [_u32, _vp]
    lib.attn_prefill_window.restype = ctypes.c_int
    lib.attn_prefill_window.argtypes = lib.attn_prefill.argtypes[:-1] + [_u32, _vp]
    lib.attn_decode_append.restype = ctypes.c_int
    lib.attn_decode_append.argtypes = [_vp] * 7 + [_u32] * 4 + [_vp, ctypes.c_size_t, _vp]
    lib.attn_decode_paged.restype = ctypes.c_int
    lib.attn_decode_paged.argtypes = [_vp] * 6 + [_u32] * 6 + [_vp, ctypes.c_size_t, _u32, _vp]
    lib.attn_prefill_paged.restype = ctypes.c_int
    lib.attn_prefill_paged.argtypes = [_vp] * 5 + [_u32] * 8 + [ctypes.c_float] + [_u32] * 4 + \
        [ctypes.c_int, _u32, _vp]
    lib.attn_rope_table.restype = ctypes.c_int
    lib.attn_rope_table.argtypes = [_vp, _u32, _u32, ctypes.c_double, _vp]
    lib.attn_forward_rope.restype = ctypes.c_int
    lib.attn_forward_rope.argtypes = [_vp] * 5 + [_u32] * 5 + [ctypes.c_int, ctypes.c_int, _u32, _vp, _u32, _vp]
    lib.attn_backward.restype = ctypes.c_int
    lib.attn_backward.argtypes = [_vp] * 9 + [_u32] * 5 + [ctypes.c_int, ctypes.c_int, _u32, _vp]
    lib.attn_backward_rope.restype = ctypes.c_int
    lib.attn_backward_rope.argtypes = [_vp] * 9 + [_u32] * 5 + [ctypes.c_int, ctypes.c_int, _u32, _vp, _u32, _vp]
    lib.attn_get_status.restype = ctypes.c_int
    lib.attn_get_status.argtypes = [_vp]
    lib.attn_set_workspace.restype = ctypes.c_int
    lib.attn_set_workspace.argtypes = [_vp, ctypes.c_size_t]
    lib.attn_forward_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_forward_workspace_bytes.argtypes = [_u32] * 5 + [ctypes.c_int, ctypes.c_int, _u32, ctypes.c_int]
    lib.attn_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_prefill_workspace_bytes.argtypes = [_u32] * 8 + [ctypes.c_int, _u32]
    lib.attn_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.attn_backward_workspace_bytes.argtypes = [_u32] * 5 + [ctypes.c_int, ctypes.c_int]
    lib.attn_scratch_reserved_bytes.restype = ctypes.c_size_t
    lib.attn_scratch_reserved_bytes.argtypes = []
    lib.attn_scratch_peak_bytes.restype = ctypes.c_size_t
    lib.attn_scratch_peak_bytes.argtypes = [ctypes.c_int]
    lib.attn_release_scratch.restype = ctypes.c_int
    lib.attn_release_scratch.argtypes = []
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_status_string.argtypes = [ctypes.c_int]
    _lib = lib
    return lib


def _addr(x, name, dtype=None, host_ok=False):
    """Device address of a tensor (checked to be CUDA and of `dtype`), an int, or None.
    With host_ok, a pinned host tensor is accepted too (its address is valid on
    the device under unified addressing)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch
    if not isinstance(x, torch.Tensor):
        raise TypeError("%s must be a CUDA tensor, a device address or None" % name)
    if not x.is_cuda and not (host_ok and x.is_pinned()):
        raise ValueError("%s must be in device memory%s" % (name, " or pinned host memory" if host_ok else ""))
    if dtype is not None and x.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, x.dtype))
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, where):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _f32():
    import torch
    return torch.float32


def attn_forward(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                 prec=ATTN_FP32, stream=None):
    """Self / cross attention forward with per-row (max, log-sum); see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_forward(
        _addr(q, "q", f), _addr(k, "k", f), _addr(v, "v", f), _addr(out, "out", f), _addr(lse, "lse", f),
        q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, _stream(stream)), "attn_forward")


def attn_forward_window(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec,
                        window, stream=None):
    """attn_forward restricted to each row's last `window` keys (0 = all); see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_forward_window(
        _addr(q, "q", f), _addr(k, "k", f), _addr(v, "v", f), _addr(out, "out", f), _addr(lse, "lse", f),
        q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, window, _stream(stream)),
        "attn_forward_window")


def attn_backward(q, k, v, out, dout, lse, dq, dk, dv, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                  prec=ATTN_FP32, window=0, stream=None):
    """Gradients of the forward's out for upstream dout (out and lse from the forward); see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_backward(
        _addr(q, "q", f), _addr(k, "k", f), _addr(v, "v", f), _addr(out, "out", f), _addr(dout, "dout", f),
        _addr(lse, "lse", f), _addr(dq, "dq", f), _addr(dk, "dk", f), _addr(dv, "dv", f), q_seq, kv_seq,
        num_heads, num_kv_heads, head_dim, mask, prec, window, _stream(stream)), "attn_backward")


def attn_rope_table(table, max_pos, head_dim, base=10000.0, stream=None):
    """Fill a device [max_pos, head_dim] fp32 RoPE table (cos | sin per position); see attn_gqa.h."""
    _check(load_library().attn_rope_table(_addr(table, "table", _f32()), max_pos, head_dim, float(base),
                                          _stream(stream)), "attn_rope_table")


def attn_forward_rope(q, k, v, out, lse, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, window,
                      rope_table, table_rows=None, stream=None):
    """attn_forward_window with RoPE on q and k (table from attn_rope_table); see attn_gqa.h."""
    f = _f32()
    if table_rows is None:
        table_rows = rope_table.shape[0]
    _check(load_library().attn_forward_rope(
        _addr(q, "q", f), _addr(k, "k", f), _addr(v, "v", f), _addr(out, "out", f), _addr(lse, "lse", f),
        q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, window, _addr(rope_table, "rope_table", f),
        table_rows, _stream(stream)), "attn_forward_rope")


def attn_backward_rope(q, k, v, out, dout, lse, dq, dk, dv, q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                       prec, window, rope_table, table_rows=None, stream=None):
    """Backward of attn_forward_rope (gradients for the unturned q, k); see attn_gqa.h."""
    f = _f32()
    if table_rows is None:
        table_rows = rope_table.shape[0]
    _check(load_library().attn_backward_rope(
        _addr(q, "q", f), _addr(k, "k", f), _addr(v, "v", f), _addr(out, "out", f), _addr(dout, "dout", f),
        _addr(lse, "lse", f), _addr(dq, "dq", f), _addr(dk, "dk", f), _addr(dv, "dv", f), q_seq, kv_seq,
        num_heads, num_kv_heads, head_dim, mask, prec, window, _addr(rope_table, "rope_table", f), table_rows,
        _stream(stream)), "attn_backward_rope")


def attn_decode_workspace_bytes(num_heads, num_kv_heads, head_dim, max_seq):
    return int(load_library().attn_decode_workspace_bytes(num_heads, num_kv_heads, head_dim, max_seq))


def attn_decode_cached(q, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim, max_seq,
                       workspace, workspace_bytes=None, stream=None):
    """Cached single-token decode over positions 0..*kv_pos_dev; see attn_gqa.h."""
    f = _f32()
    if hasattr(kv_pos_dev, "element_size") and kv_pos_dev.element_size() != 4:
        raise ValueError("kv_pos_dev must hold one 32-bit unsigned position")
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().attn_decode_cached(
        _addr(q, "q", f, True), _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f),
        _addr(kv_pos_dev, "kv_pos_dev", None, True),
        _addr(out, "out", f, True), num_heads, num_kv_heads, head_dim, max_seq,
        _addr(workspace, "workspace"), workspace_bytes, _stream(stream)), "attn_decode_cached")


def attn_decode_cached_window(q, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim, max_seq,
                              workspace, workspace_bytes, window, stream=None):
    """attn_decode_cached over the last `window` positions up to *kv_pos_dev (0 = all); see attn_gqa.h."""
    f = _f32()
    if hasattr(kv_pos_dev, "element_size") and kv_pos_dev.element_size() != 4:
        raise ValueError("kv_pos_dev must hold one 32-bit unsigned position")
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().attn_decode_cached_window(
        _addr(q, "q", f), _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f),
        _addr(kv_pos_dev, "kv_pos_dev"),
        _addr(out, "out", f), num_heads, num_kv_heads, head_dim, max_seq,
        _addr(workspace, "workspace"), workspace_bytes, window, _stream(stream)), "attn_decode_cached_window")


def attn_prefill(q_batch, k_cache, v_cache, out_batch, n_queries, n_heads, n_kv_heads, head_dim, kv_dim,
                 max_seq, scale, start_pos, q_stride, out_stride, q_base, prec=ATTN_FP32, stream=None):
    """Batched causal prefill against a KV cache; see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_prefill(
        _addr(q_batch, "q_batch", f), _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f),
        _addr(out_batch, "out_batch", f), n_queries, n_heads, n_kv_heads, head_dim, kv_dim, max_seq,
        float(scale), start_pos, q_stride, out_stride, q_base, prec, _stream(stream)), "attn_prefill")


def attn_prefill_window(q_batch, k_cache, v_cache, out_batch, n_queries, n_heads, n_kv_heads, head_dim, kv_dim,
                        max_seq, scale, start_pos, q_stride, out_stride, q_base, prec, window, stream=None):
    """attn_prefill restricted to each row's last `window` keys (0 = all); see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_prefill_window(
        _addr(q_batch, "q_batch", f), _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f),
        _addr(out_batch, "out_batch", f), n_queries, n_heads, n_kv_heads, head_dim, kv_dim, max_seq,
        float(scale), start_pos, q_stride, out_stride, q_base, prec, window, _stream(stream)), "attn_prefill_window")


def attn_decode_append(q, k_new, v_new, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim,
                       max_seq, workspace, workspace_bytes=None, stream=None):
    """Write the new token's K/V row at *kv_pos_dev, then decode over 0..kv_pos; see attn_gqa.h."""
    f = _f32()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().attn_decode_append(
        _addr(q, "q", f, True), _addr(k_new, "k_new", f, True), _addr(v_new, "v_new", f, True),
        _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f), _addr(kv_pos_dev, "kv_pos_dev", None, True),
        _addr(out, "out", f, True), num_heads,
        num_kv_heads, head_dim, max_seq, _addr(workspace, "workspace"), workspace_bytes, _stream(stream)),
        "attn_decode_append")


def attn_decode_paged(q, k_pages, v_pages, block_table, kv_pos_dev, out, num_heads, num_kv_heads, head_dim,
                      page_rows, num_pages, max_blocks, workspace, workspace_bytes=None, window=0, stream=None):
    """Cached decode against a paged cache (block_table: device uint32); see attn_gqa.h."""
    f = _f32()
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().attn_decode_paged(
        _addr(q, "q", f), _addr(k_pages, "k_pages", f), _addr(v_pages, "v_pages", f),
        _addr(block_table, "block_table"), _addr(kv_pos_dev, "kv_pos_dev"), _addr(out, "out", f), num_heads,
        num_kv_heads, head_dim, page_rows, num_pages, max_blocks, _addr(workspace, "workspace"), workspace_bytes,
        window, _stream(stream)), "attn_decode_paged")


def attn_prefill_paged(q_batch, k_pages, v_pages, block_table, out_batch, n_queries, n_heads, n_kv_heads, head_dim,
                       kv_dim, page_rows, num_pages, max_blocks, scale, start_pos, q_stride, out_stride, q_base,
                       prec=ATTN_FP32, window=0, stream=None):
    """Batched causal prefill against a paged cache; see attn_gqa.h."""
    f = _f32()
    _check(load_library().attn_prefill_paged(
        _addr(q_batch, "q_batch", f), _addr(k_pages, "k_pages", f), _addr(v_pages, "v_pages", f),
        _addr(block_table, "block_table"), _addr(out_batch, "out_batch", f), n_queries, n_heads, n_kv_heads,
        head_dim, kv_dim, page_rows, num_pages, max_blocks, float(scale), start_pos, q_stride, out_stride, q_base,
        prec, window, _stream(stream)), "attn_prefill_paged")


def attn_decode_cached_noalloc(q, k_cache, v_cache, kv_pos_dev, out, num_heads, num_kv_heads, head_dim, max_seq,
                               stream=None):
    """Cached decode with no workspace argument: the library uses a fixed
    4 MiB device array of its own instead (for callers that cannot allocate
    device memory); see attn_gqa.h for its limits and sharing rules."""
    lib = load_library()
    fn = lib.attn_decode_cached_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [_vp, _vp, _vp, _vp, _vp, _u32, _u32, _u32, _u32, _vp]
    f = _f32()
    if hasattr(kv_pos_dev, "element_size") and kv_pos_dev.element_size() != 4:
        raise ValueError("kv_pos_dev must hold one 32-bit unsigned position")
    _check(fn(_addr(q, "q", f), _addr(k_cache, "k_cache", f), _addr(v_cache, "v_cache", f),
              _addr(kv_pos_dev, "kv_pos_dev"), _addr(out, "out", f), num_heads, num_kv_heads, head_dim, max_seq,
              _stream(stream)), "attn_decode_cached_noalloc")


def attn_set_workspace(workspace, workspace_bytes=None):
    """Bind a caller-owned device buffer (256-byte aligned) for the scratch of
    this thread's later calls, or unbind with None; see attn_gqa.h."""
    if workspace is None:
        _check(load_library().attn_set_workspace(None, 0), "attn_set_workspace")
        return
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().attn_set_workspace(_addr(workspace, "workspace"), workspace_bytes), "attn_set_workspace")


def attn_forward_workspace_bytes(q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask, prec, window=0, rope=False):
    return int(load_library().attn_forward_workspace_bytes(q_seq, kv_seq, num_heads, num_kv_heads, head_dim, mask,
                                                           prec, window, 1 if rope else 0))


def attn_prefill_workspace_bytes(n_queries, n_heads, n_kv_heads, head_dim, kv_dim, max_seq, start_pos, q_base, prec,
                                 window=0):
    return int(load_library().attn_prefill_workspace_bytes(n_queries, n_heads, n_kv_heads, head_dim, kv_dim, max_seq,
                                                           start_pos, q_base, prec, window))


def attn_backward_workspace_bytes(q_seq, kv_seq, num_heads, num_kv_heads, head_dim, prec, rope=False):
    return int(load_library().attn_backward_workspace_bytes(q_seq, kv_seq, num_heads, num_kv_heads, head_dim, prec,
                                                            1 if rope else 0))


def attn_scratch_reserved_bytes():
    return int(load_library().attn_scratch_reserved_bytes())


def attn_scratch_peak_bytes(reset=False):
    return int(load_library().attn_scratch_peak_bytes(1 if reset else 0))


def attn_release_scratch():
    _check(load_library().attn_release_scratch(), "attn_release_scratch")


def attn_selftest_wait_timeout(timeout_us=10000, stream=None):
    """Run the bounded-wait failure path once (see attn_gqa.h); read the
    outcome with attn_get_status()."""
    lib = load_library()
    fn = lib.attn_selftest_wait_timeout
    fn.restype = ctypes.c_int
    fn.argtypes = [_u32, _vp]
    _check(fn(timeout_us, _stream(stream)), "attn_selftest_wait_timeout")


def attn_get_status(stream=None):
    """Synchronise `stream`, return and clear the device status word."""
    return int(load_library().attn_get_status(_stream(stream)))


def attn_status_string(code):
    try:
        return load_library().attn_status_string(code).decode()
    except RuntimeError:
        return "status %d" % code
