"""fp64 CPU oracle for GQA online-softmax attention -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The CUDA library never imports it and it imports nothing from the
library.  The arithmetic lives in ``attn_oracle.c`` (plain C, fp64); this file
only marshals numpy arrays through ctypes.

Every function takes fp32 inputs (numpy, C-contiguous) and returns fp64
results.  Layouts and window rules are those of the three shader pages:
meganeura 0.2.0 src/shaders/attention.wgsl (forward), meganeura 0.2.0
src/shaders/cached_attention.wgsl (decode) and cera
src/backend/shaders/attention_prefill.wgsl (prefill).
"""
import ctypes
import os

import numpy as np

from . import build as _build

CAUSAL, FULL, CROSS = 0, 1, 2

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_c_int = ctypes.c_int


def load(lib_path=None):
    """Load (building first if needed) an oracle shared library."""
    path = lib_path or _build.build()
    lib = ctypes.CDLL(path)
    lib.oracle_forward.restype = _c_int
    lib.oracle_forward.argtypes = [_f32p, _f32p, _f32p, _f64p, ctypes.c_void_p,
                                   _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   ctypes.c_void_p, _c_int, _c_int]
    lib.oracle_decode.restype = _c_int
    lib.oracle_decode.argtypes = [_f32p, _f32p, _f32p, ctypes.c_uint, _f64p,
                                  _c_int, _c_int, _c_int, _c_int, _c_int]
    lib.oracle_prefill.restype = _c_int
    lib.oracle_prefill.argtypes = [_f32p, _f32p, _f32p, _f64p] + [_c_int] * 6 + \
        [ctypes.c_float] + [_c_int] * 4 + [ctypes.c_void_p, _c_int, _c_int]
    lib.oracle_forward_rope.restype = _c_int
    lib.oracle_forward_rope.argtypes = [_f32p, _f32p, _f32p, _f64p, ctypes.c_void_p] + [_c_int] * 6 + \
        [ctypes.c_void_p, _c_int, _c_int, ctypes.c_double]
    lib.oracle_backward.restype = _c_int
    lib.oracle_backward.argtypes = [_f32p, _f32p, _f32p, _f32p, _f64p, _f64p, _f64p] + [_c_int] * 7
    lib.oracle_backward_rope.restype = _c_int
    lib.oracle_backward_rope.argtypes = [_f32p, _f32p, _f32p, _f32p, _f64p, _f64p, _f64p] + [_c_int] * 7 + \
        [ctypes.c_double]
    lib.oracle_num_threads.restype = _c_int
    lib.oracle_num_threads.argtypes = []
    return lib


class Oracle:
    """numpy front end over one oracle shared library."""

    def __init__(self, lib_path=None):
        self.lib = load(lib_path)

    def num_threads(self):
        return int(self.lib.oracle_num_threads())

    @staticmethod
    def _rows(rows):
        if rows is None:
            return None, 0, None
        arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        return arr.ctypes.data_as(ctypes.c_void_p), int(arr.size), arr

    def forward(self, q, k, v, q_seq, kv_seq, H, G, D, mask, rows=None, want_lse=True, window=0):
        """Returns (out [q_seq, H*D], lse [q_seq, H, 2]); rows not listed stay NaN.
        window > 0 keeps the last `window` keys of every row's window."""
        q, k, v = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v))
        out = np.full((max(q_seq, 0), H * D), np.nan)
        lse = np.full((max(q_seq, 0), H, 2), np.nan)
        rp, nr, keep = self._rows(rows)
        rc = self.lib.oracle_forward(q.reshape(-1), k.reshape(-1), v.reshape(-1), out.reshape(-1),
                                     lse.ctypes.data_as(ctypes.c_void_p) if want_lse else None,
                                     q_seq, kv_seq, H, G, D, mask, rp, nr, int(window))
        del keep
        if rc != 0:
            raise ValueError("oracle_forward rejected its arguments")
        return out, lse

    def forward_rope(self, q, k, v, q_seq, kv_seq, H, G, D, mask, rope_base, rows=None, want_lse=True, window=0):
        """forward() with RoPE on q (row i at position i) and k (row t at position t)."""
        q, k, v = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v))
        out = np.full((max(q_seq, 0), H * D), np.nan)
        lse = np.full((max(q_seq, 0), H, 2), np.nan)
        rp, nr, keep = self._rows(rows)
        rc = self.lib.oracle_forward_rope(q.reshape(-1), k.reshape(-1), v.reshape(-1), out.reshape(-1),
                                          lse.ctypes.data_as(ctypes.c_void_p) if want_lse else None,
                                          q_seq, kv_seq, H, G, D, mask, rp, nr, int(window), float(rope_base))
        del keep
        if rc != 0:
            raise ValueError("oracle_forward_rope rejected its arguments")
        return out, lse

    def decode(self, q, k_cache, v_cache, kv_pos, H, G, D, max_seq, window=0):
        """Returns out [1, H*D]."""
        q, k_cache, v_cache = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k_cache, v_cache))
        out = np.full((1, H * D), np.nan)
        rc = self.lib.oracle_decode(q.reshape(-1), k_cache.reshape(-1), v_cache.reshape(-1),
                                    int(kv_pos), out.reshape(-1), H, G, D, max_seq, int(window))
        if rc != 0:
            raise ValueError("oracle_decode rejected its arguments")
        return out

    def backward_rope(self, q, k, v, dout, q_seq, kv_seq, H, G, D, mask, rope_base, window=0):
        """backward() of forward_rope(): returns (dq, dk, dv) with respect to the unturned q, k."""
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
        dq = np.full((max(q_seq, 0), H * D), np.nan)
        dk = np.full((max(kv_seq, 0), G * D), np.nan)
        dv = np.full((max(kv_seq, 0), G * D), np.nan)
        rc = self.lib.oracle_backward_rope(q.reshape(-1), k.reshape(-1), v.reshape(-1), dout.reshape(-1),
                                           dq.reshape(-1), dk.reshape(-1), dv.reshape(-1), q_seq, kv_seq, H, G, D,
                                           mask, int(window), float(rope_base))
        if rc != 0:
            raise ValueError("oracle_backward_rope rejected its arguments")
        return dq, dk, dv

    # Paged KV cache.  The pages name paged KV only as future work for caches
    # that overflow one buffer; the layout read here: the cache is cut into
    # pages of page_rows consecutive positions, the pool holds num_pages pages
    # [num_pages, page_rows, kv_dim], and logical position t lives in pool page
    # block_table[t // page_rows] at row t % page_rows.  The oracle gathers the
    # logical cache [len(block_table) * page_rows, kv_dim] from the pool and
    # runs the contiguous computation on it.
    @staticmethod
    def gather_pages(pool, block_table, page_rows):
        pool = np.asarray(pool, dtype=np.float32)
        table = np.asarray(block_table, dtype=np.int64)
        num_pages = pool.shape[0] // page_rows
        if pool.shape[0] != num_pages * page_rows or table.min(initial=0) < 0 or \
                table.max(initial=0) >= num_pages:
            raise ValueError("bad page pool or block table")
        pages = pool.reshape(num_pages, page_rows, pool.shape[1])
        return np.ascontiguousarray(pages[table].reshape(len(table) * page_rows, pool.shape[1]))

    def decode_paged(self, q, k_pool, v_pool, block_table, kv_pos, H, G, D, page_rows, window=0):
        """Decode over a paged cache (capacity len(block_table) * page_rows rows); returns out [1, H*D]."""
        kc = self.gather_pages(k_pool, block_table, page_rows)
        vc = self.gather_pages(v_pool, block_table, page_rows)
        return self.decode(q, kc, vc, kv_pos, H, G, D, kc.shape[0], window=window)

    def prefill_paged(self, q_batch, k_pool, v_pool, block_table, out_rows, n_queries, H, G, D, kv_dim, page_rows,
                      scale, start_pos, q_stride, out_stride, q_base, rows=None, window=0):
        """Prefill against a paged cache (max_seq = len(block_table) * page_rows)."""
        kc = self.gather_pages(k_pool, block_table, page_rows)
        vc = self.gather_pages(v_pool, block_table, page_rows)
        return self.prefill(q_batch, kc, vc, out_rows, n_queries, H, G, D, kv_dim, kc.shape[0], scale, start_pos,
                            q_stride, out_stride, q_base, rows=rows, window=window)

    def backward(self, q, k, v, dout, q_seq, kv_seq, H, G, D, mask, window=0):
        """Gradients of out for upstream dout: returns (dq [q_seq, H*D], dk, dv [kv_seq, G*D])."""
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
        dq = np.full((max(q_seq, 0), H * D), np.nan)
        dk = np.full((max(kv_seq, 0), G * D), np.nan)
        dv = np.full((max(kv_seq, 0), G * D), np.nan)
        rc = self.lib.oracle_backward(q.reshape(-1), k.reshape(-1), v.reshape(-1), dout.reshape(-1),
                                      dq.reshape(-1), dk.reshape(-1), dv.reshape(-1), q_seq, kv_seq, H, G, D,
                                      mask, int(window))
        if rc != 0:
            raise ValueError("oracle_backward rejected its arguments")
        return dq, dk, dv

    def prefill(self, q_batch, k_cache, v_cache, out_rows, n_queries, H, G, D, kv_dim, max_seq,
                scale, start_pos, q_stride, out_stride, q_base, rows=None, window=0):
        """Returns out_batch [out_rows, out_stride] (fp64, NaN where not written)."""
        q_batch, k_cache, v_cache = (np.ascontiguousarray(x, dtype=np.float32)
                                     for x in (q_batch, k_cache, v_cache))
        out = np.full((out_rows, out_stride), np.nan)
        rp, nr, keep = self._rows(rows)
        rc = self.lib.oracle_prefill(q_batch.reshape(-1), k_cache.reshape(-1), v_cache.reshape(-1),
                                     out.reshape(-1), n_queries, H, G, D, kv_dim, max_seq,
                                     float(scale), start_pos, q_stride, out_stride, q_base, rp, nr, int(window))
        del keep
        if rc != 0:
            raise ValueError("oracle_prefill rejected its arguments")
        return out


_default = None


def default():
    """Process-wide oracle instance (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
