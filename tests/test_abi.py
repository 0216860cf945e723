"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching the device.

The calls below pass made-up device addresses, which host validation must
refuse before anything is launched.  They therefore never run where a GPU is
visible: there, test_abi_device_hidden.py runs this module in a child process
with CUDA_VISIBLE_DEVICES="" instead, so that a validation regression shows
as a wrong status code (no device to launch on) and never as a kernel
reading a made-up address on a shared GPU."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # never dereferenced: every call below fails validation first


def gpu_visible():
    """True when this process can see a CUDA device."""
    if os.environ.get("CUDA_VISIBLE_DEVICES") == "":
        return False
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


pytestmark = pytest.mark.skipif(gpu_visible(), reason="a GPU is visible: test_abi_device_hidden.py runs this "
                                                      "module in a child process with the device hidden")


@pytest.fixture(scope="module")
def lib():
    from attention_gqa_online_gb300 import build
    build.build()
    import attention_gqa_online_gb300 as A
    return A.load_library()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"ATTN_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"attn_forward", "attn_decode_cached", "attn_prefill", "attn_decode_workspace_bytes",
            "attn_get_status", "attn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(5):
        assert lib.attn_status_string(code)
    assert lib.attn_status_string(99) == b"unknown status"


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, q_seq=16, kv_seq=16, H=4, G=2, D=64, mask=0, prec=0):
    return lib.attn_forward(q, k, v, out, lse, q_seq, kv_seq, H, G, D, mask, prec, None)


@pytest.mark.parametrize("kw", [
    dict(H=5, G=2), dict(G=0), dict(D=0), dict(D=129), dict(mask=3), dict(mask=-1), dict(prec=7),
    dict(mask=0, kv_seq=17), dict(mask=1, kv_seq=8), dict(q=None), dict(out=None), dict(k=None),
    dict(mask=2, kv_seq=5, v=None), dict(q_seq=2 ** 31),
])
def test_forward_rejects(lib, kw):
    assert fwd(lib, **kw) == 1


def test_forward_empty_query_is_noop(lib):
    assert fwd(lib, q=None, k=None, v=None, out=None, q_seq=0, kv_seq=0) == 0
    assert fwd(lib, q=None, k=None, v=None, out=None, q_seq=0, kv_seq=5, mask=2) == 0


def pre(lib, q=FAKE, k=FAKE, v=FAKE, out=FAKE, n=8, H=4, G=2, D=64, kv_dim=128, max_seq=64, scale=0.125,
        start=0, q_stride=256, out_stride=256, q_base=0, prec=0):
    return lib.attn_prefill(q, k, v, out, n, H, G, D, kv_dim, max_seq, scale, start, q_stride, out_stride,
                            q_base, prec, None)


@pytest.mark.parametrize("kw", [
    dict(H=6, G=4), dict(D=130), dict(kv_dim=127), dict(q_stride=255), dict(out_stride=100),
    dict(start=50, n=15), dict(start=40, q_base=20, n=5), dict(scale=math.inf), dict(scale=math.nan),
    dict(q=None), dict(k=None), dict(v=None), dict(out=None), dict(prec=3), dict(max_seq=2 ** 31, n=1),
])
def test_prefill_rejects(lib, kw):
    assert pre(lib, **kw) == 1


def test_prefill_empty_batch_is_noop(lib):
    assert pre(lib, q=None, k=None, v=None, out=None, n=0) == 0


def dec(lib, q=FAKE, k=FAKE, v=FAKE, pos=FAKE, out=FAKE, H=32, G=8, D=128, max_seq=100, ws=FAKE, nbytes=1 << 20):
    return lib.attn_decode_cached(q, k, v, pos, out, H, G, D, max_seq, ws, nbytes, None)


@pytest.mark.parametrize("kw", [
    dict(H=30), dict(G=0), dict(D=0), dict(D=200), dict(max_seq=0), dict(q=None), dict(k=None), dict(v=None),
    dict(pos=None), dict(out=None),
])
def test_decode_rejects(lib, kw):
    assert dec(lib, **kw) == 1


def test_workspace_query_rejects_bad_sizes(lib):
    assert lib.attn_decode_workspace_bytes(5, 2, 64, 100) == 0
    assert lib.attn_decode_workspace_bytes(4, 2, 64, 0) == 0
    assert lib.attn_decode_workspace_bytes(4, 2, 0, 10) == 0


# ---------------------------------------------------------------- windowed entry points
@pytest.mark.parametrize("kw", [
    dict(H=5, G=2), dict(D=129), dict(mask=3), dict(mask=0, kv_seq=17), dict(q=None), dict(prec=7),
])
@pytest.mark.parametrize("window", [0, 1, 2 ** 32 - 1])
def test_forward_window_rejects(lib, kw, window):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, lse=None, q_seq=16, kv_seq=16, H=4, G=2, D=64, mask=0, prec=0)
    a.update(kw)
    assert lib.attn_forward_window(a["q"], a["k"], a["v"], a["out"], a["lse"], a["q_seq"], a["kv_seq"], a["H"],
                                   a["G"], a["D"], a["mask"], a["prec"], window, None) == 1


def test_forward_window_empty_query_is_noop(lib):
    assert lib.attn_forward_window(None, None, None, None, None, 0, 0, 4, 2, 64, 0, 0, 7, None) == 0


@pytest.mark.parametrize("kw", [dict(kv_dim=127), dict(start=50, n=15), dict(scale=math.nan), dict(out=None)])
def test_prefill_window_rejects(lib, kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, n=8, H=4, G=2, D=64, kv_dim=128, max_seq=64, scale=0.125,
             start=0, q_stride=256, out_stride=256, q_base=0, prec=0)
    a.update(kw)
    assert lib.attn_prefill_window(a["q"], a["k"], a["v"], a["out"], a["n"], a["H"], a["G"], a["D"], a["kv_dim"],
                                   a["max_seq"], a["scale"], a["start"], a["q_stride"], a["out_stride"],
                                   a["q_base"], a["prec"], 16, None) == 1


@pytest.mark.parametrize("kw", [dict(H=30), dict(max_seq=0), dict(pos=None)])
def test_decode_window_rejects(lib, kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, pos=FAKE, out=FAKE, H=32, G=8, D=128, max_seq=100)
    a.update(kw)
    assert lib.attn_decode_cached_window(a["q"], a["k"], a["v"], a["pos"], a["out"], a["H"], a["G"], a["D"],
                                         a["max_seq"], FAKE, 1 << 20, 16, None) == 1


@pytest.mark.parametrize("kw", [
    dict(H=5, G=2), dict(D=129), dict(mask=3), dict(mask=0, kv_seq=17), dict(q=None), dict(dout=None),
    dict(lse=None), dict(out=None), dict(dq=None), dict(dk=None), dict(dv=None), dict(prec=7),
])
def test_backward_rejects(lib, kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, out=FAKE, dout=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, q_seq=16, kv_seq=16,
             H=4, G=2, D=64, mask=0, prec=0)
    a.update(kw)
    assert lib.attn_backward(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"],
                             a["q_seq"], a["kv_seq"], a["H"], a["G"], a["D"], a["mask"], a["prec"], 0, None) == 1


def test_backward_empty_query_is_noop(lib):
    assert lib.attn_backward(None, None, None, None, None, None, None, None, None, 0, 0, 4, 2, 64, 0, 0, 0,
                             None) == 0


@pytest.mark.parametrize("kw", [dict(page_rows=0), dict(num_pages=0), dict(max_blocks=0), dict(table=None),
                                dict(H=5), dict(page_rows=2 ** 20, max_blocks=2 ** 12)])
def test_decode_paged_rejects(lib, kw):
    a = dict(table=FAKE, H=32, G=8, D=128, page_rows=32, num_pages=10, max_blocks=8)
    a.update(kw)
    assert lib.attn_decode_paged(FAKE, FAKE, FAKE, a["table"], FAKE, FAKE, a["H"], a["G"], a["D"], a["page_rows"],
                                 a["num_pages"], a["max_blocks"], FAKE, 1 << 20, 0, None) == 1


@pytest.mark.parametrize("kw", [dict(page_rows=0), dict(table=None), dict(start=60, n=10), dict(kv_dim=100)])
def test_prefill_paged_rejects(lib, kw):
    a = dict(table=FAKE, page_rows=32, num_pages=4, max_blocks=2, start=0, n=8, kv_dim=128)
    a.update(kw)
    assert lib.attn_prefill_paged(FAKE, FAKE, FAKE, a["table"], FAKE, a["n"], 4, 2, 64, a["kv_dim"], a["page_rows"],
                                  a["num_pages"], a["max_blocks"], 0.125, a["start"], 256, 256, 0, 0, 0, None) == 1


@pytest.mark.parametrize("D,base,rows", [(0, 1e4, 8), (7, 1e4, 8), (130, 1e4, 8), (64, 1.0, 8), (64, math.inf, 8),
                                         (64, math.nan, 8)])
def test_rope_table_rejects(lib, D, base, rows):
    assert lib.attn_rope_table(FAKE, rows, D, base, None) == 1


def test_forward_rope_rejects_odd_and_short(lib):
    assert lib.attn_forward_rope(FAKE, FAKE, FAKE, FAKE, None, 8, 8, 2, 1, 63, 0, 0, 0, FAKE, 8, None) == 1
    assert lib.attn_forward_rope(FAKE, FAKE, FAKE, FAKE, None, 8, 8, 2, 1, 64, 0, 0, 0, FAKE, 7, None) == 1
    assert lib.attn_forward_rope(FAKE, FAKE, FAKE, FAKE, None, 8, 8, 2, 1, 64, 0, 0, 0, None, 8, None) == 1


@pytest.mark.parametrize("kw", [dict(H=30), dict(max_seq=0), dict(kn=None), dict(vn=None), dict(pos=None)])
def test_decode_append_rejects(lib, kw):
    a = dict(kn=FAKE, vn=FAKE, pos=FAKE, H=32, G=8, D=128, max_seq=100)
    a.update(kw)
    assert lib.attn_decode_append(FAKE, a["kn"], a["vn"], FAKE, FAKE, a["pos"], FAKE, a["H"], a["G"], a["D"],
                                  a["max_seq"], FAKE, 1 << 20, None) == 1


def test_backward_rope_rejects(lib):
    args = [FAKE] * 9 + [8, 8, 2, 1, 64, 0, 0, 0]
    assert lib.attn_backward_rope(*args, None, 8, None) == 1          # no table
    assert lib.attn_backward_rope(*args, FAKE, 7, None) == 1          # table one row short
    odd = [FAKE] * 9 + [8, 8, 2, 1, 63, 0, 0, 0]
    assert lib.attn_backward_rope(*odd, FAKE, 8, None) == 1           # odd head_dim


def test_workspace_queries(lib):
    """Scratch sizes per call: what the tensor-core paths copy K/V into, the
    RoPE-turned K of the fp32 path, the backward's per-row values."""
    r = lambda b: (b + 255) // 256 * 256  # noqa: E731
    n, H, G, D = 300, 8, 2, 128
    tiles = (n + 127) // 128
    # ATTN_BF16: fp16 K and bf16 V (4 bytes per K/V element pair), one float per (tile, kv head)
    assert lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, 2, 0, 0) == r(r(n * G * D * 4) + tiles * G * 4)
    # ATTN_TF32: fp16 K only
    assert lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, 1, 0, 0) == r(r(n * G * D * 2) + tiles * G * 4)
    assert lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, 0, 0, 0) == 0
    assert lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, 0, 0, 1) == r(n * G * D * 4)
    assert lib.attn_forward_workspace_bytes(n, n + 1, H, G, D, 0, 2, 0, 0) == 0  # causal needs kv_seq == q_seq
    # prefill 40 queries from position 100 of a 300-row cache: keys 0..139 are read
    assert lib.attn_prefill_workspace_bytes(40, H, G, D, G * D, 300, 100, 0, 2, 0) == r(r(140 * G * D * 4) + 2 * G * 4)
    assert lib.attn_prefill_workspace_bytes(40, H, G, D, G * D, 100, 100, 0, 2, 0) == 0  # past the cache
    assert lib.attn_backward_workspace_bytes(n, n, H, G, D, 0, 0) == r(n * H * 8)
    assert lib.attn_backward_workspace_bytes(n, n, H, G, D, 0, 1) == r((n * H + n * G) * D * 4) + r(n * H * 8)
    qe, ke = n * H * D, n * G * D
    assert lib.attn_backward_workspace_bytes(n, n, H, G, D, 2, 0) == 2 * r(n * H * 4) + 2 * r(qe * 2) + 2 * r(ke * 2)
    # A tensor-core call whose layout runs on the fp32 kernel needs that kernel's
    # scratch: the tensor-core precisions report at least the fp32 size.
    for rope in (0, 1):
        fp32 = lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, 0, 0, rope)
        for prec in (1, 2):
            assert lib.attn_forward_workspace_bytes(n, n, H, G, D, 0, prec, 0, rope) >= fp32
    assert lib.attn_backward_workspace_bytes(n, n, 6, 2, D, 2, 0) >= lib.attn_backward_workspace_bytes(n, n, 6, 2, D, 0, 0)


def test_set_workspace_rejects_misaligned(lib):
    assert lib.attn_set_workspace(FAKE + 16, 4096) == 1
    assert lib.attn_set_workspace(None, 0) == 0
