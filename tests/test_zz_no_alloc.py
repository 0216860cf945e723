"""attn_decode_cached_noalloc through the C ABI, against attn_decode_cached and the oracle.

The no-allocation decode is for callers that cannot give the library device
scratch memory (a plugin inside a framework that owns every allocation, a
serving loop that must never call cudaMalloc).  It must give the same answer
as the workspace-taking decode, call after call, even though every call
reuses one fixed scratch array that keeps the previous call's contents.
This file is collected last so that a failure here never hides another
test's result.
"""
import ctypes

import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import FP32, assert_out_close, dev

pytestmark = pytest.mark.gpu


def c_noalloc(lib):
    fn = lib.attn_decode_cached_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_uint32] * 4 + [ctypes.c_void_p]
    return fn


@pytest.mark.parametrize("H,G,D,max_seq,positions", [
    (32, 8, 128, 16384, [16383, 511]),   # the decode benchmark shape, then a short window
    (16, 2, 64, 3000, [2999, 64]),
    (32, 2, 128, 4096, [4095, 100]),     # 16 query heads per kv head: four head groups per kv head
])
def test_noalloc_matches_workspace_decode_and_oracle(cuda_lib, orc, H, G, D, max_seq, positions):
    lib = cuda_lib.load_library()
    noalloc = c_noalloc(lib)
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=11)
    dq, dk, dv = dev(q), dev(kc), dev(vc)
    ws = torch.zeros(cuda_lib.attn_decode_workspace_bytes(H, G, D, max_seq), dtype=torch.uint8, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    vmax = float(vc.abs().max())
    for kv_pos in positions:
        pos.fill_(kv_pos)
        ref = torch.full((1, H * D), float("nan"), device="cuda")
        cuda_lib.attn_decode_cached(dq, dk, dv, pos, ref, H, G, D, max_seq, ws)
        exact = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), kv_pos, H, G, D, max_seq)
        for call in range(2):  # two calls in a row share (and reuse) the fixed scratch
            out = torch.full((1, H * D), float("nan"), device="cuda")
            rc = noalloc(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), pos.data_ptr(), out.data_ptr(),
                         H, G, D, max_seq, stream)
            assert rc == 0, cuda_lib.attn_status_string(rc)
            torch.cuda.synchronize()
            assert cuda_lib.attn_get_status() == 0
            got = out.cpu().numpy()
            where = "noalloc call %d at kv_pos %d" % (call, kv_pos)
            assert_out_close(got, ref.cpu().numpy(), FP32, vmax, where + " vs workspace decode")
            assert_out_close(got, exact, FP32, vmax, where + " vs oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    """Real (small) buffers throughout, so that even a call that wrongly went
    ahead would stay inside its allocations."""
    lib = cuda_lib.load_library()
    noalloc = c_noalloc(lib)
    # 16384 heads over 4096 kv heads at D = 128 need about 8.5 MiB of scratch
    # with a one-row cache (one split per head group).
    H, G, D, max_seq = 16384, 4096, 128, 1
    q = torch.zeros(H * D, device="cuda")
    out = torch.zeros(H * D, device="cuda")
    kc = torch.zeros(max_seq * G * D, device="cuda")
    vc = torch.zeros(max_seq * G * D, device="cuda")
    pos = torch.zeros(4, dtype=torch.int32, device="cuda")
    ptrs = [x.data_ptr() for x in (q, kc, vc, pos, out)]
    rc = noalloc(*ptrs, H, G, D, max_seq, None)
    assert rc == cuda_lib.ATTN_ERR_UNSUPPORTED
    assert noalloc(0, *ptrs[1:], 32, 8, 128, max_seq, None) == cuda_lib.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
