"""attn_decode_cached on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import FP32, assert_out_close, dev

pytestmark = pytest.mark.gpu


def make_state(A, H, G, D, max_seq):
    nbytes = A.attn_decode_workspace_bytes(H, G, D, max_seq)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    return ws, pos


def run_decode(A, q, kc, vc, pos_t, ws, kv_pos, H, G, D, max_seq):
    pos_t.fill_(int(kv_pos) if kv_pos < 2 ** 31 else int(kv_pos) - 2 ** 32)
    out = torch.full((1, H * D), float("nan"), device="cuda")
    A.attn_decode_cached(q, kc, vc, pos_t, out, H, G, D, max_seq, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("kv_pos", [0, 7, 511, 4095, 16383])
def test_decode_config_sweep(cuda_lib, orc, kv_pos):
    """Q [1, 32*128], caches [16384, 8*128] N(0,1), 32 heads over 8 kv heads."""
    H, G, D, max_seq = 32, 8, 128, 16384
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=0)
    dq, dk, dv = dev(q), dev(kc), dev(vc)
    ws, pos = make_state(cuda_lib, H, G, D, max_seq)
    ref = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), kv_pos, H, G, D, max_seq)
    for _ in range(2):  # the workspace must be reusable call after call
        out = run_decode(cuda_lib, dq, dk, dv, pos, ws, kv_pos, H, G, D, max_seq)
        assert cuda_lib.attn_get_status() == 0
        assert_out_close(out, ref, FP32, float(vc.abs().max()), "decode kv_pos=%d" % kv_pos)


@pytest.mark.parametrize("H,G,D,max_seq,positions", [
    (16, 2, 64, 3000, [0, 63, 64, 65, 2999]),   # split kernel, gs = 8
    (8, 8, 128, 700, [0, 1, 699]),              # split kernel, MHA
    (4, 2, 64, 1, [0]),                         # one-row cache
    (6, 2, 80, 513, [0, 200, 512]),             # generic kernel (D = 80, gs = 3)
    (64, 4, 128, 260, [5, 259]),                # split kernel, gs = 16: four head groups per kv head
    (64, 8, 128, 4096, [0, 31, 32, 4095]),      # split kernel, gs = 8 at D = 128: two head groups
    (32, 2, 64, 1000, [0, 999]),                # split kernel, gs = 16 at D = 64: two head groups
    (96, 3, 128, 500, [100, 499]),              # gs = 32: eight head groups
    (2, 1, 12, 40, [0, 39]),                    # generic kernel, small D
])
def test_decode_shapes(cuda_lib, orc, H, G, D, max_seq, positions):
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=max_seq)
    dq, dk, dv = dev(q), dev(kc), dev(vc)
    ws, pos = make_state(cuda_lib, H, G, D, max_seq)
    for kp in positions:
        out = run_decode(cuda_lib, dq, dk, dv, pos, ws, kp, H, G, D, max_seq)
        assert cuda_lib.attn_get_status() == 0
        ref = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), kp, H, G, D, max_seq)
        assert_out_close(out, ref, FP32, float(vc.abs().max()), "H%d G%d D%d kv_pos=%d" % (H, G, D, kp))


def test_decode_kv_pos_zero_is_v0(cuda_lib):
    H, G, D, max_seq = 32, 8, 128, 16384
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=3)
    ws, pos = make_state(cuda_lib, H, G, D, max_seq)
    out = run_decode(cuda_lib, dev(q), dev(kc), dev(vc), pos, ws, 0, H, G, D, max_seq)
    for h in range(H):
        g = h // 4
        np.testing.assert_allclose(out[0, h * D:(h + 1) * D], vc[0, g * D:(g + 1) * D].numpy(), rtol=0, atol=1e-6)


@pytest.mark.parametrize("H,G,D", [(32, 8, 128), (6, 2, 80)])
def test_decode_kv_pos_past_cache_is_clamped_and_flagged(cuda_lib, orc, H, G, D):
    max_seq = 300
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=4)
    dq, dk, dv = dev(q), dev(kc), dev(vc)
    ws, pos = make_state(cuda_lib, H, G, D, max_seq)
    assert cuda_lib.attn_get_status() == 0
    for kp in (max_seq, max_seq + 77, 2 ** 32 - 1):
        out = run_decode(cuda_lib, dq, dk, dv, pos, ws, kp, H, G, D, max_seq)
        assert cuda_lib.attn_get_status() == cuda_lib.ATTN_ERR_INVALID_ARG
        ref = orc.decode(q.numpy(), kc.numpy(), vc.numpy(), max_seq - 1, H, G, D, max_seq)
        assert_out_close(out, ref, FP32, float(vc.abs().max()), "clamped kv_pos=%d" % kp)
    assert cuda_lib.attn_get_status() == 0


@pytest.mark.parametrize("H,G,D,max_seq", [(32, 8, 128, 4096), (16, 2, 64, 700), (6, 2, 80, 300),
                                            (64, 8, 128, 600)])
def test_decode_append(cuda_lib, orc, H, G, D, max_seq):
    """attn_decode_append writes the new row at kv_pos (and nothing else), then
    decodes over 0..kv_pos: a serving loop of steps against the oracle."""
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=max_seq + 3)
    rng = np.random.default_rng(max_seq)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    dk, dv = dev(kc), dev(vc)
    ws, pos = make_state(cuda_lib, H, G, D, max_seq)
    for kv_pos in (0, 1, 2, 63, max_seq // 2, max_seq - 1):
        kn = rng.standard_normal(G * D).astype(np.float32)
        vn = rng.standard_normal(G * D).astype(np.float32)
        qn = rng.standard_normal((1, H * D)).astype(np.float32)
        pos.fill_(kv_pos)
        out = torch.full((1, H * D), float("nan"), device="cuda")
        cuda_lib.attn_decode_append(dev(torch.from_numpy(qn)), dev(torch.from_numpy(kn)), dev(torch.from_numpy(vn)),
                                    dk, dv, pos, out, H, G, D, max_seq, ws)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        kh[kv_pos], vh[kv_pos] = kn, vn
        assert np.array_equal(dk.cpu().numpy(), kh) and np.array_equal(dv.cpu().numpy(), vh)
        ref = orc.decode(qn, kh, vh, kv_pos, H, G, D, max_seq)
        assert_out_close(out.cpu().numpy(), ref, FP32, float(np.abs(vh).max()), "append kv_pos=%d" % kv_pos)
    # past the cache: nothing written, status flagged
    before = dk.cpu().numpy().copy()
    pos.fill_(max_seq)
    out = torch.empty((1, H * D), device="cuda")
    cuda_lib.attn_decode_append(dev(q), dev(torch.zeros(G * D)), dev(torch.zeros(G * D)), dk, dv, pos, out, H, G, D,
                                max_seq, ws)
    assert cuda_lib.attn_get_status() == cuda_lib.ATTN_ERR_INVALID_ARG
    assert np.array_equal(dk.cpu().numpy(), before)


@pytest.mark.parametrize("H,G,D,max_seq", [(32, 8, 128, 4096), (16, 2, 64, 700)])
def test_decode_append_pinned_host_io(cuda_lib, orc, H, G, D, max_seq):
    """A serving step with its small inputs (q, the new K/V row, kv_pos) and its
    output in pinned host memory, read and written by the split decode kernel
    directly, against the oracle."""
    q, kc, vc = synthetic.decode_inputs(max_seq, H, G, D, seed=max_seq + 5)
    rng = np.random.default_rng(max_seq + 1)
    kh, vh = kc.numpy().copy(), vc.numpy().copy()
    dk, dv = dev(kc), dev(vc)
    ws, _ = make_state(cuda_lib, H, G, D, max_seq)
    qh = torch.empty((1, H * D)).pin_memory()
    knh, vnh = torch.empty(G * D).pin_memory(), torch.empty(G * D).pin_memory()
    posh = torch.zeros(4, dtype=torch.int32).pin_memory()
    outh = torch.empty((1, H * D)).pin_memory()
    for kv_pos in (0, 5, max_seq // 3, max_seq - 1):
        kn = rng.standard_normal(G * D).astype(np.float32)
        vn = rng.standard_normal(G * D).astype(np.float32)
        qn = rng.standard_normal((1, H * D)).astype(np.float32)
        qh.copy_(torch.from_numpy(qn)); knh.copy_(torch.from_numpy(kn)); vnh.copy_(torch.from_numpy(vn))
        posh[0] = kv_pos
        outh.fill_(float("nan"))
        cuda_lib.attn_decode_append(qh, knh, vnh, dk, dv, posh, outh, H, G, D, max_seq, ws)
        torch.cuda.synchronize()
        assert cuda_lib.attn_get_status() == 0
        kh[kv_pos], vh[kv_pos] = kn, vn
        assert np.array_equal(dk.cpu().numpy(), kh) and np.array_equal(dv.cpu().numpy(), vh)
        ref = orc.decode(qn, kh, vh, kv_pos, H, G, D, max_seq)
        assert_out_close(outh.numpy(), ref, FP32, float(np.abs(vh).max()), "pinned append kv_pos=%d" % kv_pos)
