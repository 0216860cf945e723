"""attn_forward on the GPU against the fp64 oracle (same seeded inputs)."""
import math

import numpy as np
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import BF16, FP32, TF32, assert_lse_close, assert_out_close, dev, tc_supported

pytestmark = pytest.mark.gpu
CAUSAL, FULL, CROSS = 0, 1, 2
PRECS = [FP32, TF32, BF16]


def run_forward(A, q, k, v, q_seq, kv_seq, H, G, D, mask, prec):
    out = torch.full((q_seq, H * D), float("nan"), device="cuda")
    lse = torch.full((q_seq, H, 2), float("nan"), device="cuda")
    A.attn_forward(dev(q) if q_seq else None, dev(k) if kv_seq else None, dev(v) if kv_seq else None,
                   out, lse, q_seq, kv_seq, H, G, D, mask, prec)
    torch.cuda.synchronize()
    assert A.attn_get_status() == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def check(A, orc, q_seq, kv_seq, H, G, D, mask, prec, seed=0, rows=None, **kw):
    q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=seed, **kw)
    out, lse = run_forward(A, q, k, v, q_seq, kv_seq, H, G, D, mask, prec)
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, kv_seq, H, G, D, mask, rows=rows)
    sel = slice(None) if rows is None else np.asarray(rows)
    vmax = float(v.abs().max()) if kv_seq else 1.0
    where = "q%d kv%d H%d G%d D%d mask%d prec%d" % (q_seq, kv_seq, H, G, D, mask, prec)
    assert_out_close(out[sel], ro[sel], prec, vmax, where)
    assert_lse_close(lse[sel], rl[sel], prec, float(np.abs(rl[sel][..., 0]).max()) if q_seq else 1.0, where)
    return out, lse


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("mask,kv", [(CAUSAL, 16), (FULL, 16), (CROSS, 24)])
def test_small_config(cuda_lib, orc, prec, mask, kv):
    """q_seq=16, 4 heads over 2 kv heads, D=64, N(0,1), seed 0."""
    check(cuda_lib, orc, 16, kv, 4, 2, 64, mask, prec)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("q_seq,kv_seq,H,G,D,mask", [
    (67, 67, 6, 2, 80, CAUSAL),      # gs = 3, several row tiles, ragged tail
    (67, 67, 6, 2, 80, FULL),
    (45, 131, 8, 8, 64, CROSS),      # MHA, ragged key tail
    (130, 130, 16, 2, 128, CAUSAL),  # gs = 8
    (33, 33, 4, 1, 32, CAUSAL),
    (20, 20, 2, 1, 12, CAUSAL),      # head_dim not a multiple of 16
    (9, 9, 3, 3, 1, FULL),           # head_dim 1
    (5, 300, 2, 2, 100, CROSS),
    (1, 1, 4, 2, 64, CAUSAL),        # single query: window of one key
    (200, 200, 1, 1, 128, CAUSAL),
    (67, 67, 6, 2, 128, CAUSAL),     # gs = 3: 42 queries (126 of 128 rows) per block
    (150, 150, 12, 4, 64, FULL),     # gs = 3, D = 64
    (90, 90, 10, 2, 128, CAUSAL),    # gs = 5
    (61, 200, 14, 2, 64, CROSS),     # gs = 7
    (40, 40, 48, 1, 128, CAUSAL),    # gs = 48: two queries per block
    (5, 5, 128, 1, 64, FULL),        # gs = 128: one query per block
])
def test_shapes(cuda_lib, orc, prec, q_seq, kv_seq, H, G, D, mask):
    if prec != FP32 and not tc_supported(H, G, D):
        q, k, v = synthetic.forward_inputs(q_seq, kv_seq, H, G, D, seed=1)
        with pytest.raises(cuda_lib.AttnError) as e:
            run_forward(cuda_lib, q, k, v, q_seq, kv_seq, H, G, D, mask, prec)
        assert e.value.code == cuda_lib.ATTN_ERR_UNSUPPORTED
        return
    check(cuda_lib, orc, q_seq, kv_seq, H, G, D, mask, prec, seed=q_seq + D)


@pytest.mark.parametrize("prec", PRECS)
def test_window_one_returns_v0(cuda_lib, prec):
    q, k, v = synthetic.forward_inputs(3, 3, 4, 2, 64, seed=21)
    out, lse = run_forward(cuda_lib, q, k, v, 3, 3, 4, 2, 64, CAUSAL, prec)
    for h in range(4):
        g = h // 2
        np.testing.assert_allclose(out[0, h * 64:(h + 1) * 64], v[0, g * 64:(g + 1) * 64].numpy(), rtol=0,
                                   atol=1e-6 if prec == FP32 else 1e-2)
        assert abs(lse[0, h, 1]) < 1e-6


@pytest.mark.parametrize("prec", PRECS)
def test_empty_cross_window(cuda_lib, prec):
    q, _, _ = synthetic.forward_inputs(7, 0, 4, 2, 64, seed=22)
    out, lse = run_forward(cuda_lib, q, None, None, 7, 0, 4, 2, 64, CROSS, prec)
    assert np.all(out == 0.0) and np.all(lse == np.float32(-1e30))


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("mask,q_seq,kv_seq", [(FULL, 2048, 2048), (CROSS, 1024, 4096)])
def test_mha_full_and_cross(cuda_lib, orc, prec, mask, q_seq, kv_seq):
    """16 heads = 16 kv heads, D=64; Q,K N(0,1), V U(-1,1)."""
    rows = None if mask == CROSS else list(range(0, 2048, 7)) + [2047]
    check(cuda_lib, orc, q_seq, kv_seq, 16, 16, 64, mask, prec, seed=4, v_dist="uniform", rows=rows)


@pytest.mark.parametrize("prec", PRECS)
@pytest.mark.parametrize("q_seq", [8192, 8193])
def test_long_causal_stress(cuda_lib, orc, prec, q_seq):
    """q_seq 8192/8193, 32 heads over 8 kv heads, D=128, Q,K N(0,3^2): sampled rows."""
    rng = np.random.default_rng(q_seq)
    rows = sorted(set(range(16)) | set(range(q_seq - 16, q_seq)) | set(rng.integers(0, q_seq, 16).tolist()))
    check(cuda_lib, orc, q_seq, q_seq, 32, 8, 128, CAUSAL, prec, seed=5, rows=rows, qk_sigma=3.0)


@pytest.mark.parametrize("prec", [TF32, BF16])
@pytest.mark.parametrize("seed", [11, 12, 13])
def test_long_causal_stress_seeds(cuda_lib, orc, prec, seed):
    """The tensor-core precisions on further seeds of the long causal stress
    distribution (Q,K N(0,3^2)): 64 rows spread over the sequence."""
    q_seq = 8192
    rng = np.random.default_rng(seed)
    rows = sorted(set(rng.integers(0, q_seq, 56).tolist()) | set(range(q_seq - 8, q_seq)))
    check(cuda_lib, orc, q_seq, q_seq, 32, 8, 128, CAUSAL, prec, seed=seed, rows=rows, qk_sigma=3.0)


@pytest.mark.parametrize("prec", [TF32, BF16])
@pytest.mark.parametrize("qs,ks", [(1e-6, 1e6), (1e6, 1e-6), (2.0 ** 40, 2.0 ** -40), (2.0 ** -60, 2.0 ** 60)])
def test_operand_range(cuda_lib, orc, prec, qs, ks):
    """Scaling Q by qs and K by ks = 1/qs leaves every score, and so the result,
    unchanged.  The 16-bit path's fp16 score operands carry powers of two that
    keep them inside fp16's range whatever the fp32 magnitudes (plain fp16 would
    overflow beyond 65504 or lose everything below 6e-8)."""
    q_seq, H, G, D = 300, 8, 2, 128
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=23)
    ref, _ = run_forward(cuda_lib, q, k, v, q_seq, q_seq, H, G, D, CAUSAL, prec)
    out, _ = run_forward(cuda_lib, q * qs, k * ks, v, q_seq, q_seq, H, G, D, CAUSAL, prec)
    ro, _ = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, q_seq, H, G, D, CAUSAL)
    vmax = float(v.abs().max())
    assert_out_close(out, ro, prec, vmax, "scaled operands")
    if math.frexp(qs)[0] == 0.5:  # exact powers of two change no operand bit
        assert np.array_equal(out, ref)


def test_bf16_mixed_magnitude_tile(cuda_lib, orc):
    """One key row a million times larger than the others in its 128-key tile:
    the tile's power of two follows that row, and the other keys' scores keep
    their accuracy (fp16 subnormals only start far below their magnitude)."""
    q_seq, H, G, D = 256, 4, 1, 64
    q, k, v = synthetic.forward_inputs(q_seq, q_seq, H, G, D, seed=24)
    k[200] *= 1e6
    out, _ = run_forward(cuda_lib, q, k, v, q_seq, q_seq, H, G, D, FULL, BF16)
    ro, _ = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, q_seq, H, G, D, FULL)
    assert_out_close(out, ro, BF16, float(v.abs().max()), "mixed-magnitude tile")


@pytest.mark.parametrize("prec", PRECS)
def test_reference_max_moves_at_every_tile(cuda_lib, orc, prec):
    """Rows whose score max rises by 26 (base 2) at every 128-key tile, just
    above the tensor kernels' rescale threshold of 24: every tile moves the
    reference max, so O and the row sums are rescaled at every tile, and the
    16-bit kernel's two softmax groups hand the reference over at every tile.
    A skipped or wrong rescale leaves an earlier tile's value at weight ~1
    instead of 2^-26: an error of order max|V|.  Q is the unit vector e_0 (plus
    small noise); the last key of tile j is e_0 times the value that gives
    score 26 (j + 1) in base 2; the other keys are N(0,1)."""
    q_seq = kv_seq = 128 * 12
    H, G, D = 8, 2, 128
    gen = torch.Generator().manual_seed(17)
    q = 0.01 * torch.randn((q_seq, H * D), generator=gen)
    q.view(q_seq, H, D)[:, :, 0] += 1.0
    k = torch.randn((kv_seq, G * D), generator=gen)
    v = torch.randn((kv_seq, G * D), generator=gen)
    scale_log2 = (1.0 / math.sqrt(D)) * 1.4426950408889634
    for j in range(kv_seq // 128):
        kv = k.view(kv_seq, G, D)[128 * j + 127]
        kv.zero_()
        kv[:, 0] = 26.0 * (j + 1) / scale_log2
    out, lse = run_forward(cuda_lib, q, k, v, q_seq, kv_seq, H, G, D, CAUSAL, prec)
    rows = list(range(0, q_seq, 37)) + [127, 128, 255, 256, q_seq - 1]
    ro, rl = orc.forward(q.numpy(), k.numpy(), v.numpy(), q_seq, kv_seq, H, G, D, CAUSAL, rows=rows)
    sel = np.asarray(rows)
    assert_out_close(out[sel], ro[sel], prec, float(v.abs().max()), "score max rising 26 per tile")
    assert_lse_close(lse[sel], rl[sel], prec, float(np.abs(rl[sel][..., 0]).max()), "score max rising 26 per tile")
