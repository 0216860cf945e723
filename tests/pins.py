"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with something it must reproduce.  They are run on
the real oracle (tests/test_oracle.py) and on deliberately broken copies of it
(tests/test_oracle_mutants.py), which shows that a plausible slip in the
oracle -- a dropped term, a wrong sign or index, a transposed operand --
fails at least one of them.

Nothing here re-types the oracle's materialised formula.  The pins are:
  * PyTorch's own scaled_dot_product_attention (fp64, CPU) as an independent
    library routine for the same definition, GQA head map included;
  * the pages' own streaming recurrence (attention.wgsl, fn main: running
    max, correction, weight; final (max_score, log(sum_exp)) store), run
    element by element in pure Python on tiny shapes;
  * closed forms (one-key window, constant V rows, Q = 0, a three-key case
    worked by hand, the empty window);
  * invariants (GQA == MHA with replicated K/V heads, softmax normalisation,
    joint permutation of keys, causal prefix independence, shift of K along a
    fixed vector, decode/prefill/forward window consistency, strides).
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

from attention_gqa_online_gb300 import synthetic

CAUSAL, FULL, CROSS = 0, 1, 2
EMPTY_LSE = -1e30


def _np(t):
    return t.numpy() if isinstance(t, torch.Tensor) else t


def _small(seed=0, q_seq=16, kv_seq=None, H=4, G=2, D=64, **kw):
    kv = q_seq if kv_seq is None else kv_seq
    q, k, v = synthetic.forward_inputs(q_seq, kv, H, G, D, seed=seed, **kw)
    return _np(q), _np(k), _np(v)


def _scores(q, k, H, G, D, pos, h, n):
    """Score row of (pos, h) over keys [0, n), fp64 (used by invariants only)."""
    g = h // (H // G)
    qv = q[pos, h * D:(h + 1) * D].astype(np.float64)
    kk = k[:n, g * D:(g + 1) * D].astype(np.float64)
    return kk @ qv / math.sqrt(D)


# ---------------------------------------------------------------- library routine
def _sdpa(q, k, v, q_seq, kv_seq, H, G, D, causal):
    qt = torch.from_numpy(q.astype(np.float64)).reshape(q_seq, H, D).transpose(0, 1)[None]
    kt = torch.from_numpy(k.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None]
    vt = torch.from_numpy(v.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal, enable_gqa=True)
    return o[0].transpose(0, 1).reshape(q_seq, H * D).numpy()


def pin_sdpa_causal(orc):
    q, k, v = _small(seed=0)
    out, _ = orc.forward(q, k, v, 16, 16, 4, 2, 64, CAUSAL)
    ref = _sdpa(q, k, v, 16, 16, 4, 2, 64, True)
    assert np.max(np.abs(out - ref)) < 1e-12


def pin_sdpa_full(orc):
    q, k, v = _small(seed=0)
    out, _ = orc.forward(q, k, v, 16, 16, 4, 2, 64, FULL)
    ref = _sdpa(q, k, v, 16, 16, 4, 2, 64, False)
    assert np.max(np.abs(out - ref)) < 1e-12


def pin_sdpa_cross(orc):
    q, k, v = _small(seed=0, kv_seq=24)
    out, _ = orc.forward(q, k, v, 16, 24, 4, 2, 64, CROSS)
    ref = _sdpa(q, k, v, 16, 24, 4, 2, 64, False)
    assert np.max(np.abs(out - ref)) < 1e-12


def pin_sdpa_gqa_8_to_1(orc):
    q, k, v = _small(seed=3, q_seq=9, H=8, G=1, D=16)
    out, _ = orc.forward(q, k, v, 9, 9, 8, 1, 16, CAUSAL)
    ref = _sdpa(q, k, v, 9, 9, 8, 1, 16, True)
    assert np.max(np.abs(out - ref)) < 1e-12


# ---------------------------------------------------------------- the pages' recurrence
def _streaming_row(qv, krows, vrows, scale):
    """Per-key online softmax exactly as the forward page walks it, in fp64.

    Running state starts at (max -1e30, sum 0, out 0); each key updates
    new_max, correction = exp(max - new_max), weight = exp(score - new_max).
    Returns (out / safe_sum, max, log(sum) or -1e30)."""
    m, l = -1e30, 0.0
    o = [0.0] * len(qv)
    for kt, vt in zip(krows, vrows):
        s = sum(float(a) * float(b) for a, b in zip(qv, kt)) * scale
        nm = max(m, s)
        corr = math.exp(m - nm)
        w = math.exp(s - nm)
        l = l * corr + w
        o = [oi * corr + w * float(vi) for oi, vi in zip(o, vt)]
        m = nm
    safe = 1.0 if l == 0.0 else l
    return [oi / safe for oi in o], m, (EMPTY_LSE if l == 0.0 else math.log(l))


def _check_streaming(orc, q, k, v, q_seq, kv_seq, H, G, D, mask):
    out, lse = orc.forward(q, k, v, q_seq, kv_seq, H, G, D, mask)
    gs = H // G
    for pos in range(q_seq):
        n = pos + 1 if mask == CAUSAL else kv_seq
        for h in range(H):
            g = h // gs
            ref, m, logl = _streaming_row(q[pos, h * D:(h + 1) * D],
                                          k[:n, g * D:(g + 1) * D], v[:n, g * D:(g + 1) * D],
                                          1.0 / math.sqrt(D))
            assert np.max(np.abs(out[pos, h * D:(h + 1) * D] - np.array(ref))) < 1e-12
            assert abs(lse[pos, h, 0] - m) < 1e-12
            assert abs(lse[pos, h, 1] - logl) < 1e-12


def pin_streaming_causal(orc):
    q, k, v = _small(seed=1, q_seq=7, H=4, G=2, D=8)
    _check_streaming(orc, q, k, v, 7, 7, 4, 2, 8, CAUSAL)


def pin_streaming_cross(orc):
    q, k, v = _small(seed=2, q_seq=3, kv_seq=11, H=6, G=3, D=4, qk_sigma=3.0)
    _check_streaming(orc, q, k, v, 3, 11, 6, 3, 4, CROSS)


def pin_streaming_full(orc):
    q, k, v = _small(seed=4, q_seq=5, H=2, G=1, D=12, v_dist="uniform")
    _check_streaming(orc, q, k, v, 5, 5, 2, 1, 12, FULL)


# ---------------------------------------------------------------- closed forms
def pin_window_one_is_v0(orc):
    """Causal row 0 sees key 0 only: out = V[0] of its kv head, lse = (s_0, 0)."""
    q, k, v = _small(seed=5)
    out, lse = orc.forward(q, k, v, 16, 16, 4, 2, 64, CAUSAL)
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, h * 64:(h + 1) * 64], v[0, g * 64:(g + 1) * 64].astype(np.float64))
        s0 = float(np.dot(q[0, h * 64:(h + 1) * 64].astype(np.float64),
                          k[0, g * 64:(g + 1) * 64].astype(np.float64))) / 8.0
        assert abs(lse[0, h, 0] - s0) < 1e-12 and lse[0, h, 1] == 0.0


def pin_constant_v(orc):
    """Every V row equal to c (per kv head): any convex combination is c."""
    q, k, _ = _small(seed=6, kv_seq=24)
    c = np.linspace(-2, 3, 2 * 64, dtype=np.float32)
    v = np.tile(c, (24, 1))
    for mask, kv in ((CROSS, 24),):
        out, _ = orc.forward(q, k, v, 16, kv, 4, 2, 64, mask)
        for h in range(4):
            g = h // 2
            assert np.max(np.abs(out[:, h * 64:(h + 1) * 64] - c[g * 64:(g + 1) * 64])) < 1e-12


def pin_zero_query(orc):
    """Q = 0: all scores are 0, so out = mean of V over the window, lse = (0, log n)."""
    _, k, v = _small(seed=7)
    q = np.zeros((16, 4 * 64), np.float32)
    out, lse = orc.forward(q, k, v, 16, 16, 4, 2, 64, CAUSAL)
    for pos in range(16):
        for h in range(4):
            g = h // 2
            mean = v[:pos + 1, g * 64:(g + 1) * 64].astype(np.float64).mean(axis=0)
            assert np.max(np.abs(out[pos, h * 64:(h + 1) * 64] - mean)) < 1e-13
            assert lse[pos, h, 0] == 0.0 and abs(lse[pos, h, 1] - math.log(pos + 1)) < 1e-14


def pin_hand_worked(orc):
    """Three keys, D = 4 (scale 1/2), q = (2,0,0,0): scores are k_t[0] = 0, 1, 2.

    Weights are e^0, e^1, e^2 over 1 + e + e^2; V rows are unit vectors, so
    out = (1, e, e^2, 0) / (1 + e + e^2); lse = (2, log(1 + e^-1 + e^-2))."""
    q = np.array([[2, 0, 0, 0]], np.float32)
    k = np.array([[0, 5, -1, 2], [1, 0, 7, 0], [2, -3, 0, 1]], np.float32)
    v = np.eye(3, 4, dtype=np.float32)
    out, lse = orc.forward(q, k, v, 1, 3, 1, 1, 4, CROSS)
    e = math.e
    z = 1 + e + e * e
    assert np.max(np.abs(out[0] - np.array([1 / z, e / z, e * e / z, 0.0]))) < 1e-15
    assert lse[0, 0, 0] == 2.0 and abs(lse[0, 0, 1] - math.log(1 + 1 / e + 1 / (e * e))) < 1e-15


def pin_empty_window(orc):
    """Cross attention over zero keys writes zeros and lse = (-1e30, -1e30)."""
    q, _, _ = _small(seed=8)
    k = np.zeros((0, 128), np.float32)
    out, lse = orc.forward(q, k, k, 16, 0, 4, 2, 64, CROSS)
    assert np.all(out == 0.0) and np.all(lse == EMPTY_LSE)


# ---------------------------------------------------------------- invariants
def pin_gqa_equals_replicated_mha(orc):
    q, k, v = _small(seed=9, q_seq=12, H=8, G=2, D=32)
    out, lse = orc.forward(q, k, v, 12, 12, 8, 2, 32, CAUSAL)
    kr = np.repeat(k.reshape(12, 2, 32), 4, axis=1).reshape(12, 8 * 32)
    vr = np.repeat(v.reshape(12, 2, 32), 4, axis=1).reshape(12, 8 * 32)
    out2, lse2 = orc.forward(q, kr, vr, 12, 12, 8, 8, 32, CAUSAL)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_softmax_normalisation(orc):
    """slot0 is the row max, and sum_t exp(s_t - slot0 - slot1) = 1."""
    q, k, v = _small(seed=10, kv_seq=24, qk_sigma=3.0)
    _, lse = orc.forward(q, k, v, 16, 24, 4, 2, 64, CROSS)
    for pos in range(16):
        for h in range(4):
            s = _scores(q, k, 4, 2, 64, pos, h, 24)
            assert abs(lse[pos, h, 0] - s.max()) < 1e-12
            tot = np.exp(s - lse[pos, h, 0] - lse[pos, h, 1]).sum()
            assert abs(tot - 1.0) < 1e-12


def pin_key_permutation(orc):
    """Full/cross attention does not depend on the order of the (K, V) pairs."""
    q, k, v = _small(seed=11, kv_seq=24)
    perm = np.random.default_rng(11).permutation(24)
    out, lse = orc.forward(q, k, v, 16, 24, 4, 2, 64, CROSS)
    out2, lse2 = orc.forward(q, k[perm].copy(), v[perm].copy(), 16, 24, 4, 2, 64, CROSS)
    assert np.max(np.abs(out - out2)) < 1e-12 and np.max(np.abs(lse - lse2)) < 1e-12


def pin_causal_prefix(orc):
    """Causal row r is unchanged when K/V rows after r are overwritten."""
    q, k, v = _small(seed=12)
    out, lse = orc.forward(q, k, v, 16, 16, 4, 2, 64, CAUSAL)
    for r in (0, 5, 14):
        k2, v2 = k.copy(), v.copy()
        k2[r + 1:] = 1e3
        v2[r + 1:] = -7.0
        o2, l2 = orc.forward(q, k2, v2, 16, 16, 4, 2, 64, CAUSAL)
        assert np.array_equal(out[:r + 1], o2[:r + 1]) and np.array_equal(lse[:r + 1], l2[:r + 1])
        assert not np.array_equal(out[r + 1:], o2[r + 1:])


def pin_shift_invariance(orc):
    """K_t += u shifts every score of a row by scale * q.u: out unchanged,
    slot0 moves by that amount, slot1 unchanged."""
    q, k, v = _small(seed=13, kv_seq=24)
    k = (np.round(k * 1024.0) / 1024.0).astype(np.float32)   # k on a 2^-10 grid ...
    u = np.zeros(2 * 64, np.float32)
    u[:64] = 0.5        # ... so k + u is exact in fp32; kv head 0 only
    k2 = k + u
    assert np.array_equal(k2.astype(np.float64), k.astype(np.float64) + u.astype(np.float64))
    out, lse = orc.forward(q, k, v, 16, 24, 4, 2, 64, CROSS)
    out2, lse2 = orc.forward(q, k2, v, 16, 24, 4, 2, 64, CROSS)
    assert np.max(np.abs(out - out2)) < 1e-10
    for pos in range(16):
        for h in range(4):
            g = h // 2
            d = float(np.dot(q[pos, h * 64:(h + 1) * 64].astype(np.float64),
                             u[g * 64:(g + 1) * 64].astype(np.float64))) / 8.0
            assert abs(lse2[pos, h, 0] - lse[pos, h, 0] - d) < 1e-10
            assert abs(lse2[pos, h, 1] - lse[pos, h, 1]) < 1e-10


def pin_decode_prefill_forward_agree(orc):
    """Prefill row i == decode at kv_pos = start_pos + q_base + i, and a
    prefill from position 0 == causal forward (window rules of the three pages)."""
    H, G, D, max_seq = 4, 2, 16, 40
    qb, kc, vc = (_np(x) for x in synthetic.prefill_inputs(10, 80, max_seq, G * D, seed=14))
    start, qbase = 20, 3
    scale = np.float32(1.0 / math.sqrt(D))
    outp = orc.prefill(qb, kc, vc, 10, 7, H, G, D, G * D, max_seq, scale, start, 80, 80, qbase)
    for i in range(7):
        qrow = qb[qbase + i, :H * D].reshape(1, H * D)
        od = orc.decode(qrow, kc, vc, start + qbase + i, H, G, D, max_seq)
        assert np.max(np.abs(outp[qbase + i, :H * D] - od[0])) < 1e-12
    qf, kf, vf = _small(seed=15, q_seq=9, H=H, G=G, D=D)
    of, _ = orc.forward(qf, kf, vf, 9, 9, H, G, D, CAUSAL)
    op = orc.prefill(qf, kf, vf, 9, 9, H, G, D, G * D, 9, scale, 0, H * D, H * D, 0)
    assert np.max(np.abs(of - op)) < 1e-12


def pin_prefill_strides_and_clamp(orc):
    """Padding columns and rows before q_base stay untouched; a window that
    would pass max_seq is cut at max_seq (attention over all max_seq keys)."""
    H, G, D, max_seq = 2, 1, 16, 12
    qb, kc, vc = (_np(x) for x in synthetic.prefill_inputs(9, 40, max_seq, 24, seed=16))
    scale = np.float32(1.0 / math.sqrt(D))
    out = orc.prefill(qb, kc, vc, 9, 6, H, G, D, 24, max_seq, scale, 8, 40, 36, 2)
    assert np.all(np.isnan(out[:2])) and np.all(np.isnan(out[:, H * D:]))
    assert np.all(np.isfinite(out[2:8, :H * D]))
    # rows with start_pos + q_base + i + 1 >= max_seq see exactly max_seq keys
    kx = np.ascontiguousarray(kc[:, :D])
    vx = np.ascontiguousarray(vc[:, :D])
    qx = np.ascontiguousarray(qb[:, :H * D])
    ofull, _ = orc.forward(qx, kx, vx, 9, max_seq, H, 1, D, CROSS)
    for i in (2, 3, 5):        # positions 12, 13, 15 -> clamped to 12 keys
        assert np.max(np.abs(out[2 + i, :H * D] - ofull[2 + i])) < 1e-12


def pin_decode_clamp(orc):
    """kv_pos past the cache is cut at max_seq; kv_pos = 0 returns V[0]."""
    H, G, D, max_seq = 4, 2, 16, 10
    q, kc, vc = (_np(x) for x in synthetic.decode_inputs(max_seq, H, G, D, seed=17))
    a = orc.decode(q, kc, vc, 9, H, G, D, max_seq)
    b = orc.decode(q, kc, vc, 1000, H, G, D, max_seq)
    assert np.array_equal(a, b)
    z = orc.decode(q, kc, vc, 0, H, G, D, max_seq)
    for h in range(H):
        g = h // 2
        assert np.array_equal(z[0, h * D:(h + 1) * D], vc[0, g * D:(g + 1) * D].astype(np.float64))


def pin_prefill_scale_argument(orc):
    """The prefill scale argument multiplies the scores: scale 2/sqrt(D) on Q
    equals scale 1/sqrt(D) on 2Q (2Q is exact in fp32)."""
    H, G, D, max_seq = 2, 1, 16, 8
    qb, kc, vc = (_np(x) for x in synthetic.prefill_inputs(4, 32, max_seq, 16, seed=18))
    s1 = np.float32(1.0 / math.sqrt(D))
    a = orc.prefill(qb, kc, vc, 4, 4, H, G, D, 16, max_seq, np.float32(2.0 * s1), 4, 32, 32, 0)
    b = orc.prefill((2 * qb).astype(np.float32), kc, vc, 4, 4, H, G, D, 16, max_seq, s1, 4, 32, 32, 0)
    assert np.max(np.abs(a[:, :H * D] - b[:, :H * D])) < 1e-12
    c = orc.prefill(qb, kc, vc, 4, 4, H, G, D, 16, max_seq, s1, 4, 32, 32, 0)
    assert np.max(np.abs(a[:, :H * D] - c[:, :H * D])) > 1e-3



# ---------------------------------------------------------------- sliding window
def _sdpa_banded(q, k, v, q_seq, kv_seq, H, G, D, ends, window):
    """SDPA with an explicit boolean mask: row i attends keys [lo_i, ends[i]),
    lo_i = max(0, ends[i] - window) (window 0 = no lower bound)."""
    allow = np.zeros((q_seq, kv_seq), dtype=bool)
    for i, n in enumerate(ends):
        lo = max(0, n - window) if window > 0 else 0
        allow[i, lo:n] = True
    qt = torch.from_numpy(q.astype(np.float64)).reshape(q_seq, H, D).transpose(0, 1)[None]
    kt = torch.from_numpy(k.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None]
    vt = torch.from_numpy(v.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(allow), enable_gqa=True)
    return o[0].transpose(0, 1).reshape(q_seq, H * D).numpy()


def pin_window_sdpa_forward(orc):
    """Sliding window on all three masks against SDPA with a banded mask."""
    q, k, v = _small(seed=20, q_seq=13, kv_seq=13, H=4, G=2, D=16)
    for w in (1, 3, 5):
        out, _ = orc.forward(q, k, v, 13, 13, 4, 2, 16, CAUSAL, window=w)
        ref = _sdpa_banded(q, k, v, 13, 13, 4, 2, 16, [i + 1 for i in range(13)], w)
        assert np.max(np.abs(out - ref)) < 1e-12
        out, _ = orc.forward(q, k, v, 13, 13, 4, 2, 16, FULL, window=w)
        ref = _sdpa_banded(q, k, v, 13, 13, 4, 2, 16, [13] * 13, w)
        assert np.max(np.abs(out - ref)) < 1e-12
    q, k, v = _small(seed=21, q_seq=5, kv_seq=19, H=6, G=3, D=8)
    out, _ = orc.forward(q, k, v, 5, 19, 6, 3, 8, CROSS, window=7)
    ref = _sdpa_banded(q, k, v, 5, 19, 6, 3, 8, [19] * 5, 7)
    assert np.max(np.abs(out - ref)) < 1e-12


def pin_window_streaming_lse(orc):
    """The (max, log-sum) pair under a window follows the pages' recurrence run
    over the kept keys only."""
    q, k, v = _small(seed=22, q_seq=9, H=2, G=1, D=4, qk_sigma=3.0)
    w = 4
    out, lse = orc.forward(q, k, v, 9, 9, 2, 1, 4, CAUSAL, window=w)
    for pos in range(9):
        lo = max(0, pos + 1 - w)
        for h in range(2):
            ref, m, logl = _streaming_row(q[pos, h * 4:(h + 1) * 4], k[lo:pos + 1, :4], v[lo:pos + 1, :4], 0.5)
            assert np.max(np.abs(out[pos, h * 4:(h + 1) * 4] - np.array(ref))) < 1e-12
            assert abs(lse[pos, h, 0] - m) < 1e-12 and abs(lse[pos, h, 1] - logl) < 1e-12


def pin_window_one_is_last_v(orc):
    """window = 1 keeps only key n - 1: out = V[n-1] of the kv head, lse = (s, 0)."""
    q, k, v = _small(seed=23, q_seq=6, kv_seq=10, H=2, G=1, D=8)
    for mask, kv, ends in ((CAUSAL, 6, list(range(1, 7))), (CROSS, 10, [10] * 6)):
        kk, vv = k[:kv], v[:kv]
        out, lse = orc.forward(q, kk, vv, 6, kv, 2, 1, 8, mask, window=1)
        for pos, n in enumerate(ends):
            for h in range(2):
                assert np.array_equal(out[pos, h * 8:(h + 1) * 8], vv[n - 1, :8].astype(np.float64))
                s = float(np.dot(q[pos, h * 8:(h + 1) * 8].astype(np.float64),
                                 kk[n - 1, :8].astype(np.float64))) / math.sqrt(8)
                assert abs(lse[pos, h, 0] - s) < 1e-12 and lse[pos, h, 1] == 0.0


def pin_window_wide_is_no_window(orc):
    """A window at least as long as every row's window changes nothing."""
    q, k, v = _small(seed=24, q_seq=11, H=4, G=2, D=16)
    a = orc.forward(q, k, v, 11, 11, 4, 2, 16, CAUSAL)
    for w in (11, 12, 1000):
        b = orc.forward(q, k, v, 11, 11, 4, 2, 16, CAUSAL, window=w)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    c = orc.forward(q, k, v, 11, 11, 4, 2, 16, CAUSAL, window=10)
    assert np.array_equal(a[0][:10], c[0][:10]) and not np.array_equal(a[0][10], c[0][10])


def pin_window_decode_shifted_cache(orc):
    """Decode with window W at kv_pos p equals decode without one on the cache
    cut to start at p + 1 - W (the kept keys moved to the front)."""
    H, G, D, max_seq = 4, 2, 16, 30
    q, kc, vc = (_np(x) for x in synthetic.decode_inputs(max_seq, H, G, D, seed=25))
    for p, w in ((20, 6), (5, 6), (29, 1), (40, 4)):
        n = min(p + 1, max_seq)
        lo = max(0, n - w)
        a = orc.decode(q, kc, vc, p, H, G, D, max_seq, window=w)
        b = orc.decode(q, np.ascontiguousarray(kc[lo:]), np.ascontiguousarray(vc[lo:]),
                       n - 1 - lo, H, G, D, max_seq - lo)
        assert np.max(np.abs(a - b)) < 1e-15


def pin_window_prefill_matches_decode(orc):
    """Prefill row i with a window equals decode at kv_pos = start_pos + q_base + i
    with the same window, and differs from the unwindowed prefill."""
    H, G, D, max_seq = 4, 2, 16, 40
    qb, kc, vc = (_np(x) for x in synthetic.prefill_inputs(10, 80, max_seq, G * D, seed=26))
    start, qbase, w = 20, 3, 5
    scale = np.float32(1.0 / math.sqrt(D))
    outp = orc.prefill(qb, kc, vc, 10, 7, H, G, D, G * D, max_seq, scale, start, 80, 80, qbase, window=w)
    full = orc.prefill(qb, kc, vc, 10, 7, H, G, D, G * D, max_seq, scale, start, 80, 80, qbase)
    for i in range(7):
        qrow = qb[qbase + i, :H * D].reshape(1, H * D)
        od = orc.decode(qrow, kc, vc, start + qbase + i, H, G, D, max_seq, window=w)
        assert np.max(np.abs(outp[qbase + i, :H * D] - od[0])) < 1e-12
    assert np.max(np.abs(outp[qbase:qbase + 7, :H * D] - full[qbase:qbase + 7, :H * D])) > 1e-3



# ---------------------------------------------------------------- backward
def _grad_inputs(seed, q_seq, kv_seq, H, G, D):
    """Q, K, V and an upstream gradient dout, all N(0,1) fp32."""
    rng = np.random.default_rng(seed)
    f = lambda *sh: rng.standard_normal(sh).astype(np.float32)  # noqa: E731
    return f(q_seq, H * D), f(kv_seq, G * D), f(kv_seq, G * D), f(q_seq, H * D)


def _autograd(q, k, v, dout, q_seq, kv_seq, H, G, D, ends, window):
    """Gradients from PyTorch autograd through fp64 SDPA with a banded boolean mask."""
    allow = np.zeros((q_seq, kv_seq), dtype=bool)
    for i, n in enumerate(ends):
        allow[i, (max(0, n - window) if window > 0 else 0):n] = True
    qt = torch.from_numpy(q.astype(np.float64)).reshape(q_seq, H, D).transpose(0, 1)[None].requires_grad_()
    kt = torch.from_numpy(k.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None].requires_grad_()
    vt = torch.from_numpy(v.astype(np.float64)).reshape(kv_seq, G, D).transpose(0, 1)[None].requires_grad_()
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(allow), enable_gqa=True)
    go = torch.from_numpy(dout.astype(np.float64)).reshape(q_seq, H, D).transpose(0, 1)[None]
    o.backward(go)
    flat = lambda t, n, c: t.grad[0].transpose(0, 1).reshape(n, c).numpy()  # noqa: E731
    return flat(qt, q_seq, H * D), flat(kt, kv_seq, G * D), flat(vt, kv_seq, G * D)


def pin_backward_autograd(orc):
    """The three masks, with and without a sliding window, against autograd of SDPA."""
    for mask, q_seq, kv_seq, w in ((CAUSAL, 11, 11, 0), (FULL, 9, 9, 0), (CROSS, 6, 13, 0),
                                   (CAUSAL, 11, 11, 4), (CROSS, 6, 13, 5)):
        H, G, D = 6, 2, 8
        q, k, v, do = _grad_inputs(30 + mask + w, q_seq, kv_seq, H, G, D)
        got = orc.backward(q, k, v, do, q_seq, kv_seq, H, G, D, mask, window=w)
        ends = [i + 1 for i in range(q_seq)] if mask == CAUSAL else [kv_seq] * q_seq
        ref = _autograd(q, k, v, do, q_seq, kv_seq, H, G, D, ends, w)
        for a, b in zip(got, ref):
            assert np.max(np.abs(a - b)) < 1e-12


def pin_backward_finite_difference(orc):
    """Central differences of L = sum(dout * out) through the forward oracle.

    Inputs sit on a 2^-10 grid and the step is 2^-12, so x +- h is exact in
    fp32 and the difference quotient is accurate to O(h^2)."""
    H, G, D, n = 4, 2, 4, 7
    q, k, v, do = _grad_inputs(40, n, n, H, G, D)
    q, k, v = (np.round(x * 1024.0) / 1024.0 for x in (q, k, v))
    q, k, v = (x.astype(np.float32) for x in (q, k, v))
    dq, dk, dv = orc.backward(q, k, v, do, n, n, H, G, D, CAUSAL)
    h = 2.0 ** -12

    def loss(qq, kk, vv):
        out, _ = orc.forward(qq, kk, vv, n, n, H, G, D, CAUSAL)
        return float(np.sum(out * do.astype(np.float64)))

    for arr, grad, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        for idx in ((0, 0), (3, 5), (6, 7), (2, 3)):
            plus, minus = [x.copy() for x in (q, k, v)], [x.copy() for x in (q, k, v)]
            plus[which][idx] += np.float32(h)
            minus[which][idx] -= np.float32(h)
            assert plus[which][idx] - arr[idx] == np.float32(h)
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - grad[idx]) < 2e-6, (which, idx, fd, grad[idx])


def pin_backward_sums(orc):
    """Each row's softmax sums to 1 and its score gradient sums to 0, so over all
    keys of a kv head: sum_t dv_t = sum of dout over that head's query rows, and
    sum_t dk_t = 0 (any mask, any window)."""
    H, G, D = 8, 2, 16
    for mask, q_seq, kv_seq, w in ((CAUSAL, 20, 20, 0), (CROSS, 9, 30, 7), (FULL, 12, 12, 3)):
        q, k, v, do = _grad_inputs(50 + mask, q_seq, kv_seq, H, G, D)
        _, dk, dv = orc.backward(q, k, v, do, q_seq, kv_seq, H, G, D, mask, window=w)
        dsum = do.astype(np.float64).reshape(q_seq, G, H // G, D).sum(axis=(0, 2)).reshape(G * D)
        assert np.max(np.abs(dv.sum(axis=0) - dsum)) < 1e-11
        assert np.max(np.abs(dk.sum(axis=0))) < 1e-11


def pin_backward_window_one(orc):
    """window 1: each row copies one V row, so dq = dk = 0 and dv_t collects the
    dout of every query head of the group at the row that keeps key t."""
    H, G, D, n = 4, 2, 8, 6
    q, k, v, do = _grad_inputs(60, n, n, H, G, D)
    dq, dk, dv = orc.backward(q, k, v, do, n, n, H, G, D, CAUSAL, window=1)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    ref = do.astype(np.float64).reshape(n, G, H // G, D).sum(axis=2).reshape(n, G * D)
    assert np.max(np.abs(dv - ref)) < 1e-15


def pin_backward_gqa_is_summed_mha(orc):
    """GQA gradients of a shared kv head are the sums over its query heads of the
    MHA gradients with that head's K/V replicated."""
    H, G, D, n = 6, 2, 8, 10
    q, k, v, do = _grad_inputs(70, n, n, H, G, D)
    kr = np.repeat(k.reshape(n, G, D), H // G, axis=1).reshape(n, H * D)
    vr = np.repeat(v.reshape(n, G, D), H // G, axis=1).reshape(n, H * D)
    dq, dk, dv = orc.backward(q, k, v, do, n, n, H, G, D, CAUSAL)
    dq2, dk2, dv2 = orc.backward(q, kr, vr, do, n, n, H, H, D, CAUSAL)
    assert np.max(np.abs(dq - dq2)) < 1e-13
    assert np.max(np.abs(dk - dk2.reshape(n, G, H // G, D).sum(axis=2).reshape(n, G * D))) < 1e-13
    assert np.max(np.abs(dv - dv2.reshape(n, G, H // G, D).sum(axis=2).reshape(n, G * D))) < 1e-13



# ---------------------------------------------------------------- paged KV cache
def _paged_case(seed, max_blocks, page_rows, kv_dim, spare=3):
    """A contiguous cache, and a pool holding its pages shuffled among `spare`
    extra NaN pages, with the block table that maps them back."""
    rng = np.random.default_rng(seed)
    kc = rng.standard_normal((max_blocks * page_rows, kv_dim)).astype(np.float32)
    vc = rng.standard_normal((max_blocks * page_rows, kv_dim)).astype(np.float32)
    num_pages = max_blocks + spare
    where = rng.permutation(num_pages)[:max_blocks]  # pool page of logical page b
    kp = np.full((num_pages * page_rows, kv_dim), np.nan, np.float32)
    vp = np.full((num_pages * page_rows, kv_dim), np.nan, np.float32)
    for b in range(max_blocks):
        kp[where[b] * page_rows:(where[b] + 1) * page_rows] = kc[b * page_rows:(b + 1) * page_rows]
        vp[where[b] * page_rows:(where[b] + 1) * page_rows] = vc[b * page_rows:(b + 1) * page_rows]
    return kc, vc, kp, vp, where.astype(np.uint32)


def pin_paged_decode_equals_contiguous(orc):
    """Shuffled pages (with unused NaN pages in the pool) give the contiguous cache's bits,
    with and without a window."""
    H, G, D, P, nb = 4, 2, 16, 8, 5
    kc, vc, kp, vp, table = _paged_case(80, nb, P, G * D)
    q = np.random.default_rng(81).standard_normal((1, H * D)).astype(np.float32)
    for pos, w in ((0, 0), (17, 0), (39, 0), (39, 9), (100, 0)):
        a = orc.decode(q, kc, vc, pos, H, G, D, nb * P, window=w)
        b = orc.decode_paged(q, kp, vp, table, pos, H, G, D, P, window=w)
        assert np.array_equal(a, b)


def pin_paged_prefill_equals_contiguous(orc):
    H, G, D, P, nb = 4, 2, 16, 16, 4
    kc, vc, kp, vp, table = _paged_case(82, nb, P, G * D)
    qb = np.random.default_rng(83).standard_normal((12, H * D)).astype(np.float32)
    sc = np.float32(0.25)
    a = orc.prefill(qb, kc, vc, 12, 10, H, G, D, G * D, nb * P, sc, 30, H * D, H * D, 2)
    b = orc.prefill_paged(qb, kp, vp, table, 12, 10, H, G, D, G * D, P, sc, 30, H * D, H * D, 2)
    assert np.array_equal(a, b, equal_nan=True)


def pin_paged_shared_page(orc):
    """Two logical pages may map to one pool page (a shared prefix page): the
    result is that of the contiguous cache holding the page twice."""
    H, G, D, P = 2, 1, 8, 4
    rng = np.random.default_rng(84)
    kp = rng.standard_normal((2 * P, G * D)).astype(np.float32)
    vp = rng.standard_normal((2 * P, G * D)).astype(np.float32)
    table = np.array([1, 1, 0], np.uint32)
    kc = np.concatenate([kp[P:], kp[P:], kp[:P]])
    vc = np.concatenate([vp[P:], vp[P:], vp[:P]])
    q = rng.standard_normal((1, H * D)).astype(np.float32)
    a = orc.decode(q, kc, vc, 10, H, G, D, 3 * P)
    b = orc.decode_paged(q, kp, vp, table, 10, H, G, D, P)
    assert np.array_equal(a, b)



# ---------------------------------------------------------------- RoPE forward
def pin_rope_hand_worked(orc):
    """D = 4, base 100 (so the pair (1, 3) turns by 100^(-1/2) = 0.1 rad per
    position, the pair (0, 2) by 1 rad).  Query row 2 (position 2) is
    e0 + e1; key row 0 (position 0) is e2, key row 1 (position 1) is e0 + e3.
    Rotated: q' = (cos 2, cos 0.2, sin 2, sin 0.2), k0' = e2,
    k1' = (cos 1, -sin 0.1, sin 1, cos 0.1), so the scores (scale 1/2) are
    sin(2)/2 and (cos(1) + sin(0.1))/2; V rows are e0 and e1."""
    q = np.zeros((3, 4), np.float32)
    q[2] = [1, 1, 0, 0]
    k = np.array([[0, 0, 1, 0], [1, 0, 0, 1]], np.float32)
    v = np.eye(2, 4, dtype=np.float32)
    out, lse = orc.forward_rope(q, k, v, 3, 2, 1, 1, 4, CROSS, 100.0)
    s = np.array([math.sin(2.0), math.cos(1.0) + math.sin(0.1)]) / 2
    w = np.exp(s - s.max())
    assert np.max(np.abs(out[2] - np.array([w[0], w[1], 0, 0]) / w.sum())) < 1e-15
    assert abs(lse[2, 0, 0] - s.max()) < 1e-15 and abs(lse[2, 0, 1] - math.log(w.sum())) < 1e-15


def _rope_complex(x, H, D, base):
    """Rotate [rows, H*D] with row r at position r, pairs (i, i + D/2) as the
    complex numbers x_i + i x_(i+D/2) multiplied by exp(i r base^(-2i/D))."""
    rows = x.shape[0]
    xt = torch.from_numpy(x.astype(np.float64)).reshape(rows, H, D)
    z = torch.complex(xt[..., :D // 2], xt[..., D // 2:])
    ang = torch.arange(rows, dtype=torch.float64)[:, None] * \
        torch.pow(torch.tensor(base, dtype=torch.float64), -2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
    z = z * torch.polar(torch.ones_like(ang), ang)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1).reshape(rows, H * D).numpy()


def pin_rope_complex_sdpa(orc):
    """Causal and cross RoPE forwards against SDPA on q, k rotated as complex pairs."""
    for mask, q_seq, kv_seq, w in ((CAUSAL, 12, 12, 0), (CROSS, 7, 15, 0), (CAUSAL, 12, 12, 5)):
        H, G, D = 6, 2, 8
        q, k, v = _small(seed=90 + mask + w, q_seq=q_seq, kv_seq=kv_seq, H=H, G=G, D=D)
        out, _ = orc.forward_rope(q, k, v, q_seq, kv_seq, H, G, D, mask, 10000.0, window=w)
        qr, kr = _rope_complex(q, H, D, 10000.0), _rope_complex(k, G, D, 10000.0)
        ends = [i + 1 for i in range(q_seq)] if mask == CAUSAL else [kv_seq] * q_seq
        ref = _sdpa_banded(qr, kr, v, q_seq, kv_seq, H, G, D, ends, w)
        assert np.max(np.abs(out - ref)) < 1e-12


def pin_rope_gqa_equals_replicated_mha(orc):
    q, k, v = _small(seed=95, q_seq=10, H=8, G=2, D=16)
    out, lse = orc.forward_rope(q, k, v, 10, 10, 8, 2, 16, CAUSAL, 500.0)
    kr = np.repeat(k.reshape(10, 2, 16), 4, axis=1).reshape(10, 8 * 16)
    vr = np.repeat(v.reshape(10, 2, 16), 4, axis=1).reshape(10, 8 * 16)
    out2, lse2 = orc.forward_rope(q, kr, vr, 10, 10, 8, 8, 16, CAUSAL, 500.0)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)



def pin_rope_backward_autograd(orc):
    """The RoPE backward against autograd through the complex-pair rotation and
    fp64 SDPA (causal, cross with a window)."""
    for mask, q_seq, kv_seq, w in ((CAUSAL, 10, 10, 0), (CROSS, 6, 11, 4)):
        H, G, D = 4, 2, 8
        q, k, v, do = _grad_inputs(110 + mask, q_seq, kv_seq, H, G, D)
        got = orc.backward_rope(q, k, v, do, q_seq, kv_seq, H, G, D, mask, 500.0, window=w)

        def turned(x, heads):
            rows = x.shape[0]
            xt = x.reshape(rows, heads, D)
            z = torch.complex(xt[..., :D // 2], xt[..., D // 2:])
            ang = torch.arange(rows, dtype=torch.float64)[:, None] * torch.pow(
                torch.tensor(500.0, dtype=torch.float64), -2.0 * torch.arange(D // 2, dtype=torch.float64) / D)
            z = z * torch.polar(torch.ones_like(ang), ang)[:, None, :]
            return torch.cat([z.real, z.imag], dim=-1).reshape(rows, heads * D)

        qt = torch.from_numpy(q.astype(np.float64)).requires_grad_()
        kt = torch.from_numpy(k.astype(np.float64)).requires_grad_()
        vt = torch.from_numpy(v.astype(np.float64)).requires_grad_()
        allow = np.zeros((q_seq, kv_seq), dtype=bool)
        for i in range(q_seq):
            n = i + 1 if mask == CAUSAL else kv_seq
            allow[i, (max(0, n - w) if w else 0):n] = True
        qs = turned(qt, H).reshape(q_seq, H, D).transpose(0, 1)[None]
        ks = turned(kt, G).reshape(kv_seq, G, D).transpose(0, 1)[None]
        vs = vt.reshape(kv_seq, G, D).transpose(0, 1)[None]
        o = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=torch.from_numpy(allow), enable_gqa=True)
        o.backward(torch.from_numpy(do.astype(np.float64)).reshape(q_seq, H, D).transpose(0, 1)[None])
        for a, b in zip(got, (qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy())):
            assert np.max(np.abs(a - b)) < 1e-12


ALL_PINS = [obj for name, obj in sorted(globals().items()) if name.startswith("pin_")]
