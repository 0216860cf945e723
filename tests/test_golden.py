"""Closed-form fixtures (tests/golden/closed_forms.json, written by
tests/golden/make_golden.py from formulas worked by hand) against the oracle
(CPU) and the CUDA library (GPU, fp32 path)."""
import json
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = json.load(open(os.path.join(HERE, "golden", "closed_forms.json")))


def arr(x, cols):
    a = np.asarray(x, dtype=np.float32)
    return a.reshape(-1, cols) if a.size else np.zeros((0, cols), np.float32)


def inputs(c):
    H, G, D = c["H"], c["G"], c["D"]
    return arr(c["q"], H * D), arr(c["k"], G * D), arr(c["v"], G * D)


def test_oracle_forward_cases(orc):
    for name in ("three_keys", "empty_cross"):
        c = CASES[name]
        q, k, v = inputs(c)
        out, lse = orc.forward(q, k, v, c["q_seq"], c["kv_seq"], c["H"], c["G"], c["D"], c["mask"])
        assert np.max(np.abs(out - np.asarray(c["out"]))) < 1e-15, name
        assert np.max(np.abs(lse - np.asarray(c["lse"]))) < 1e-15, name


def test_oracle_rope_case(orc):
    c = CASES["rope_d4"]
    q, k, v = inputs(c)
    out, lse = orc.forward_rope(q, k, v, c["q_seq"], c["kv_seq"], c["H"], c["G"], c["D"], c["mask"], c["base"])
    assert np.max(np.abs(out[c["row"]] - np.asarray(c["out_row"]))) < 1e-15
    assert np.max(np.abs(lse[c["row"], 0] - np.asarray(c["lse_row"]))) < 1e-15


def test_oracle_backward_case(orc):
    c = CASES["backward_d1"]
    q, k, v = inputs(c)
    dq, dk, dv = orc.backward(q, k, v, arr(c["dout"], 1), 1, 2, 1, 1, 1, c["mask"])
    for got, want in ((dq, c["dq"]), (dk, c["dk"]), (dv, c["dv"])):
        assert np.max(np.abs(got - np.asarray(want))) < 1e-15


@pytest.mark.gpu
def test_library_cases(cuda_lib):
    """The fp32 path on the same fixtures (head dims 4 and 1 run on the CUDA-core kernels)."""
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    for name in ("three_keys", "empty_cross"):
        c = CASES[name]
        q, k, v = inputs(c)
        out = torch.full((c["q_seq"], c["H"] * c["D"]), float("nan"), device="cuda")
        lse = torch.full((c["q_seq"], c["H"], 2), float("nan"), device="cuda")
        cuda_lib.attn_forward(dev(q), dev(k) if c["kv_seq"] else None, dev(v) if c["kv_seq"] else None, out, lse,
                              c["q_seq"], c["kv_seq"], c["H"], c["G"], c["D"], c["mask"], cuda_lib.ATTN_FP32)
        torch.cuda.synchronize()
        assert np.max(np.abs(out.cpu().numpy() - np.asarray(c["out"]))) < 1e-6, name
        # -1e30 is stored in fp32 (relative rounding 6e-8)
        assert np.allclose(lse.cpu().numpy(), np.asarray(c["lse"]), rtol=1e-6, atol=1e-6), name
