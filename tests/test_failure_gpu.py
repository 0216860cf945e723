"""The kernels' failure path on the GPU, without faulting it: a bounded wait
on a barrier that nothing completes gives up, records ATTN_ERR_TIMEOUT in the
status word, and leaves the context usable for the next call."""
import pytest
import torch

from attention_gqa_online_gb300 import synthetic
from helpers import FP32, assert_out_close, dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives(cuda_lib, orc):
    assert cuda_lib.attn_get_status() == 0
    cuda_lib.attn_selftest_wait_timeout(20000)          # 20 ms limit
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == cuda_lib.ATTN_ERR_TIMEOUT
    assert cuda_lib.attn_get_status() == 0              # reading clears it
    # the context is intact: a normal call still runs and is correct
    q, k, v = synthetic.forward_inputs(40, 40, 4, 2, 64, seed=31)
    out, lse = cuda_lib.forward(dev(q), dev(k), dev(v), 4, 2, cuda_lib.ATTN_CAUSAL, cuda_lib.ATTN_FP32)
    torch.cuda.synchronize()
    assert cuda_lib.attn_get_status() == 0
    ro, _ = orc.forward(q.numpy(), k.numpy(), v.numpy(), 40, 40, 4, 2, 64, 0)
    assert_out_close(out.cpu().numpy(), ro, FP32, float(v.abs().max()), "after timeout")


def test_selftest_rejects_bad_limits(cuda_lib):
    with pytest.raises(cuda_lib.AttnError):
        cuda_lib.attn_selftest_wait_timeout(0)
    with pytest.raises(cuda_lib.AttnError):
        cuda_lib.attn_selftest_wait_timeout(2000000)
