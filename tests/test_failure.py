"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies must end with FA_ERR_DEVICE_TIMEOUT and leave the context usable."""
import pytest
import torch

from flash_attention_gqa_gb300 import binding, inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    dev = torch.device("cuda")
    assert binding.fa_set_wait_limit_ns(50_000_000) == binding.FA_OK   # 50 ms
    try:
        assert binding.fa_selftest_wait_timeout() == binding.FA_ERR_DEVICE_TIMEOUT
        # the error word was read and cleared
        assert binding.fa_check_status() == binding.FA_OK
    finally:
        assert binding.fa_set_wait_limit_ns(2_000_000_000) == binding.FA_OK
    # the context still runs real work correctly
    x = inputs.make_tensors(1, 1, 4, 256, 256, 128, seed=3, backward=False)
    o, lse = binding.attention_forward(x.q.to(dev), x.k.to(dev), x.v.to(dev), causal=True)
    torch.cuda.synchronize()
    assert binding.fa_check_status() == binding.FA_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_device_sm_count():
    n = binding.fa_device_sm_count()
    assert n == torch.cuda.get_device_properties(0).multi_processor_count
