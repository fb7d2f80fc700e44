"""Failure detection without a GPU fault: a bounded device wait that nothing
satisfies gives up, the host reads TE_MX_ERR_DEVICE_TIMEOUT from the status
word, and the context stays usable for the next call."""
import numpy as np
import pytest
import torch

from mxfp8_block_scaled_quantize_gb300 import binding
from oracle import mx_oracle as O
from tests import _util as U

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    binding.te_mx_device_status()                       # start clean
    binding.te_mx_selftest_timeout(2000)                # 2 ms wait on a flag nothing sets
    with pytest.raises(binding.TemxError, match="DEVICE_TIMEOUT"):
        binding.te_mx_device_status()
    binding.te_mx_device_status()                       # the word was cleared
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    got = U.gpu_quantize(x.cuda(), True, False)         # the context still works
    q, s = O.quantize_rowwise(U.bf16_bits(x))
    assert np.array_equal(got["q_row"], q) and np.array_equal(got["s_row"], s)


def test_selftest_rejects_bad_limits():
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_selftest_timeout(0)
    with pytest.raises(binding.TemxError, match="INVALID_ARG"):
        binding.te_mx_selftest_timeout(3_000_000)
