"""Device-side failure detection on the GPU, without a fault.

Every hand-off inside the library's kernels is a bounded mbarrier wait: when the limit runs out
the kernel sets MSA_DEVICE_TIMEOUT in the workspace's status word and leaves, so the host sees an
error code instead of a hung GPU.  Here that path runs on purpose through the library's self-test
(one thread waits on a barrier that nothing arrives at), and the same context then has to run a
forward and backward that match the oracle.
"""
import pytest
import torch

from block_sparse_attention_qp_gb300 import binding as msa
from block_sparse_attention_qp_gb300.inputs import Workload
from tests.test_gpu_parity import run_sparse

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MSA_DEVICE_TIMEOUT = 4


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    assert msa.msa_device_status(ws) == 0
    msa.selftest_wait_timeout(ws, limit_us=2000)
    assert msa.msa_device_status(ws) == MSA_DEVICE_TIMEOUT
    assert msa.msa_device_status(ws) == 0  # the read clears the word
    # the context still computes: a small sparse step against the oracle
    run_sparse(Workload("after_timeout", B=1, S=512, Hq=8, Hkv=2, Hp=2, top_k=3), 177)


def test_selftest_argument_errors():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    for bad in (0, 2_000_000):
        with pytest.raises(msa.MSAError, match="invalid argument"):
            msa.selftest_wait_timeout(ws, limit_us=bad)
    assert msa.msa_device_status(ws) == 0  # nothing was launched
