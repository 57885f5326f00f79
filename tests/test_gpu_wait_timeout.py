"""Failure detection without a GPU fault: the kernels' bounded mbarrier waits
(single-CTA and CTA-pair forms) give up after their budget, report
FLCE_DEVERR_TIMEOUT through the error word and return, and the context stays
usable. The self-test waits on a barrier that nothing arrives on, with a
50 ms budget; nothing traps, faults or spins without bound."""
import time

import pytest
import torch

from _parity import to_dev
from linear_cross_entropy_vocab_gb300 import abi, api
from linear_cross_entropy_vocab_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    res = torch.full((3,), 7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    abi.flce_selftest_wait_timeout(err.data_ptr(), res.data_ptr(), 0.05,
                                   torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(err.item()) & abi.FLCE_DEVERR_TIMEOUT
    assert res.tolist() == [0, 0, 0]
    assert 0.05 <= dt < 5.0, dt
    # the context is still usable: a forward runs and reports no error
    w = Workload("after_timeout", 256, 128, 1000, "bf16")
    x = to_dev(make_inputs(w))
    err2 = torch.zeros((), dtype=torch.int32, device="cuda")
    out = api.flce_forward_tensors(x["hidden"], x["weight"], x["targets"], err_word=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    assert torch.isfinite(out["loss"]).item()


def test_selftest_argument_checks():
    err = torch.zeros((), dtype=torch.int32, device="cuda")
    res = torch.zeros((3,), dtype=torch.int32, device="cuda")
    for bad in (0.0, -1.0, 2.0):
        st = abi.flce_selftest_wait_timeout(err.data_ptr(), res.data_ptr(), bad, None, check=False)
        assert st == abi.FLCE_ERR_INVALID_ARG
