"""Failure detection on the GPU without a fault: a bounded wait inside a
kernel that runs out reports PA_DEV_TIMEOUT in the status word, and the
context stays usable for the next calls (a decode step after it is still
correct)."""

import time

import pytest
import torch

from paged_kv_gqa_rope_gb300 import pa
from tests.gpu_helpers import DecodeRun, assert_attention_close, oracle_decode_step
from tests.test_gpu_decode import custom_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(libpa):
    assert torch.cuda.is_available()
    assert pa.check_device() == pa.PA_OK
    return libpa


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    st = pa.new_status()
    t0 = time.perf_counter()
    pa.selftest_wait_timeout(st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == pa.PA_DEV_TIMEOUT
    assert 0.5 < dt < 30.0
    # the context is usable: a decode step afterwards is correct
    case, init = custom_case(8, 2, 128, [100, 1000], seed=31)
    run = DecodeRun(case, init)
    out = run.run()
    assert int(run.status.item()) == 0
    _, _, _, want = oracle_decode_step(case, init)
    assert_attention_close(out, want)
