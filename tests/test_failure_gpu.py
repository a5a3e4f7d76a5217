"""Failure detection on the GPU without a fault: every wait in the kernels is bounded and ends
with an error status instead of a hang.  The library's self-test waits on a barrier that nothing
arrives at, with a 20 ms limit; the status word must show the timeout and the context must stay
usable (a prefill right after it still matches the oracle)."""

import pytest
import torch

from fa_workloads import PrefillCase, make_prefill
from tests._util import check, gather_prefill_rows, oracle_prefill_rows, sample_rows

pytestmark = pytest.mark.gpu


def test_wait_that_never_completes_reports_timeout_and_context_survives():
    import flashattention_forward_fa_gb300 as fa
    fa.fa_device_status(clear=True)
    fa.fa_selftest_wait_timeout(20)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) & 1, "the timed-out wait did not set the timeout bit"
    assert fa.fa_device_status(clear=True) == 0, "reading the status did not clear it"
    case = PrefillCase("after_timeout", B=1, Hq=2, Hkv=2, Nq=300, Nk=300, d=128, causal=True, seed=601)
    x = make_prefill(case)
    o, lse = fa.fa_fwd(x.q.cuda(), x.k.cuda(), x.v.cuda(), causal=True)
    torch.cuda.synchronize()
    rows = sample_rows(x, 40)
    go, gl = gather_prefill_rows(x, o, lse, rows)
    ro, rl = oracle_prefill_rows(x, rows)
    check(go, gl, ro, rl, case.name)
    assert fa.fa_device_status() == 0
