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


# The prefill kernel's own abort path: each CTA's V loads stop after two tiles, so the MMA
# issuer's wait for the third gives up (2 s) and every role unwinds — including the P handoffs,
# named barriers without a time limit that both sides complete without work.  The kernel must
# end with the timeout bit, and a normal prefill right after it must match the oracle.
ABORT_CASES = [
    dict(name="abort_d128_causal", B=1, Hq=4, Hkv=4, Nq=1024, Nk=1024, d=128, causal=True),
    dict(name="abort_d64_alibi_gqa", B=2, Hq=8, Hkv=2, Nq=640, Nk=640, d=64, causal=False, alibi=True),
    dict(name="abort_d128_window_rope", B=1, Hq=4, Hkv=2, Nq=900, Nk=900, d=128, causal=True, window=300,
         rope=True),
]


@pytest.mark.parametrize("cfg", ABORT_CASES, ids=[c["name"] for c in ABORT_CASES])
def test_prefill_abort_path_ends_with_timeout_and_context_survives(cfg):
    import flashattention_forward_fa_gb300 as fa
    case = PrefillCase(cfg["name"], B=cfg["B"], Hq=cfg["Hq"], Hkv=cfg["Hkv"], Nq=cfg["Nq"], Nk=cfg["Nk"],
                       d=cfg["d"], causal=cfg["causal"], window=cfg.get("window", 0), seed=611)
    x = make_prefill(case)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    slopes = fa.alibi_slopes(case.Hq) if cfg.get("alibi") else None
    rope = fa.rope_tables(case.Nk, case.d, device="cuda") if cfg.get("rope") else None
    fa.fa_device_status(clear=True)
    fa.fa_selftest_prefill_abort(q, k, v, 2, causal=case.causal, window=case.window, alibi_slopes=slopes, rope=rope)
    assert fa.fa_device_status(clear=True) & 1, "the stalled prefill did not report a timeout"
    o, lse = fa.fa_fwd(q, k, v, causal=case.causal, window=case.window)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    rows = sample_rows(x, 48)
    go, gl = gather_prefill_rows(x, o, lse, rows)
    ro, rl = oracle_prefill_rows(x, rows)
    check(go, gl, ro, rl, case.name)
