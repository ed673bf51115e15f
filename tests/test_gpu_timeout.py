"""Failure detection on the GPU without a GPU fault: a bounded wait runs out.

A host-set fault (svw_set_fault) leaves CTA 0 of spec_verify's stats kernel,
or cluster 0 of the OPD fast kernel (opd_loss, spec_verify_opd), without its
bulk copies, and the kernels' wait deadline is shortened (svw_set_wait_limit,
about 0.5 ms) so that the test is quick.  The wait for that first copy runs
out with no copy in flight: the call returns, the status word holds
SVW_DEV_TIMEOUT, and afterwards (fault cleared, default deadline) the same
call on the same GPU gives bit-identical results to the call before.
"""
import numpy as np
import pytest

import synth
from helpers import to_torch_i32, to_torch_logits

pytestmark = pytest.mark.gpu

SHORT_WAIT = 1_000_000  # SM cycles: far above a healthy wait (microseconds), far below the default


@pytest.fixture(autouse=True)
def _hooks():
    import torch
    import serving_vocab_wide_gb300 as svw
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    svw.build()
    svw.lib()
    yield
    svw.set_fault(0)
    svw.set_wait_limit()


def _inputs(T=1.0):
    b = synth.config(5, N=16, V=32768, seed=7)
    return b, (to_torch_logits(b.target), to_torch_logits(b.draft), to_torch_i32(b.cu),
               to_torch_i32(b.tokens[float(T)]))


def _run_three(call):
    """call(status) before, under and after the fault; returns the results and status words."""
    import torch
    import serving_vocab_wide_gb300 as svw
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = [x.clone() for x in call(st)]
    torch.cuda.synchronize()
    s0 = int(st.item())
    svw.set_wait_limit(SHORT_WAIT)
    svw.set_fault(1)
    st.zero_()
    call(st)
    torch.cuda.synchronize()
    s1 = int(st.item())
    svw.set_fault(0)
    svw.set_wait_limit()
    st.zero_()
    after = [x.clone() for x in call(st)]
    torch.cuda.synchronize()
    s2 = int(st.item())
    return before, after, (s0, s1, s2)


def _assert_recovered(before, after, words):
    import serving_vocab_wide_gb300 as svw
    s0, s1, s2 = words
    assert s0 == 0 and s2 == 0, words
    assert s1 & svw.SVW_DEV_TIMEOUT, f"status {s1:#x}: no timeout reported"
    assert svw.device_status(s1) == svw.SVW_ERR_TIMEOUT
    for x, y in zip(before, after):
        assert np.array_equal(x.cpu().numpy(), y.cpu().numpy(), equal_nan=True)


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_spec_verify_wait_runs_out(T):
    import serving_vocab_wide_gb300 as svw
    b, (t, d, cu, tok) = _inputs(T)

    def call(st):
        return svw.spec_verify(t, d, cu, tok, T, b.seed, max_len=16, total_draft_rows=b.total_rows, status=st)

    _assert_recovered(*_run_three(call))


def test_opd_loss_wait_runs_out():
    import serving_vocab_wide_gb300 as svw
    b = synth.config(4, N=8, V=32768, seed=9)
    t, d = to_torch_logits(b.target), to_torch_logits(b.draft)

    def call(st):
        return svw.opd_loss(t, d, status=st)

    _assert_recovered(*_run_three(call))


def test_spec_verify_opd_wait_runs_out():
    import serving_vocab_wide_gb300 as svw
    b, (t, d, cu, tok) = _inputs(1.0)

    def call(st):
        return svw.spec_verify_opd(t, d, cu, tok, 1.0, b.seed, max_len=16, total_draft_rows=b.total_rows,
                                   status=st)

    _assert_recovered(*_run_three(call))
