"""The failure path of the pipeline's bounded waits, driven on the GPU without
any fault: dsa_selftest_wait_timeout makes one CTA wait, with a 1 ms limit, on
an mbarrier that nothing arrives on.  The wait must give up, raise
DSA_ERR_TIMEOUT through the context's error word, end the CTA's next wait at
once through the abort flag, free its tensor memory and exit; afterwards the
context must still compute correctly (mstar IndexKeyStore.history: failures
are reported to the caller, not fatal)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from deepseek_sparse_attention_dsa_gb300 import dsa
from deepseek_sparse_attention_dsa_gb300 import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

DSA_ERR_INVALID_ARG = 1
DSA_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def built():
    from deepseek_sparse_attention_dsa_gb300 import build
    build.build()


def _selftest(ctx, limit_ns, result):
    L = dsa.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = ctypes.c_void_p(result.data_ptr()) if result is not None else None
    return L.dsa_selftest_wait_timeout(ctx.handle, ctypes.c_uint64(limit_ns), ptr, stream)


def test_wait_times_out_reports_and_leaves_the_context_usable():
    wl = H.deepseek_small(seed=41, decode_ctx=(3000, 2100), chunk=(2100, 12))
    ctx = dsa.Context(wl.shape, 0)
    L = dsa.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    limit_ns = 1_000_000
    for _ in range(2):   # a second time on the same context: the error word was cleared in between
        result = torch.full((5,), -1, dtype=torch.int64, device="cuda")
        assert _selftest(ctx, limit_ns, result) == dsa.DSA_OK
        assert L.dsa_get_error(ctx.handle, stream) == DSA_ERR_TIMEOUT
        assert L.dsa_get_error(ctx.handle, stream) == dsa.DSA_OK   # read and cleared
        first_ok, first_ns, second_ok, second_ns, abort_flag = result.cpu().tolist()
        assert first_ok == 0 and second_ok == 0 and abort_flag == 1
        assert limit_ns <= first_ns < limit_ns + 250_000_000, first_ns
        assert second_ns < limit_ns, second_ns   # ended by the abort flag, not by its own limit

    # the same context still computes the step correctly
    ic, lc, st = H.host_inputs(wl)
    ref = oracle.run_all(wl, ic, lc, st)
    dev = W.StepInputs(*(H.to_dev(x) for x in (st.q, st.w, st.keys, st.q_nope, st.q_pe, st.sink)))
    got = H.gpu_pipeline(ctx, wl, ic.cuda(), lc.cuda(), dev)
    H.check_selection(got["selection"], ref["selection"], ref["scores"], ref["offsets"], wl.shape.topk)
    ref_e2e = oracle.attend(wl.shape, wl.spans, wl.num_pages, got["selection"], st.q_nope, st.q_pe, lc, st.sink)
    H.check_attention(got["out"], ref_e2e)


def test_selftest_rejects_bad_arguments():
    ctx = dsa.Context(W.DSAShape(**W.DEEPSEEK), 0)
    result = torch.zeros(5, dtype=torch.int64, device="cuda")
    assert _selftest(ctx, 0, result) == DSA_ERR_INVALID_ARG
    assert _selftest(ctx, 2_000_000_000, result) == DSA_ERR_INVALID_ARG
    assert _selftest(ctx, 1000, None) == DSA_ERR_INVALID_ARG
    assert int(np.count_nonzero(result.cpu().numpy())) == 0   # nothing ran
