"""Failure detection on the GPU without a fault: the kernels' bounded pipeline wait is run out on
purpose (an mbarrier that nothing arrives on, a short poll limit) and must end in an error status
the host reads, with the context still usable afterwards."""
import ctypes

import pytest
import torch

import workloads as W
from tests.kda_harness import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_pipeline_wait_runs_out_and_the_host_reads_the_timeout():
    import gated_linear_attention_kda_gb300 as kda
    kda.check_device_status()  # nothing pending from earlier tests
    res = kda.probe_wait_timeout(4096)
    # both waits gave up; the first one to run out set the CTA's abort flag
    assert res == [0, 0, 1]
    with pytest.raises(kda.KDAError, match="KDA_ERR_DEVICE"):
        kda.check_device_status()
    assert b"pipeline wait timed out" in kda.library().kda_last_error()
    kda.check_device_status()  # the word was read and cleared in one step


def test_context_stays_usable_after_a_wait_ran_out():
    import gated_linear_attention_kda_gb300 as kda
    kda.probe_wait_timeout(256)
    with pytest.raises(kda.KDAError):
        kda.check_device_status()
    d = W.make("b2_t128_h8", T=45)
    o, s = run_gpu(d)  # checks the device status itself: clean
    o_ref, s_ref = run_oracle(d)
    assert_close("out", o, o_ref)
    assert_close("final_state", s, s_ref)
