"""Failure handling on the GPU without a fault: a bounded wait that runs out.

Every spin-wait in the library's kernels is bounded; when one gives up it raises
its block's abort flag and the GATTN_DEVICE_TIMEOUT status bit, the block's other
roles leave their waits on that flag, and the kernel returns.  The self-test entry
point runs that machinery on an mbarrier nothing arrives on, with a 1 ms limit;
the test checks the status, the wait's duration, and that the CUDA context still
computes a correct prefill afterwards.  Nothing faults, traps or waits without a
limit.
"""
import ctypes

import pytest
import torch

import oracle
from gated_softmax_attention_gqa_gb300 import (_lib, gattn_get_device_status, gattn_prefill,
                                               gattn_selftest_wait_timeout)
from gated_softmax_attention_gqa_gb300.workloads import Workload, make_prefill_inputs
from tests.parity import assert_close_to_oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TIMEOUT_BIT = 0x2
ERR_DEVICE_TIMEOUT = 6


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    torch.cuda.set_device(0)
    gattn_get_device_status()  # start from a clear status word
    waited = torch.zeros(1, dtype=torch.int64, device=DEV)
    limit = 1_000_000  # 1 ms
    gattn_selftest_wait_timeout(limit, waited)
    torch.cuda.synchronize()
    # the C entry point reports the timeout as its own status, then clears the word
    bits = ctypes.c_uint(0)
    st = _lib.load().gattn_get_device_status(ctypes.byref(bits),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ERR_DEVICE_TIMEOUT and bits.value & TIMEOUT_BIT, (st, bits.value)
    assert gattn_get_device_status() == 0
    ns = int(waited.item())
    assert limit <= ns < 50 * limit, ns  # gave up after the limit, long before the kernels' own 2 s

    # the context is intact: a prefill right after matches the oracle
    w = Workload("after", "prefill", B=1, S=300, H=8, G=2, d=128, rotary_dim=64, rope_base=1e6,
                 gate_mode="elementwise", dtype="bf16", seed=17)
    inp = make_prefill_inputs(w)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out = gattn_prefill(d["q"], d["k"], d["v"], d["gate"], d["qnorm_w"], d["knorm_w"], rotary_dim=w.rotary_dim,
                        rope_base=w.rope_base, eps=w.eps, gate_mode=w.gate_mode)
    torch.cuda.synchronize()
    ref = oracle.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], inp["qnorm_w"], inp["knorm_w"], None,
                         w.rotary_dim, w.rope_base, w.eps, w.gate_mode)
    assert_close_to_oracle(out, ref, torch.bfloat16, "prefill after a timed-out wait")
    assert gattn_get_device_status() == 0


def test_selftest_twice_in_a_row():
    """The self-test leaves nothing behind: a second run times out the same way."""
    for _ in range(2):
        gattn_selftest_wait_timeout(2_000_000)
        torch.cuda.synchronize()
        assert gattn_get_device_status() & TIMEOUT_BIT
    assert gattn_get_device_status() == 0
