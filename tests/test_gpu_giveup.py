"""The give-up path of the single-pass tensor-core forward, without a fault.

The kernel's CTAs wait on one another's published segment states, each wait
bounded.  A test hook shortens the limit to 1 ms and withholds the publication
of one segment, so that its successors' look-backs run out of time: the launch
must end by itself, report LA_ERR_TIMEOUT through la_get_device_status, and
leave the context usable -- the next normal forward matches the oracle.
"""
import pytest
import torch

import oracle
from gpu_util import TOL, rel_err_rows, to_np

pytestmark = pytest.mark.gpu

la = pytest.importorskip("kernelised_causal_linear_gb300")
from kernelised_causal_linear_gb300 import synth  # noqa: E402

LA_ERR_TIMEOUT = 4


@pytest.fixture(autouse=True)
def _restore_hooks():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    yield
    la.la_debug_set_tc_faults(2_000_000_000, -1)


def test_withheld_segment_times_out_then_recovers():
    # eight sequences keep the call on the single-pass kernel; 64 chunks each
    w = synth.Workload("giveup", 1, 8, 8192, 64, 64, torch.bfloat16, seed_id=80)
    assert la.la_forward_path(w.B, w.H, w.N, 64, 64, True, "elu1", False, w.dtype) == "tcgen05"
    q, k, v = synth.qkv(w, device="cuda")
    assert la.la_get_device_status() == 0
    la.la_debug_set_tc_faults(1_000_000, 100)  # 1 ms; withhold ticket 100
    out = la.la_forward(q, k, v)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == LA_ERR_TIMEOUT
    assert la.la_get_device_status() == 0  # read and cleared
    # back to the library's behaviour: the same call is complete and correct
    la.la_debug_set_tc_faults(2_000_000_000, -1)
    out = la.la_forward(q, k, v)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    ref = oracle.load().forward(to_np(q), to_np(k), to_np(v))
    assert rel_err_rows(out, ref) <= TOL[torch.bfloat16]


def test_short_limit_alone_changes_nothing():
    """A 1 ms limit with nothing withheld: every wait of a small launch ends
    well inside it."""
    w = synth.Workload("giveup2", 1, 8, 4096, 64, 64, torch.bfloat16, seed_id=81)
    q, k, v = synth.qkv(w, device="cuda")
    la.la_debug_set_tc_faults(1_000_000, -1)
    out = la.la_forward(q, k, v)
    torch.cuda.synchronize()
    assert la.la_get_device_status() == 0
    ref = oracle.load().forward(to_np(q), to_np(k), to_np(v))
    assert rel_err_rows(out, ref) <= TOL[torch.bfloat16]
