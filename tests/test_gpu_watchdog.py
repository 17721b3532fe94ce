"""The device-side watchdog: a bounded wait that runs out reports
LI_ERR_TIMEOUT through the status word and leaves the context usable.

The wait is made to run out by a barrier that nothing arrives on (the test
kernel li_selftest_wait_timeout); nothing faults, traps or hangs."""
import time

import pytest

import li_inputs
from parity import RTOL, assert_scores_close, assert_topk_row

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_wait_that_runs_out_reports_timeout_and_context_survives(li, orc):
    assert li.li_device_status() == 0
    t0 = time.perf_counter()
    assert li.li_selftest_wait_timeout(20000) == 0           # 20 ms limit
    assert li.li_device_status() == -6                        # LI_ERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.015 <= waited < 5.0                              # gave up after its limit
    assert li.li_device_status() == 0                         # read-and-clear
    # the same context still runs the scan and returns the oracle's results
    w = li_inputs.spec("fp8_32k_b32", B=2, L=700, native=False)
    x = li_inputs.make_workload(w, seed=7)
    qa, qs = li.absorb_queries(x["q"].to(DEV), x["D"].to(DEV), "fp8")
    s = li.score_group(x["latent"].to(DEV), x["lat_scale"].to(DEV), qa, qs, x["w"].to(DEV))
    idx = li.topk(s, w.k)
    assert li.li_device_status() == 0
    o = orc.score(x["latent"], x["lat_scale"], orc.absorb(x["q"], x["D"]), x["w"])
    assert_scores_close(s.cpu().numpy(), o, RTOL["fp8"])
    gi = idx.cpu().numpy()
    for b in range(w.B):
        for l in range(w.G):
            assert_topk_row(gi[b, 0, l], o[b, 0, l], w.k, w.L, RTOL["fp8"], f"b{b} l{l}")


def test_repeated_timeouts_each_reported_once(li):
    for _ in range(3):
        assert li.li_selftest_wait_timeout(2000) == 0
        assert li.li_device_status() == -6
    assert li.li_device_status() == 0
