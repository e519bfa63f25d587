"""Failure detection without a GPU fault: a bounded wait on an mbarrier that
nothing arrives on runs out, the device status the host reads says so
(QSA_DEV_WAIT_TIMEOUT), the wait lasted its limit, and the context stays usable
for a parity-checked attention step afterwards."""
import numpy as np
import pytest

from oracle import oracle
from sparse_selected_cell_gb300 import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 32


def test_wait_runs_out_and_is_reported():
    from sparse_selected_cell_gb300 import qsa
    assert torch.cuda.is_available()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    qsa.wait_selftest(20000, st)            # 20 ms
    e1.record()
    torch.cuda.synchronize()
    assert int(st.item()) == WAIT_TIMEOUT
    assert e0.elapsed_time(e1) >= 19.0      # it waited its limit (ms)
    # the context is still usable: one small prompt step against the oracle
    w = gen.make(2, n_q=16, seed=31)
    d = qsa.to_device(w)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qsa.prompt_attn(d["q"], d["k_pool"], d["v_pool"], d["k_scale"], d["v_scale"], d["page_table"],
                          d["sel"], d["sel_count"], dev_status=st2).cpu().numpy()
    assert int(st2.item()) == 0
    ref = oracle.attn_ref_workload(w)
    err = np.abs(out - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()


def test_wait_selftest_rejects_bad_limits():
    from sparse_selected_cell_gb300 import qsa
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for bad in (0, -5, 10000001):
        with pytest.raises(RuntimeError):
            qsa.wait_selftest(bad, st)
    assert int(st.item()) == 0
