"""GPU: the decode's bounded waits, exercised without any fault.

Every wait inside the decode kernel gives up after a bound
(nvfp4_mla_set_wait_limit); a unit whose wait runs out drains the copies and
tensor-core work it has in flight, frees its tensor memory and writes NaN
outputs and LSE. Here the bound is set far below the waits of a healthy
launch (a gather from device memory alone takes longer), so units give up;
each query token's result must then be all NaN or correct, the launch must
end normally, and the next launch with the default bound must be correct.
"""
import numpy as np
import pytest

from tests.gpu_cases import assert_parity, build_case, gpu_decode, oracle_decode
from workloads import make_workload

pytestmark = pytest.mark.gpu


# q_per_seq 100: 200 units, more than the device holds clusters at once, so a
# cluster that gives up also leaves the later units it would have taken NaN
@pytest.mark.parametrize("row_format,splits,q_per_seq", [(0, 1, 2), (0, 3, 2), (1, 2, 2),
                                                         (0, 1, 100), (1, 1, 100)])
def test_waits_that_run_out_give_nan_and_the_next_launch_is_correct(row_format, splits,
                                                                     q_per_seq):
    import nvfp4_compressed_mla_gb300 as nm
    wl = make_workload("tiny", num_seqs=2, seq_len=3000, num_heads=64, topk=900,
                       q_per_seq=q_per_seq)
    case = build_case(wl, "referenced", row_format)
    ref, ref_lse, _ = oracle_decode(case)
    nm.nvfp4_mla_set_wait_limit(2000)
    try:
        out, lse = gpu_decode(case, num_splits=splits)
    finally:
        nm.nvfp4_mla_set_wait_limit(0)
    failed = np.isnan(lse).all(axis=1)
    assert failed.any(), "no unit gave up under a 2000-cycle wait bound"
    assert np.isnan(out[failed]).all()
    ok = ~failed
    if ok.any():
        assert_parity(out[ok], lse[ok], ref[ok], ref_lse[ok])
    out2, lse2 = gpu_decode(case, num_splits=splits)
    assert_parity(out2, lse2, ref, ref_lse)

