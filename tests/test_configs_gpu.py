"""GPU parity at the five workloads' full sizes, element by element, in the launch
configuration the benchmark times (tg_gemm_persistent on one GPU, one persistent CTA
per SM).  The oracle is the full binary64 product (numpy's float64 matrix product on the
host cores) rounded once to the output type.
"""

import pytest

from persistent_warp_specialized_gb300 import workloads as wl

from gpu_helpers import (assert_within_accumulation_bound, assert_within_tolerance, ensure_library, oracle_bits, run_gpu,
                         ulp_diff_stats)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workload_matches_oracle(name):
    w = wl.WORKLOADS[name]
    a, b = wl.workload_inputs(w)
    got = run_gpu(a, b, w.dtype)
    ref = oracle_bits(a, b, w.dtype)
    assert_within_tolerance(got, ref, w.dtype, name)
    # beyond the gate: within the fp32 summation bound; ulp distances are reported only
    assert_within_accumulation_bound(got, ref, a, b, w.dtype, name)
    far, worst = ulp_diff_stats(got, ref, w.dtype)
    print(f"{name}: {far} elements more than 1 ulp from C_ref (max {worst:.2f} ulp)")
