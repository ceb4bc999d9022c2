"""GPU parity at the five workloads' full sizes, element by element.  Each workload runs
through tg_gemm_persistent (the variant the library picks, which is what the benchmark
times) and through each kernel variant explicitly.  The oracle is the full binary64
product (numpy's float64 matrix product on the host cores) rounded once to the output type.
"""

import pytest

import persistent_warp_specialized_gb300 as tg
from persistent_warp_specialized_gb300 import workloads as wl

from gpu_helpers import (assert_within_accumulation_bound, VARIANTS, assert_within_tolerance, ensure_library, oracle_bits, run_gpu,
                         ulp_diff_stats)

pytestmark = pytest.mark.gpu

_cache = {}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_library()


def _inputs_and_oracle(name):
    if name not in _cache:
        _cache.clear()
        w = wl.WORKLOADS[name]
        a, b = wl.workload_inputs(w)
        _cache[name] = (w, a, b, oracle_bits(a, b, w.dtype))
    return _cache[name]


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
@pytest.mark.parametrize("variant", [None] + VARIANTS)
def test_workload_matches_oracle(name, variant):
    w, a, b, ref = _inputs_and_oracle(name)
    if variant is None:
        assert tg.tg_gemm_launch_shape(w.M, w.N, w.K)["variant"] in (
            tg.TG_VARIANT_SINGLE, tg.TG_VARIANT_PAIR, tg.TG_VARIANT_PAIR_WIDE)
    got = run_gpu(a, b, w.dtype, variant=variant)
    assert_within_tolerance(got, ref, w.dtype, f"{name} {variant or 'auto'}")
    # beyond the gate: within the fp32 summation bound; ulp distances are reported only
    assert_within_accumulation_bound(got, ref, a, b, w.dtype, name)
    far, worst = ulp_diff_stats(got, ref, w.dtype)
    print(f"{name} {variant or 'auto'}: {far} elements more than 1 ulp from C_ref (max {worst:.2f} ulp)")
