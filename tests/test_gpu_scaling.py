"""GPU parity on inputs that run every branch of the per-block scaling step
(BatchLAS page "algo_steqr", the scaling paragraph after the deflation
criterion): blocks above ssfmax (and close to overflow), below ssfmin, with
squared entries below the smallest normal number, and with subnormal norms,
in both precisions and every kernel family, against the oracle on the same
inputs.  Bounds as check_parity states them (one subnormal spacing added
where results are rounded to the subnormal grid)."""
import numpy as np
import pytest

from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H
from tests.gpu_helpers import check_parity, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

F32, F64 = np.float32, np.float64


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("jobz", [True, False])
@pytest.mark.parametrize("n", [2, 5, 12, 16, 32, 48])
@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_scaled_extremes(dt, jobz, n, kernel):
    """kernel 0: the library's default (split-role kernel for float
    9 <= n <= 16 V); 1: static-position family (n <= 32); 2: dynamic."""
    if kernel == 1 and n > 32:
        pytest.skip("the static-position family stops at n = 32")
    d, e, k = inputs.scaled_problems(n, 1400 + 3 * n, dt, seed=500 + n)
    ref = oracle_ref(d, e, jobz=jobz)
    assert np.all(ref.info == 0)
    lam, Q, info = run_gpu(d, e, jobz=jobz, kernel=kernel)
    check_parity(d, e, lam, Q, info, ref, what=f"scaled {np.dtype(dt).name} n={n} jobz={jobz} kernel={kernel}")
    # every class is present, and its eigenvalues carry its scale
    for kk in inputs.SCALE_EXPONENTS[np.dtype(dt)]:
        sel = k == kk
        assert np.any(sel)
        mag = np.abs(lam[sel].astype(np.float64)).max(1)
        assert np.all((mag == 0) | (np.abs(np.log2(np.maximum(mag, 1e-320)) - kk) < 12)), kk


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("n", [12, 20, 32])
@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_blocks_scaled_independently(dt, n, kernel):
    """Two blocks of different scale per problem: each block is scaled on
    its own, and every eigenvector stays on one block."""
    d, e, rsplit, k1, k2 = inputs.block_scaled_problems(n, 2000 + n, dt, seed=600 + n)
    ref = oracle_ref(d, e, jobz=True)
    lam, Q, info = run_gpu(d, e, jobz=True, kernel=kernel)
    check_parity(d, e, lam, Q, info, ref, what=f"block-scaled {np.dtype(dt).name} n={n} kernel={kernel}")
    for b in range(0, len(d), 7):
        rb = int(rsplit[b])
        top = np.abs(Q[b, :rb, :]).sum(0) > 0
        bot = np.abs(Q[b, rb:, :]).sum(0) > 0
        assert np.all(top ^ bot) and np.count_nonzero(top) == rb, b


@pytest.mark.parametrize("sched", [1, 2])
@pytest.mark.parametrize("dt", [F32, F64])
def test_scaled_extremes_nested_equals_flat(dt, sched):
    """Both schedulers on the scaled classes: within the bounds, and equal
    to each other where they run the same kernel family."""
    n = 14
    d, e, k = inputs.scaled_problems(n, 3000, dt, seed=700)
    ref = oracle_ref(d, e, jobz=True)
    a = run_gpu(d, e, jobz=True, scheduler=sched, kernel=2)
    check_parity(d, e, *a, ref, what=f"scaled sched={sched}")
    b = run_gpu(d, e, jobz=True, scheduler=3 - sched, kernel=2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("jobz", [True, False])
@pytest.mark.parametrize("tiny", [2.0 ** -420, 2.0 ** -1060])
def test_mixed_float64_classes_beyond_thresholds(jobz, tiny):
    """The n = 32 mixed hard-case batch in float64 at full size, with its
    'big' class at 2^520 (above ssfmax ~ 2.2e153) and its 'tiny' class below
    ssfmin (2^-405), once with subnormal norms."""
    n, batch = 32, 32768
    d, e, labels, ab = inputs.mixed_problems(n, batch, F64, seed=0, big=2.0 ** 520, tiny=tiny)
    ref = oracle_ref(d, e, jobz=jobz)
    lam, Q, info = run_gpu(d, e, jobz=jobz)
    check_parity(d, e, lam, Q, info, ref, what=f"mixed f64 big=2^520 tiny={tiny:g} jobz={jobz}")
    for cls in ("big", "tiny"):
        sel = labels == inputs.CLASS_INDEX[cls]
        assert np.count_nonzero(sel) > 1000
        assert np.all(np.abs(lam[sel]).max(1) > 0)


@pytest.mark.parametrize("jobz", [True, False])
def test_mixed_float32_subnormal_tiny_class(jobz):
    """The float32 mixed batch with its 'tiny' class at 2^-140 (subnormal
    norms, the exact 2^24 lift) and 'big' at 2^64 (above ssfmax)."""
    n, batch = 32, 32768
    d, e, labels, ab = inputs.mixed_problems(n, batch, F32, seed=1, big=2.0 ** 64, tiny=2.0 ** -140)
    ref = oracle_ref(d, e, jobz=jobz)
    lam, Q, info = run_gpu(d, e, jobz=jobz)
    check_parity(d, e, lam, Q, info, ref, what=f"mixed f32 subnormal jobz={jobz}")
