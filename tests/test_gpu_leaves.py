"""GPU parity of the stedc leaf solve (bstq_stedc_leaves through the C ABI)
against the oracle's leaf solve on the same seeded inputs: each leaf under
the benchmark spec's bounds of its own torn block, info exactly, and the exact
cases (one-row leaves return the torn diagonal bit for bit; one leaf is the
plain solve; the result equals solving the torn leaves one size group at a
time)."""
import numpy as np
import pytest

import oracle
from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests.gpu_helpers import ORACLE_THREADS, check_parity, run_gpu

pytestmark = pytest.mark.gpu

F32, F64 = np.float32, np.float64


class _LeafRef:
    def __init__(self, lam, Q, info):
        self.lam, self.Q, self.info = lam, Q, info


def run_leaves(d, e, leaf, jobz=True, **params):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dev = torch.device("cuda:0")
    dg = torch.from_numpy(np.ascontiguousarray(d)).to(dev)
    eg = torch.from_numpy(np.ascontiguousarray(e)).to(dev)
    lam, Qf, Qt, info = bstq.stedc_leaves(dg, eg, leaf, jobz=jobz, **params)
    torch.cuda.synchronize()
    return (lam.cpu().numpy(), None if Qf is None else Qf.cpu().numpy(),
            None if Qt is None else Qt.cpu().numpy(), info.cpu().numpy())


def _leaf_q(Qf, Qt, k, nfull):
    if Qf is None:
        return None
    return Qf[:, k] if k < nfull else Qt


def _check(d, e, leaf, jobz=True, **params):
    ref = oracle.stedc_leaves(d, e, leaf, jobz=jobz, nthreads=ORACLE_THREADS)
    lam, Qf, Qt, info = run_leaves(d, e, leaf, jobz=jobz, **params)
    assert info.shape == ref.info.shape
    assert np.array_equal(info, ref.info)
    nfull = (Qf.shape[1] if Qf is not None else sum(1 for m in ref.sizes if m == ref.sizes[0]))
    for k, (s, m) in enumerate(zip(ref.starts, ref.sizes)):
        dl = ref.d_torn[:, s:s + m]
        el = e[:, s:s + m - 1]
        lref = _LeafRef(ref.lam[:, s:s + m], None if ref.Q is None else ref.Q[k], ref.info[:, k])
        check_parity(dl, el, lam[:, s:s + m], _leaf_q(Qf, Qt, k, nfull), info[:, k], lref,
                     what=f"leaf {k} ({s}:{s + m}) n={d.shape[1]} leaf={leaf}")
    return ref, lam, Qf, Qt, info


@pytest.mark.parametrize("jobz", [True, False])
def test_pages_case_float_n64_leaves_of_32(jobz):
    """float n = 64 cut into two leaves of 32, batch 8,192."""
    d, e = inputs.normal_problems(64, 8192, F32, seed=0)
    _check(d, e, 32, jobz=jobz)


@pytest.mark.parametrize("dt,n,leaf,batch", [
    (F64, 64, 32, 2048), (F32, 70, 32, 1000), (F64, 37, 8, 1500), (F32, 130, 16, 300),
    (F64, 100, 24, 400), (F32, 33, 32, 900), (F64, 12, 5, 2000), (F32, 96, 48, 300), (F64, 128, 64, 120),
    (F32, 250, 100, 100)])
def test_leaf_parity(dt, n, leaf, batch):
    d, e = inputs.normal_problems(n, batch, dt, seed=n + leaf)
    _check(d, e, leaf, jobz=True)


@pytest.mark.parametrize("dt", [F32, F64])
def test_mixed_hard_cases_n64(dt):
    """The mixed hard-case classes (graded, pre-split, zero, 1e+-18 scaled,
    Toeplitz) cut into leaves of 32 and of 12 (a 4-row last leaf)."""
    d, e, _, _ = inputs.mixed_problems(64, 4096, dt, seed=1)
    _check(d, e, 32, jobz=True)
    _check(d, e, 12, jobz=True)


@pytest.mark.parametrize("dt", [F32, F64])
def test_one_row_leaves_return_the_torn_diagonal(dt):
    d, e = inputs.normal_problems(9, 700, dt, seed=4)
    ref = oracle.stedc_leaves(d, e, 1, jobz=True)
    lam, Qf, Qt, info = run_leaves(d, e, 1)
    assert Qt is None and Qf.shape == (700, 9, 1, 1)
    assert np.array_equal(lam, ref.d_torn) and np.all(Qf == 1) and np.all(info == 0)


@pytest.mark.parametrize("dt", [F32, F64])
def test_single_leaf_is_the_plain_solve(dt):
    d, e = inputs.normal_problems(20, 1500, dt, seed=6)
    lam, Qf, Qt, info = run_leaves(d, e, 64)
    lam2, Q2, info2 = run_gpu(d, e)
    assert Qt is None and np.array_equal(lam, lam2) and np.array_equal(Qf[:, 0], Q2)
    assert np.array_equal(info[:, 0], info2)


@pytest.mark.parametrize("dt", [F32, F64])
def test_equals_the_torn_leaves_solved_by_size_group(dt):
    """Bit for bit the same as tearing on the host (the oracle's tear, a
    plain subtraction) and solving each leaf-size group with bstq_solve."""
    n, leaf, batch = 45, 16, 800
    d, e = inputs.normal_problems(n, batch, dt, seed=8)
    starts, sizes, dtn = oracle.tear(d, e, leaf)
    lam, Qf, Qt, info = run_leaves(d, e, leaf)
    F = n // leaf
    full_d = np.stack([dtn[:, s:s + leaf] for s in starts[:F]], axis=1).reshape(batch * F, leaf)
    full_e = np.stack([e[:, s:s + leaf - 1] for s in starts[:F]], axis=1).reshape(batch * F, leaf - 1)
    l1, q1, i1 = run_gpu(full_d, full_e)
    t = n % leaf
    l2, q2, i2 = run_gpu(np.ascontiguousarray(dtn[:, F * leaf:]), np.ascontiguousarray(e[:, F * leaf:]))
    assert np.array_equal(lam[:, :F * leaf], l1.reshape(batch, F * leaf))
    assert np.array_equal(lam[:, F * leaf:], l2)
    assert np.array_equal(Qf, q1.reshape(batch, F, leaf, leaf)) and np.array_equal(Qt, q2)
    assert np.array_equal(info[:, :F], i1.reshape(batch, F)) and np.array_equal(info[:, F], i2)
    assert Qt.shape == (batch, t, t)


@pytest.mark.parametrize("dt", [F32, F64])
def test_nonfinite_coupling_poisons_both_neighbours(dt):
    n, leaf = 24, 8
    d, e = inputs.normal_problems(n, 64, dt, seed=11)
    e[1, leaf - 1] = np.nan
    e[2, 3] = np.inf
    d[5, 20] = -np.inf
    ref, lam, Qf, Qt, info = _check(d, e, leaf)
    assert info[1].tolist() == [-1, -1, 0] and info[2].tolist() == [-1, 0, 0] and info[5].tolist() == [0, 0, -1]


def test_work_size_covers_both_solves():
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    lib = bstq.load()
    w = lib.bstq_stedc_leaves_work_size(0, 1, 70, 32, 100, None)
    assert w >= 4 * (100 * 70 + 100 * 67) + lib.bstq_work_size(0, 1, 32, 200) + lib.bstq_work_size(0, 1, 6, 100)
    assert lib.bstq_stedc_leaves_work_size(1, 0, 64, 32, 8192, None) > 0


@pytest.mark.parametrize("dt", [F32, F64])
def test_nested_scheduler_equals_flat(dt):
    d, e = inputs.normal_problems(40, 900, dt, seed=13)
    a = run_leaves(d, e, 16, scheduler=1)
    b = run_leaves(d, e, 16, scheduler=2)
    for x, y in zip(a, b):
        assert (x is None and y is None) or np.array_equal(x, y)


@pytest.mark.parametrize("dt", [F32, F64])
def test_unsorted_and_pg_leaves(dt):
    """no_sort leaves each leaf's spectrum unsorted (same values as the sorted
    call within the bound); the PG update scheme meets the same bounds."""
    n, leaf = 50, 16
    d, e = inputs.normal_problems(n, 700, dt, seed=17)
    ref = oracle.stedc_leaves(d, e, leaf, jobz=True, nthreads=ORACLE_THREADS)
    lam_u, Qf_u, Qt_u, info_u = run_leaves(d, e, leaf, no_sort=True)
    assert np.array_equal(info_u, ref.info)
    for k, (s, m) in enumerate(zip(ref.starts, ref.sizes)):
        dl, el = ref.d_torn[:, s:s + m], e[:, s:s + m - 1]
        got = np.sort(lam_u[:, s:s + m], axis=1)
        lref = _LeafRef(ref.lam[:, s:s + m], None, ref.info[:, k])
        check_parity(dl, el, got, None, info_u[:, k], lref, what=f"no_sort leaf {k}")
    _check(d, e, leaf, update_scheme="pg")


@pytest.mark.parametrize("dt", [F32, F64])
def test_exhausted_budget_matches_the_oracle_status(dt):
    d, e = inputs.normal_problems(32, 600, dt, seed=19)
    ref = oracle.stedc_leaves(d, e, 16, jobz=True, maxit_per_n=1, nthreads=ORACLE_THREADS)
    lam, Qf, Qt, info = run_leaves(d, e, 16, max_sweeps_per_n=1)
    assert np.any(ref.info > 0)
    # the count of unconverged off-diagonals matches the oracle up to the
    # rounding of deflation decisions
    assert np.mean(info == ref.info) > 0.9 and np.mean((info > 0) == (ref.info > 0)) > 0.95


@pytest.mark.parametrize("dt", [F32, F64])
def test_degenerate_sizes(dt):
    # one row per problem; one problem; leaf size equal to n
    for n, leaf, batch in ((1, 1, 50), (1, 32, 7), (33, 33, 1), (2, 1, 300), (64, 64, 200)):
        d, e = inputs.normal_problems(n, batch, dt, seed=n + batch)
        _check(d, e, leaf, jobz=True)
        _check(d, e, leaf, jobz=False)
