"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs, at every configuration of the workload."""
import numpy as np
import pytest

from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H
from tests.gpu_helpers import check_parity, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

F32, F64 = np.float32, np.float64


def _case(dt, n, batch, kind="normal", jobz=True, seed=0, **params):
    d, e = inputs.problems(kind, n, batch, dt, seed)
    ref = oracle_ref(d, e, jobz=jobz)
    lam, Q, info = run_gpu(d, e, jobz=jobz, **params)
    check_parity(d, e, lam, Q, info, ref, what=f"{np.dtype(dt).name} n={n} B={batch} {kind} jobz={jobz} {params}")
    return d, e, lam, Q, info, ref


def test_small_config_f32_n4():
    """float32, n=4, batch 1,024, jobz=V, N(0,1) from seed 0."""
    _case(F32, 4, 1024)


@pytest.mark.parametrize("jobz", [True, False])
@pytest.mark.parametrize("n,batch", [(8, 65536), (16, 32768)])
def test_float32_n8_n16_full(n, batch, jobz):
    _case(F32, n, batch, jobz=jobz)


@pytest.mark.parametrize("jobz", [True, False])
def test_float64_n12_full_flat_vs_nested(jobz):
    n, batch = 12, 32768
    d, e, lam, Q, info, ref = _case(F64, n, batch, jobz=jobz, scheduler=1)
    lam2, Q2, info2 = run_gpu(d, e, jobz=jobz, scheduler=2)
    assert np.array_equal(lam, lam2) and np.array_equal(info, info2)
    if jobz:
        assert np.array_equal(Q, Q2)


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("jobz", [True, False])
def test_mixed_hard_cases_n32(dt, jobz):
    n, batch = 32, 32768
    d, e, labels, ab = inputs.mixed_problems(n, batch, dt, seed=0)
    ref = oracle_ref(d, e, jobz=jobz)
    lam, Q, info = run_gpu(d, e, jobz=jobz)
    check_parity(d, e, lam, Q, info, ref, what=f"mixed {np.dtype(dt).name} jobz={jobz}")
    z = labels == inputs.CLASS_INDEX["zero"]
    assert np.all(lam[z] == 0)
    if jobz:
        assert np.all(Q[z] == np.eye(n, dtype=dt))
    # pre-split structure: every eigenvector lives on one block
    ps = np.nonzero(labels == inputs.CLASS_INDEX["presplit"])[0][:300]
    for b in ps:
        blk = np.concatenate([[0], np.cumsum(e[b] == 0)])
        if jobz:
            for j in range(n):
                rows = np.nonzero(Q[b, :, j])[0]
                assert len(set(blk[rows])) == 1
        singles = [i for i in range(n) if np.count_nonzero(blk == blk[i]) == 1]
        for i in singles:
            assert d[b, i] in lam[b]
    tp = np.nonzero(labels == inputs.CLASS_INDEX["toeplitz"])[0]
    tn = H.norm1(d, e).astype(np.float64)
    for b in tp[:200]:
        cf = H.toeplitz_eigenvalues(n, d[b, 0], e[b, 0]).astype(np.float64)
        assert np.max(np.abs(lam[b] - cf)) <= H.lam_tol(n, dt, tn[b])


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("jobz", [True, False])
def test_sweep_all_n(dt, jobz):
    """n = 1..32 at a batch that spans many blocks with a ragged tail."""
    for n in range(1, 33):
        _case(dt, n, 3001 + 7 * n, jobz=jobz, seed=n)


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("n", [1, 5, 9, 20, 31])
def test_sweep_full_size_samples(dt, n):
    """Full batch sizes of the n=1..32 sweep for a few n."""
    _case(dt, n, 65536 if n <= 8 else 32768, jobz=True, seed=100 + n)


@pytest.mark.parametrize("dt", [F32, F64])
def test_nonfinite_and_degenerate(dt):
    n = 10
    d, e = inputs.normal_problems(n, 200, dt, seed=3)
    d[1, 2] = np.nan
    e[2, 4] = np.inf
    d[3, 0] = -np.inf
    d[4] = 0
    e[4] = 0
    e[5] = 0                       # diagonal matrix
    e[6, ::2] = 0                  # many small blocks
    d[7] = 1.0
    e[7] = 0                       # all eigenvalues tie
    d[8] *= 1e-30
    e[8] *= 1e-30
    ref = oracle_ref(d, e)
    lam, Q, info = run_gpu(d, e)
    check_parity(d, e, lam, Q, info, ref, what="degenerate")
    assert list(info[:4]) == [0, -1, -1, -1]
    assert np.all(np.isnan(Q[1:4]))
    assert np.all(lam[4] == 0) and np.array_equal(Q[4], np.eye(n, dtype=dt))
    assert np.array_equal(lam[5], np.sort(d[5]))
    assert np.array_equal(Q[7], np.eye(n, dtype=dt))   # ties keep the caller's order


@pytest.mark.parametrize("dt", [F32, F64])
def test_sweep_budget_exhaustion(dt):
    n = 16
    d, e = inputs.normal_problems(n, 512, dt, seed=2)
    ref0 = oracle_ref(d, e, maxit_per_n=1)
    lam, Q, info = run_gpu(d, e, max_sweeps_per_n=1)
    assert np.all(info > 0) and np.all(ref0.info > 0)
    # the count of unconverged off-diagonals matches the oracle up to the
    # rounding of deflation decisions
    assert np.mean(info == ref0.info) > 0.9


@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("batch", [1, 31, 33, 1000])
def test_ragged_batches(dt, batch):
    _case(dt, 13, batch, seed=batch)


def test_batch_zero_is_noop():
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    d = torch.empty((0, 8), device="cuda", dtype=torch.float32)
    e = torch.empty((0, 7), device="cuda", dtype=torch.float32)
    lam, Q, info = bstq.solve(d, e, jobz=True)
    torch.cuda.synchronize()
    assert lam.shape == (0, 8) and Q.shape == (0, 8, 8)


@pytest.mark.parametrize("dt", [F32, F64])
def test_unsorted_output_order(dt):
    """Unsorted output: eigenpair j sits where it converged, which depends on
    deflation decisions that rounding can move; compare the spectra, check
    that the unsorted pairs are eigenpairs, and that the placement agrees
    with the oracle's for almost every problem."""
    from tests.gpu_helpers import orth_err, tri_residual
    n = 9
    d, e = inputs.normal_problems(n, 300, dt, seed=4)
    ref = oracle_ref(d, e, sort=False)
    lam, Q, info = run_gpu(d, e, no_sort=True)
    assert np.all(info == 0)
    tn = H.norm1(d, e).astype(np.float64)
    tol = H.lam_tol(n, dt, tn)
    assert np.all(np.abs(np.sort(lam, 1) - np.sort(ref.lam, 1)).max(1) <= tol)
    assert np.all(tri_residual(d, e, lam, Q) <= 64 * n * H.eps_of(dt) * tn)
    assert np.all(orth_err(Q) <= 64 * n * H.eps_of(dt))
    same = np.abs(lam - ref.lam).max(1) <= tol
    assert same.mean() >= 0.9, same.mean()
    assert not np.all(np.diff(lam, axis=1) >= 0)   # really left unsorted


# --- n > 32 (the n <= 32 cliff removed: the dynamic-position kernels at
# compile-time maxima 48 and 64) ---

@pytest.mark.parametrize("dt", [F32, F64])
@pytest.mark.parametrize("jobz", [True, False])
@pytest.mark.parametrize("n", [33, 40, 48, 49, 57, 64, 65, 80, 96, 97, 127, 128])
def test_beyond_32(dt, n, jobz):
    _case(dt, n, (2000 + 3 * n) if n <= 64 else 700 + n, jobz=jobz, seed=200 + n)


@pytest.mark.parametrize("dt", [F32, F64])
def test_mixed_hard_cases_n128(dt):
    """The mixed hard classes at the largest size, with the class checks."""
    n, batch = 128, 700
    d, e, labels, ab = inputs.mixed_problems(n, batch, dt, seed=2)
    ref = oracle_ref(d, e, jobz=True)
    lam, Q, info = run_gpu(d, e, jobz=True)
    check_parity(d, e, lam, Q, info, ref, what=f"mixed n=128 {np.dtype(dt).name}")
    z = labels == inputs.CLASS_INDEX["zero"]
    assert np.all(lam[z] == 0) and np.all(Q[z] == np.eye(n, dtype=dt))
    tn = H.norm1(d, e).astype(np.float64)
    for b in np.nonzero(labels == inputs.CLASS_INDEX["toeplitz"])[0][:20]:
        cf = H.toeplitz_eigenvalues(n, d[b, 0], e[b, 0]).astype(np.float64)
        assert np.max(np.abs(lam[b] - cf)) <= H.lam_tol(n, dt, tn[b])


@pytest.mark.parametrize("dt", [F32, F64])
def test_mixed_hard_cases_n64(dt):
    n, batch = 64, 4000
    d, e, labels, ab = inputs.mixed_problems(n, batch, dt, seed=1)
    ref = oracle_ref(d, e, jobz=True)
    lam, Q, info = run_gpu(d, e, jobz=True)
    check_parity(d, e, lam, Q, info, ref, what=f"mixed n=64 {np.dtype(dt).name}")
    z = labels == inputs.CLASS_INDEX["zero"]
    assert np.all(lam[z] == 0)
    assert np.all(Q[z] == np.eye(n, dtype=dt))
    tp = np.nonzero(labels == inputs.CLASS_INDEX["toeplitz"])[0]
    tn = H.norm1(d, e).astype(np.float64)
    for b in tp[:100]:
        cf = H.toeplitz_eigenvalues(n, d[b, 0], e[b, 0]).astype(np.float64)
        assert np.max(np.abs(lam[b] - cf)) <= H.lam_tol(n, dt, tn[b])


@pytest.mark.parametrize("dt", [F32, F64])
def test_beyond_32_variants(dt):
    """n = 64: nested = flat, PG within bounds, back_transform, unaligned Q."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    n, batch = 64, 1500
    d, e = inputs.normal_problems(n, batch, dt, seed=300)
    a = run_gpu(d, e)
    b = run_gpu(d, e, scheduler=2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    check_parity(d, e, *run_gpu(d, e, update_scheme=1), oracle_ref(d, e, True, scheme="pg"), what="pg n=64")
    Z = inputs.orthogonal_bases(n, batch, dt, seed=5)
    dev = torch.device("cuda:0")
    lam, V, info = bstq.solve(torch.from_numpy(d.copy()).to(dev), torch.from_numpy(e.copy()).to(dev), jobz=True,
                              Z=torch.from_numpy(Z).to(dev))
    torch.cuda.synchronize()
    res, orth = H.back_residual_orth(d, e, Z, lam.cpu().numpy(), V.cpu().numpy())
    tn = H.norm1(d, e).astype(np.float64)
    eps = H.eps_of(dt)
    assert np.all(res <= 64 * n * eps * tn) and np.all(orth <= 64 * n * eps)
    buf = torch.full((batch * n * n + 1,), float("nan"), dtype=lam.dtype, device=dev)
    Qu = buf[1:].view(batch, n, n)
    lam2, Q2, info2 = bstq.solve(torch.from_numpy(d.copy()).to(dev), torch.from_numpy(e.copy()).to(dev), jobz=True,
                                 Q=Qu)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Q2.cpu().numpy(), a[1])
