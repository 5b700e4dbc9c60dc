"""Kernel variants (schedulers, Q storage, block sizes, streams, the host
entry point) must agree with one another and with the oracle."""
import numpy as np
import pytest

from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests import helpers as H
from tests.gpu_helpers import check_parity, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,n", [(np.float32, 4), (np.float32, 8), (np.float32, 12), (np.float32, 16),
                                  (np.float32, 24), (np.float32, 32), (np.float64, 4), (np.float64, 8),
                                  (np.float64, 12), (np.float64, 16), (np.float64, 24), (np.float64, 32)])
@pytest.mark.parametrize("jobz", [True, False])
def test_flat_equals_nested(dt, n, jobz):
    """The flat lockstep and the nested scheduler of the static-position
    kernels run the same per-problem operations, so their results are equal
    (perf_steqr, Lockstep flat solver: bitwise equal on the dump cases)."""
    d, e, _, _ = inputs.mixed_problems(n, 4096, dt, seed=n)
    a = run_gpu(d, e, jobz=jobz, scheduler=1, kernel=1)
    b = run_gpu(d, e, jobz=jobz, scheduler=2, kernel=1)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[2], b[2])
    if jobz:
        np.testing.assert_array_equal(a[1], b[1])
    check_parity(d, e, *a, oracle_ref(d, e, jobz=jobz), what=f"flat {n}")


@pytest.mark.parametrize("dt,n,qs", [(np.float32, 16, 3), (np.float32, 16, 2), (np.float32, 32, 3), (np.float64, 12, 2),
                                     (np.float64, 12, 3), (np.float64, 16, 3)])
def test_qstore_variants_agree(dt, n, qs):
    """Q storage policies of the static-position kernels: same eigenvalues."""
    d, e = inputs.normal_problems(n, 5000, dt, seed=7)
    ref = oracle_ref(d, e)
    a = run_gpu(d, e, qstore=qs, kernel=1)
    check_parity(d, e, *a, ref, what=f"qstore={qs}")
    b = run_gpu(d, e, kernel=1)
    np.testing.assert_array_equal(a[0], b[0])


@pytest.mark.parametrize("tpb", [32, 64, 96, 224])
def test_block_size_does_not_change_results(tpb):
    """Block size changes the launch shape only (perf_steqr, Work-group
    multiplier: byte-identical outputs)."""
    d, e = inputs.normal_problems(16, 3000, np.float32, seed=8)
    # the hybrid store takes any block size (the split-role kernel has a
    # fixed 512-thread shape and rejects others)
    a = run_gpu(d, e, threads_per_block=tpb, qstore=4)
    b = run_gpu(d, e, qstore=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_host_entry_point_matches_device_path():
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    n, batch = 12, 2000
    d, e = inputs.normal_problems(n, batch, np.float64, seed=9)
    hd = torch.from_numpy(d.copy()).pin_memory()
    he = torch.from_numpy(e.copy()).pin_memory()
    hq = torch.empty((batch, n, n), dtype=torch.float64).pin_memory()
    hi = torch.empty(batch, dtype=torch.int32).pin_memory()
    dev = torch.empty(bstq.host_work_size(np.float64, True, n, batch), dtype=torch.uint8, device="cuda")
    bstq.solve_host(hd, he, hq, hi, dev, jobz=True)
    torch.cuda.synchronize()
    lam, Q, info = run_gpu(d, e)
    np.testing.assert_array_equal(hd.numpy(), lam)
    np.testing.assert_array_equal(hq.numpy().transpose(0, 2, 1), Q)
    np.testing.assert_array_equal(hi.numpy(), info)


def test_streams_are_honoured():
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    n, batch = 16, 8192
    d, e = inputs.normal_problems(n, batch, np.float32, seed=10)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for s in (s1, s2):
        with torch.cuda.stream(s):
            dg = torch.from_numpy(d.copy()).cuda()
            eg = torch.from_numpy(e.copy()).cuda()
            outs.append(bstq.solve(dg, eg, jobz=True, stream=s))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(outs[0][0].cpu().numpy(), outs[1][0].cpu().numpy())


def test_oversized_block_is_rejected_not_launched():
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    # 1024 threads x 512 B of shared Q rows exceeds what one block may hold
    with pytest.raises(bstq.BstqError) as ei:
        run_gpu(*inputs.normal_problems(16, 64, np.float32, seed=1), threads_per_block=1024, qstore=4)
    assert ei.value.code == -10
    # the split-role kernel has one block shape (512 threads)
    with pytest.raises(bstq.BstqError) as ei:
        run_gpu(*inputs.normal_problems(16, 64, np.float32, seed=1), threads_per_block=256, qstore=5)
    assert ei.value.code == -10


@pytest.mark.parametrize("dt,n", [(np.float32, 3), (np.float32, 8), (np.float32, 16), (np.float32, 21),
                                  (np.float32, 32), (np.float64, 5), (np.float64, 12), (np.float64, 17),
                                  (np.float64, 32)])
@pytest.mark.parametrize("jobz", [True, False])
def test_dynamic_family_parity_and_schedulers(dt, n, jobz):
    """Dynamic-position kernels (d, e in shared memory, rolled chase): parity
    with the oracle on the mixed hard cases, flat equal to nested."""
    d, e, _, _ = inputs.mixed_problems(n, 3000, dt, seed=77 + n)
    a = run_gpu(d, e, jobz=jobz, kernel=2, scheduler=1)
    b = run_gpu(d, e, jobz=jobz, kernel=2, scheduler=2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[2], b[2])
    if jobz:
        np.testing.assert_array_equal(a[1], b[1])
    check_parity(d, e, *a, oracle_ref(d, e, jobz=jobz), what=f"dyn {n}")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_dynamic_family_budget_and_poison(dt):
    n = 14
    d, e = inputs.normal_problems(n, 400, dt, seed=5)
    d[3, 4] = np.nan
    ref = oracle_ref(d, e, maxit_per_n=1)
    lam, Q, info = run_gpu(d, e, kernel=2, max_sweeps_per_n=1)
    assert info[3] == -1 and np.all(np.isnan(lam[3]))
    ok = np.arange(400) != 3
    assert np.all(info[ok] > 0) and np.mean(info[ok] == ref.info[ok]) > 0.9


@pytest.mark.parametrize("n", [9, 12, 13, 16, 17, 21, 24, 25, 29, 32])
def test_split_role_kernel(n):
    """Chase warps record rotations, partner warps apply them to Q one pass
    behind (above n = 16 several Q warps share a problem's rows): same
    per-problem arithmetic as the static kernel, so equal eigenvalues, and
    eigenvectors within the parity bounds."""
    d, e, _, _ = inputs.mixed_problems(n, 3333, np.float32, seed=90 + n)
    ref = oracle_ref(d, e)
    a = run_gpu(d, e, qstore=5)
    check_parity(d, e, *a, ref, what=f"split {n}")
    b = run_gpu(d, e, qstore=4 if n > 12 else 1)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[2], b[2])
    # poisoned and budget-exhausted problems too
    d[7, 3] = np.inf
    c = run_gpu(d, e, qstore=5, max_sweeps_per_n=1)
    assert c[2][7] == -1 and np.all(np.isnan(c[1][7]))


@pytest.mark.gpu
@pytest.mark.parametrize("dt,n,params", [(np.float32, 16, {}), (np.float32, 16, {"qstore": 4}),
                                         (np.float32, 8, {}), (np.float64, 12, {}), (np.float32, 13, {}),
                                         (np.float32, 7, {}), (np.float32, 27, {}), (np.float64, 3, {})])
def test_unaligned_q_matches_aligned(dt, n, params):
    """Q columns go out in 16-byte vectors when Q starts on a 16-byte boundary
    and n * sizeof(T) is a multiple of 16; otherwise (a Q that is only
    element-aligned, or a ragged n) the warp stages its columns and writes
    them together.  Both must give the same bytes."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    d, e = inputs.normal_problems(n, 1000, dt, seed=21)
    ref = run_gpu(d, e, **params)
    dev = torch.device("cuda:0")
    dg = torch.from_numpy(d.copy()).to(dev)
    eg = torch.from_numpy(e.copy()).to(dev)
    buf = torch.full((1000 * n * n + 1,), float("nan"), dtype=dg.dtype, device=dev)
    Q = buf[1:].view(1000, n, n)
    assert Q.data_ptr() % 16 != 0
    lam, Qo, info = bstq.solve(dg, eg, jobz=True, Q=Q, **params)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(lam.cpu().numpy(), ref[0])
    np.testing.assert_array_equal(Qo.cpu().numpy(), ref[1])
    np.testing.assert_array_equal(info.cpu().numpy(), ref[2])


@pytest.mark.parametrize("dt,n,params", [(np.float32, 16, {}), (np.float32, 16, {"qstore": 4}),
                                         (np.float32, 12, {}), (np.float32, 5, {}), (np.float32, 8, {}),
                                         (np.float32, 32, {}), (np.float32, 16, {"kernel": 2}),
                                         (np.float32, 16, {"qstore": 3}), (np.float64, 12, {}),
                                         (np.float64, 7, {}), (np.float64, 8, {"kernel": 1}),
                                         (np.float64, 32, {}), (np.float32, 16, {"scheduler": 2}),
                                         (np.float64, 12, {"scheduler": 2}), (np.float64, 12, {"update_scheme": 1}),
                                         (np.float32, 40, {}), (np.float64, 64, {})])
def test_back_transform_matches_oracle(dt, n, params):
    """back_transform (BatchLAS page "algo_steqr", eigenvector accumulation):
    the rotations are right-applied to the caller's basis Z.  With Z
    orthogonal, V = Z Q must hold the eigenvectors of A = Z T Z^T within the
    stated bounds, agree with the oracle run on the same Z (columns up to
    sign), and leave the eigenvalues and info as without Z."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    from tests import helpers as H
    batch = 1500
    d, e = inputs.normal_problems(n, batch, dt, seed=40 + n)
    Z = inputs.orthogonal_bases(n, batch, dt, seed=n)
    ref = oracle_ref(d, e, True)
    import oracle
    oz = oracle.steqr(d, e, jobz=True, Z=Z)
    dev = torch.device("cuda:0")
    dg = torch.from_numpy(d.copy()).to(dev)
    eg = torch.from_numpy(e.copy()).to(dev)
    lam, V, info = bstq.solve(dg, eg, jobz=True, Z=torch.from_numpy(Z).to(dev), **params)
    torch.cuda.synchronize()
    lam, V, info = lam.cpu().numpy(), V.cpu().numpy(), info.cpu().numpy()
    plain = run_gpu(d, e, **params)
    np.testing.assert_array_equal(lam, plain[0])
    np.testing.assert_array_equal(info, oz.info)
    eps = H.eps_of(dt)
    tn = H.norm1(d, e).astype(np.float64)
    assert np.all(np.abs(lam.astype(np.float64) - ref.lam).max(1) <= H.lam_tol(n, dt, tn))
    res, orth = H.back_residual_orth(d, e, Z, lam, V)
    assert np.all(res <= 64 * n * eps * tn)
    assert np.all(orth <= 64 * n * eps)
    # V against Z times the GPU's own eigenvectors (same rotations, rows of Z
    # rotated independently): within rounding
    zq = Z.astype(np.float64) @ plain[1].astype(np.float64)
    assert np.abs(zq - V).max() <= 64 * n * eps
    # against the oracle's back-transformed vectors, column by column up to
    # sign where the eigenvalue is well separated
    lam64 = ref.lam.astype(np.float64)
    gaps = np.minimum(np.abs(np.diff(lam64, axis=1, prepend=-np.inf)),
                      np.abs(np.diff(lam64, axis=1, append=np.inf)))
    ok = gaps > 1e-2 * tn[:, None]
    sgn = np.sign((V.astype(np.float64) * oz.Q.astype(np.float64)).sum(1))
    diff = np.abs(V.astype(np.float64) * sgn[:, None, :] - oz.Q.astype(np.float64)).max(1)
    bound = 64 * n * eps * tn[:, None] / np.maximum(gaps, 1e-300)
    assert np.all(diff[ok] <= np.maximum(bound[ok], 64 * n * eps))


def test_back_transform_identity_basis_equals_plain():
    """Z = I gives the plain eigenvectors exactly."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    d, e = inputs.normal_problems(16, 800, np.float32, seed=44)
    plain = run_gpu(d, e)
    dev = torch.device("cuda:0")
    I = torch.eye(16, dtype=torch.float32, device=dev).expand(800, 16, 16)
    lam, V, info = bstq.solve(torch.from_numpy(d.copy()).to(dev), torch.from_numpy(e.copy()).to(dev),
                              jobz=True, Z=I)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(V.cpu().numpy(), plain[1])
    np.testing.assert_array_equal(lam.cpu().numpy(), plain[0])


def test_host_entry_point_back_transform():
    """bstq_solve_host copies the basis in when back_transform is set."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    n, batch = 16, 1200
    d, e = inputs.normal_problems(n, batch, np.float32, seed=45)
    Z = inputs.orthogonal_bases(n, batch, np.float32, seed=3)
    hd = torch.from_numpy(d.copy()).pin_memory()
    he = torch.from_numpy(e.copy()).pin_memory()
    hq = torch.from_numpy(np.ascontiguousarray(Z.transpose(0, 2, 1))).pin_memory()  # storage [b][j][i] = Z_ij
    hi = torch.empty(batch, dtype=torch.int32).pin_memory()
    dev = torch.empty(bstq.host_work_size(np.float32, True, n, batch, back_transform=True), dtype=torch.uint8,
                      device="cuda")
    bstq.solve_host(hd, he, hq, hi, dev, jobz=True, back_transform=True)
    torch.cuda.synchronize()
    lam, V, info = bstq.solve(torch.from_numpy(d.copy()).cuda(), torch.from_numpy(e.copy()).cuda(), jobz=True,
                              Z=torch.from_numpy(Z).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hd.numpy(), lam.cpu().numpy())
    np.testing.assert_array_equal(hq.numpy().transpose(0, 2, 1), V.cpu().numpy())
    np.testing.assert_array_equal(hi.numpy(), info.cpu().numpy())


@pytest.mark.parametrize("dt,n,jobz,batch", [(np.float64, 12, True, 4000), (np.float64, 12, False, 4000),
                                             (np.float32, 16, True, 4000), (np.float64, 3, True, 3001),
                                             (np.float64, 32, True, 2000), (np.float32, 27, False, 2500),
                                             (np.float64, 12, True, 32768)])
def test_pg_update_scheme_matches_oracle(dt, n, jobz, batch):
    """PG update (page "algo_steqr", update schemes) against the oracle's PG
    scheme on the same inputs: the benchmark spec's bounds, info exactly."""
    d, e = inputs.normal_problems(n, batch, dt, seed=70 + n)
    ref = oracle_ref(d, e, jobz, scheme="pg")
    a = run_gpu(d, e, jobz=jobz, update_scheme=1)
    check_parity(d, e, *a, ref, what=f"pg n={n}")


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_pg_update_scheme_hard_cases(dt):
    d, e, _, _ = inputs.mixed_problems(32, 3000, dt, seed=9)
    ref = oracle_ref(d, e, True, scheme="pg")
    a = run_gpu(d, e, jobz=True, update_scheme=1)
    check_parity(d, e, *a, ref, what="pg mixed")


def test_pg_with_static_family_is_rejected():
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    with pytest.raises(bstq.BstqError) as ei:
        run_gpu(*inputs.normal_problems(16, 64, np.float32, seed=1), update_scheme=1, kernel=1)
    assert ei.value.code == -10


def test_pg_and_exp_agree_on_the_gpu():
    """The two update forms of the same implicit step: eigenvalues within the
    bound of each other, same info."""
    d, e = inputs.normal_problems(12, 5000, np.float64, seed=80)
    a = run_gpu(d, e, update_scheme=1)
    b = run_gpu(d, e, update_scheme=0, kernel=2)
    np.testing.assert_array_equal(a[2], b[2])
    from tests import helpers as H
    tn = H.norm1(d, e).astype(np.float64)
    assert np.all(np.abs(a[0] - b[0]).max(1) <= 2 * H.lam_tol(12, np.float64, tn))


@pytest.mark.parametrize("n", [20, 32])
def test_split_role_rows_over_several_warps_back_transform_and_unaligned(n):
    """Q warps that each hold a block of rows: the caller's basis enters row
    block by row block (back_transform), and an element-aligned Q takes the
    element path with the same bytes."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    dt = np.float32
    batch = 1500
    d, e = inputs.normal_problems(n, batch, dt, seed=400 + n)
    Z = inputs.orthogonal_bases(n, batch, dt, seed=401 + n)
    dev = torch.device("cuda:0")
    lam, V, info = bstq.solve(torch.from_numpy(d.copy()).to(dev), torch.from_numpy(e.copy()).to(dev), jobz=True,
                              Z=torch.from_numpy(Z).to(dev), qstore=5)
    torch.cuda.synchronize()
    lam, V = lam.cpu().numpy(), V.cpu().numpy()
    res, orth = H.back_residual_orth(d, e, Z, lam, V)
    tn = H.norm1(d, e).astype(np.float64)
    eps = H.eps_of(dt)
    assert np.all(res <= 64 * n * eps * tn) and np.all(orth <= 64 * n * eps)
    ref = run_gpu(d, e, qstore=5)
    buf = torch.full((batch * n * n + 1,), float("nan"), dtype=torch.float32, device=dev)
    Qu = buf[1:].view(batch, n, n)
    lam2, Q2, info2 = bstq.solve(torch.from_numpy(d.copy()).to(dev), torch.from_numpy(e.copy()).to(dev), jobz=True,
                                 Q=Qu, qstore=5)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Q2.cpu().numpy(), ref[1])
    np.testing.assert_array_equal(lam2.cpu().numpy(), ref[0])
