"""The record-and-apply kernel (float, jobz V, n > 32): the chase logs each
problem's rotations, the warp applies the logs to Q rows held in registers.

Its chase is the dynamic-position kernel's and every row of Q sees the same
rotations with the same arithmetic, so eigenvalues, eigenvectors and info
must equal the dynamic-position kernel's (Q in global scratch) to the bit;
against the oracle the usual parity bounds hold.  The log capacity
(log_entries) changes only how often Q goes through global memory, never a
bit of the result."""
import numpy as np
import pytest

from symmetric_tridiagonal_eigensolver_gb300 import inputs
from tests.gpu_helpers import check_parity, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu

F32 = np.float32
LOG = 6      # BSTQ_QSTORE_LOG
GLOBAL = 3   # BSTQ_QSTORE_GLOBAL (dynamic-position kernel)


def _same(a, b, what):
    np.testing.assert_array_equal(a[2], b[2], err_msg=f"{what}: info")
    np.testing.assert_array_equal(a[0], b[0], err_msg=f"{what}: eigenvalues")
    np.testing.assert_array_equal(a[1], b[1], err_msg=f"{what}: eigenvectors")


def _describe(n, batch, **params):
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    return bstq.describe(F32, True, n, batch, **params)


def test_default_above_32_is_record_and_apply():
    for n in (33, 64, 65, 128):
        assert "log" in _describe(n, 4096) and "nested" in _describe(n, 4096), n
        assert "log" in _describe(n, 4096, scheduler=1), n
    assert "global" in _describe(64, 4096, qstore=GLOBAL)   # the dynamic-position kernel on request
    assert "log" not in _describe(32, 4096)


@pytest.mark.parametrize("n", [40, 64, 128])
def test_flat_and_nested_chase_agree(n):
    """The chase's lockstep and per-lane loops run the same operations per
    problem, so the logs and every output are equal; also when logs run out
    of room (the finishing launch) and under the PG scheme."""
    d, e = inputs.normal_problems(n, 700, F32, seed=1200 + n)
    for kw in ({}, dict(log_entries=1), dict(update_scheme=1)):
        _same(run_gpu(d, e, qstore=LOG, scheduler=1, **kw), run_gpu(d, e, qstore=LOG, scheduler=2, **kw),
              f"n={n} {kw}")


@pytest.mark.parametrize("n", [33, 40, 47, 48, 57, 63, 64, 65, 80, 96, 101, 127, 128])
def test_matches_oracle(n):
    batch = 900 if n <= 64 else 300
    d, e = inputs.normal_problems(n, batch, F32, seed=500 + n)
    a = run_gpu(d, e, qstore=LOG)
    check_parity(d, e, *a, oracle_ref(d, e, True), what=f"record-and-apply n={n}")


@pytest.mark.parametrize("n", [33, 48, 64, 96, 128])
def test_bitwise_equal_to_dynamic_kernel(n):
    batch = 2000 if n <= 64 else 600
    d, e = inputs.normal_problems(n, batch, F32, seed=600 + n)
    _same(run_gpu(d, e, qstore=LOG), run_gpu(d, e, kernel=2, qstore=GLOBAL), f"n={n}")


@pytest.mark.parametrize("n", [40, 64, 100, 128])
def test_log_capacity_changes_no_bit(n):
    """Small logs force many apply rounds (Q through global memory between
    them, unpermuted until the last round)."""
    d, e = inputs.normal_problems(n, 300, F32, seed=700 + n)
    ref = run_gpu(d, e, qstore=LOG)
    # whole pages of 256 entries: every log runs out (1, 300, 7 n), or only
    # some do (n^2: about the mean log length)
    for cap in (1, 300, 7 * n, n * n):
        _same(run_gpu(d, e, qstore=LOG, log_entries=cap), ref, f"n={n} log_entries={cap}")


@pytest.mark.parametrize("n", [48, 64, 128])
def test_block_size_and_batch_change_no_bit(n):
    """The chase's block size and the batch only regroup the problems."""
    d, e = inputs.normal_problems(n, 5000 if n <= 64 else 1200, F32, seed=800 + n)
    ref = run_gpu(d, e, qstore=LOG)
    for tpb in (32, 96, 192):   # the chase's d and e take 8 n_pad bytes per thread
        _same(run_gpu(d, e, qstore=LOG, threads_per_block=tpb), ref, f"n={n} tpb={tpb}")
    small = run_gpu(d[:77], e[:77], qstore=LOG)
    for k in range(3):
        np.testing.assert_array_equal(small[k], ref[k][:77])


@pytest.mark.parametrize("n", [64, 128])
def test_mixed_hard_cases(n):
    d, e, labels, _ = inputs.mixed_problems(n, 700, F32, seed=3)
    a = run_gpu(d, e, qstore=LOG)
    check_parity(d, e, *a, oracle_ref(d, e, True), what=f"mixed n={n}")
    _same(a, run_gpu(d, e, kernel=2, qstore=GLOBAL), f"mixed n={n}")
    z = labels == inputs.CLASS_INDEX["zero"]
    assert np.all(a[0][z] == 0) and np.all(a[1][z] == np.eye(n, dtype=F32))


@pytest.mark.parametrize("n", [48, 128])
def test_scaled_classes(n):
    d, e, _ = inputs.scaled_problems(n, 400, F32, seed=11)
    a = run_gpu(d, e, qstore=LOG)
    check_parity(d, e, *a, oracle_ref(d, e, True), what=f"scaled n={n}")


@pytest.mark.parametrize("n", [50, 128])
def test_budget_exhaustion_and_unsorted(n):
    d, e = inputs.normal_problems(n, 400, F32, seed=900 + n)
    for kw in (dict(max_sweeps_per_n=1), dict(no_sort=True)):
        a = run_gpu(d, e, qstore=LOG, **kw)
        _same(a, run_gpu(d, e, kernel=2, qstore=GLOBAL, **kw), f"n={n} {kw}")
        if "max_sweeps_per_n" in kw:
            # the count of unconverged off-diagonals follows the oracle's up
            # to the rounding of deflation decisions, which moves it by a few
            # after n implicit steps
            ref = oracle_ref(d, e, True, maxit_per_n=1).info
            assert np.all(a[2] > 0) and np.all(ref > 0)
            assert np.abs(a[2] - ref).mean() <= 2 and np.abs(a[2] - ref).max() <= 8


@pytest.mark.parametrize("n", [64, 96])
def test_pg_and_back_transform(n):
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    batch = 500
    d, e = inputs.normal_problems(n, batch, F32, seed=1000 + n)
    _same(run_gpu(d, e, qstore=LOG, update_scheme=1), run_gpu(d, e, kernel=2, qstore=GLOBAL, update_scheme=1),
          f"pg n={n}")
    Z = inputs.orthogonal_bases(n, batch, F32, seed=1001)
    dev = torch.device("cuda:0")
    outs = []
    for kw in (dict(qstore=LOG), dict(qstore=LOG, log_entries=3 * n), dict(kernel=2, qstore=GLOBAL)):
        lam, V, info = bstq.solve(torch.from_numpy(d).to(dev), torch.from_numpy(e).to(dev), jobz=True,
                                  Z=torch.from_numpy(Z).to(dev), **kw)
        torch.cuda.synchronize()
        outs.append((lam.cpu().numpy(), V.cpu().numpy(), info.cpu().numpy()))
    _same(outs[0], outs[2], f"back_transform n={n}")
    _same(outs[1], outs[2], f"back_transform n={n}, small log")


@pytest.mark.parametrize("n", [33, 64, 127])
def test_unaligned_q(n):
    """Q that starts 4 bytes off an 8-byte boundary (and odd n) takes the
    single-float accesses; the bytes are the same."""
    import torch
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    batch = 300
    d, e = inputs.normal_problems(n, batch, F32, seed=1100 + n)
    ref = run_gpu(d, e, qstore=LOG)
    dev = torch.device("cuda:0")
    buf = torch.full((batch * n * n + 1,), float("nan"), dtype=torch.float32, device=dev)
    Q = buf[1:].view(batch, n, n)
    assert Q.data_ptr() % 8 != 0
    lam, Qo, info = bstq.solve(torch.from_numpy(d).to(dev), torch.from_numpy(e).to(dev), jobz=True, Q=Q,
                               qstore=LOG)
    torch.cuda.synchronize()
    _same((lam.cpu().numpy(), Qo.cpu().numpy(), info.cpu().numpy()), ref, f"unaligned n={n}")


def test_rejected_forms():
    from symmetric_tridiagonal_eigensolver_gb300 import bstq
    d, e = inputs.normal_problems(64, 10, F32, seed=1)
    for kw in (dict(threads_per_block=1024),):   # 1024 threads: 512 KB of d and e
        with pytest.raises(bstq.BstqError):
            run_gpu(d, e, qstore=LOG, **kw)
    d, e = inputs.normal_problems(32, 10, F32, seed=1)
    with pytest.raises(bstq.BstqError):
        run_gpu(d, e, qstore=LOG)
    d, e = inputs.normal_problems(64, 10, np.float64, seed=1)
    with pytest.raises(bstq.BstqError):
        run_gpu(d, e, qstore=LOG)
