"""bstq: batched symmetric tridiagonal eigensolver for one NVIDIA GB300."""
