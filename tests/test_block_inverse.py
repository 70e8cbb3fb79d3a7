"""The blocked unit-lower-triangular inverse of the prefill's chunk solve, X = (I + A)^-1 with A
strictly lower 64 x 64 (CPU, fp64): the four 16 x 16 diagonal blocks by forward substitution,
then merges X_[10] = -X_[11] A_[10] X_[00] from 16 to 32 rows and from 32 to 64 rows, in the
kernel's order (level two: Y = A[32:64, 0:32] X[0:32, 0:32], then X[32:64, 0:32] = -X[32:64, 32:64] Y).
Compared with a library inverse."""
import numpy as np


def _substitute(L):
    """(I + L)^-1 for a strictly lower L, one column at a time by forward substitution."""
    n = L.shape[0]
    X = np.zeros((n, n))
    for s in range(n):
        for r in range(n):
            X[r, s] = 1.0 if r == s else (0.0 if r < s else -L[r, s:r] @ X[s:r, s])
    return X


def _blocked_inverse(A):
    X = np.zeros((64, 64))
    for b in range(4):
        sl = slice(16 * b, 16 * b + 16)
        X[sl, sl] = _substitute(A[sl, sl])
    for b0 in (0, 32):  # level 1: 16 -> 32
        top, bot = slice(b0, b0 + 16), slice(b0 + 16, b0 + 32)
        X[bot, top] = -X[bot, bot] @ (A[bot, top] @ X[top, top])
    Y = A[32:64, 0:32] @ X[0:32, 0:32]  # level 2: 32 -> 64
    X[32:64, 0:32] = -X[32:64, 32:64] @ Y
    return X


def test_blocked_inverse_equals_the_library_inverse():
    rng = np.random.default_rng(7)
    for scale in (0.05, 0.3, 1.0):
        A = np.tril(rng.standard_normal((64, 64)) * scale, -1)
        ref = np.linalg.inv(np.eye(64) + A)
        got = _blocked_inverse(A)
        # scale 1 makes the inverse's entries grow to ~1e6: both sides then carry ~1e-16 relative
        # rounding amplified by that growth, so compare relative to the largest entry
        size = max(1.0, np.abs(ref).max())
        assert np.abs(got - ref).max() <= 1e-8 * size
        assert np.abs(got @ (np.eye(64) + A) - np.eye(64)).max() <= 1e-8 * size
        assert np.all(np.triu(got, 1) == 0.0) and np.all(np.diag(got) == 1.0)


def test_substitution_alone_is_the_inverse_of_a_small_block():
    rng = np.random.default_rng(8)
    L = np.tril(rng.standard_normal((16, 16)), -1)
    assert np.abs(_substitute(L) @ (np.eye(16) + L) - np.eye(16)).max() < 1e-9
