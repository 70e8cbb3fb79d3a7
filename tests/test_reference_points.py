"""The reference-point factorisation of the intra-chunk products (CPU, fp64 numpy).

Within a 64-token chunk, with G the inclusive cumulative log-decay per key channel,
  A_rs = sum_c k_rc k_sc e^{G_rc - G_sc}  (s < r)   and   M_rs = sum_c q_rc k_sc e^{G_rc - G_sc}  (s <= r)
are products of reference-scaled rows, X_r = x_r e^{G_r - R} and Y_s = k_s e^{R - G_s}, for any
reference R: the two 32-token diagonal blocks use R = G_15 and R = G_47, the block of rows >= 32
and columns < 32 uses R = G_47.  With g > -5 (Kimi K3 report walk-through, section 3.2 / Eq. 5)
every exponent in X, and in Y on the diagonal blocks, is at most 16 * 5 = 80 in magnitude (fp32
range); the off-diagonal Y factors are at most 1.  These checks pin that algebra and those bounds
in exact arithmetic; the GPU parity tests cover the kernels that use it."""
import numpy as np

C, HALF = 64, 32


def _chunk(seed, dk=8):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((C, dk))
    q = rng.standard_normal((C, dk))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((C, dk))))  # in (-5, 0)
    return q, k, g, np.cumsum(g, axis=0)


def _direct(x, k, G):
    """sum_c x_rc k_sc e^{G_rc - G_sc} for every (r, s)."""
    return np.einsum("rc,sc,rsc->rs", x, k, np.exp(G[:, None, :] - G[None, :, :]))


def _factored(x, k, G):
    """The same matrix on the lower blocks, assembled from reference-scaled rows."""
    out = np.zeros((C, C))
    for lo, R in ((0, G[15]), (HALF, G[47])):  # diagonal blocks, centred references
        rows = slice(lo, lo + HALF)
        X = x[rows] * np.exp(G[rows] - R)
        Y = k[rows] * np.exp(R - G[rows])
        out[rows, rows] = X @ Y.T
    R = G[47]  # rows >= 32, columns < 32
    X = x[HALF:] * np.exp(G[HALF:] - R)
    Y = k[:HALF] * np.exp(R - G[:HALF])
    out[HALF:, :HALF] = X @ Y.T
    return out


def test_factored_products_equal_the_definition_on_the_lower_blocks():
    for seed in range(5):
        q, k, g, G = _chunk(seed)
        lower = np.tril(np.ones((C, C), dtype=bool))
        for x in (k, q):  # A (strictly lower part used) and M (lower with the diagonal)
            d, f = _direct(x, k, G), _factored(x, k, G)
            scale = np.abs(d[lower]).max()
            assert np.abs(d[lower] - f[lower]).max() <= 1e-12 * scale


def test_exponents_stay_in_fp32_range_under_the_decay_bound():
    for seed in range(5):
        _, _, g, G = _chunk(seed)
        for lo, ref in ((0, 15), (HALF, 47)):
            e = G[lo:lo + HALF] - G[ref]
            assert np.abs(e).max() <= 80.0  # 16 tokens of g > -5 on either side of the reference
        assert np.abs(G[HALF:] - G[47]).max() <= 80.0
        assert (G[47] - G[:HALF]).max() <= 0.0  # off-diagonal key factors are at most 1
    assert np.log(np.finfo(np.float32).max) > 80.0


def test_a_single_reference_per_chunk_would_leave_fp32_range():
    """The bound that rules out one reference for the whole chunk: g near -5 on every token puts
    e^{G_63 - G_0} near e^{-315}, far below the smallest fp32 normal (about e^{-87})."""
    g = np.full((C, 1), -4.99)
    G = np.cumsum(g, axis=0)
    assert G[-1, 0] - G[0, 0] < np.log(np.finfo(np.float32).tiny) - 200
