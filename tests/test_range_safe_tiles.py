"""The exponent-range scheme of the tensor-core prefill, restated in float32 numpy (no GPU).

Over a 64-token chunk at the decay bound (g = -5 on every channel) exp(-Gam) reaches e^{320},
beyond fp32. The chunkwise form ("Kimi K3 Explained", researchpapers.dev, "Architecture at a
glance": bounding the log-decay makes the causal tiles dense matmuls) needs
exp(Gam_r - Gam_s) for s <= r, which is <= 1, but the plain factorisation (K gam)(K / gam)^T
forms the out-of-range factors separately. The kernel builds the intra-chunk matrices from
three 32 x 32 tiles with in-range factors instead:

* rows and columns 0..31: factors exp(Gam_r - Gam_15) and exp(Gam_15 - Gam_s);
* rows and columns 32..63: the same with Gam_47;
* rows 32..63 x columns 0..31: exp(Gam_r - Gam_31) and exp(Gam_31 - Gam_s), both <= 1;

and K+ = K gam, Q+ = Q gam, Khat = K gam_63 / gam from products of in-range factors. This test
builds those factors in float32 exactly as listed and checks them against the fp64 definitions.
Inside a diagonal tile the non-causal entries (r < s) are exp(Gam_r - Gam_s), up to e^{155}: they
overflow in fp32, so the read-out must drop them by selection, never by multiplying by zero.
"""

import numpy as np
import pytest

C, HALF = 64, 32


def _gam_cumsum(g):
    return np.cumsum(g, axis=0)


def _tiles_fp32(k, q, Gam):
    """A0 = K exp(Gam_r - Gam_s) K^T (all r, s) and Q's version, from the three range-safe tiles."""
    f32 = np.float32
    G = Gam.astype(f32)
    k, q = k.astype(f32), q.astype(f32)
    Ak = np.zeros((C, C), f32)
    Aq = np.zeros((C, C), f32)
    for lo, ref in ((0, G[15]), (HALF, G[47])):  # diagonal halves
        rows = slice(lo, lo + HALF)
        f = np.exp(G[rows] - ref)
        fi = np.exp(ref - G[rows])
        Ak[rows, rows] = (k[rows] * f) @ (k[rows] * fi).T
        Aq[rows, rows] = (q[rows] * f) @ (k[rows] * fi).T
    lo_r, hi_r = slice(HALF, C), slice(0, HALF)  # off-diagonal tile: rows 32..63, columns 0..31
    e_row = np.exp(G[lo_r] - G[31])
    e_col = np.exp(G[31] - G[hi_r])
    assert e_row.max() <= 1.0 and e_col.max() <= 1.0
    Ak[lo_r, hi_r] = (k[lo_r] * e_row) @ (k[hi_r] * e_col).T
    Aq[lo_r, hi_r] = (q[lo_r] * e_row) @ (k[hi_r] * e_col).T
    return Ak, Aq


def _state_operands_fp32(k, q, Gam):
    """K+ = K exp(Gam_r), Q+ = Q exp(Gam_r), Khat = K exp(Gam_63 - Gam_r) as the kernel forms them."""
    f32 = np.float32
    G = Gam.astype(f32)
    k, q = k.astype(f32), q.astype(f32)
    kp, qp, kh = (np.zeros_like(k) for _ in range(3))
    a, b = slice(0, HALF), slice(HALF, C)
    f0 = np.exp(G[a] - G[15])                    # rows 0..31: <= e^80
    kp[a], qp[a] = k[a] * f0 * np.exp(G[15]), q[a] * f0 * np.exp(G[15])
    kh[a] = k[a] * np.exp(G[31] - G[a]) * np.exp(G[63] - G[31])
    f1 = np.exp(G[b] - G[31])                    # rows 32..63: <= 1
    kp[b], qp[b] = k[b] * f1 * np.exp(G[31]), q[b] * f1 * np.exp(G[31])
    kh[b] = k[b] * np.exp(G[47] - G[b]) * np.exp(G[63] - G[47])
    return kp, qp, kh


@pytest.mark.parametrize("kind", ["saturated", "random", "zero"])
def test_range_safe_tiles_match_the_definitions(kind):
    rng = np.random.default_rng({"saturated": 0, "random": 1, "zero": 2}[kind])
    d = 32
    k = rng.standard_normal((C, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((C, d))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    g = {"saturated": np.full((C, d), -5.0),
         "random": -5.0 / (1.0 + np.exp(-rng.standard_normal((C, d)))),
         "zero": np.zeros((C, d))}[kind]
    Gam = _gam_cumsum(g)
    # fp64 definitions on the causal part: sum_c k_r,c k_s,c exp(Gam_r,c - Gam_s,c), s <= r
    E = np.exp(Gam[:, None, :] - Gam[None, :, :])                 # [r, s, c]
    mask = np.tril(np.ones((C, C), bool))
    Ak_ref = np.where(mask, np.einsum("rc,sc,rsc->rs", k, k, np.where(mask[..., None], E, 0.0)), 0.0)
    Aq_ref = np.where(mask, np.einsum("rc,sc,rsc->rs", q, k, np.where(mask[..., None], E, 0.0)), 0.0)
    with np.errstate(over="ignore", invalid="ignore"):
        Ak, Aq = _tiles_fp32(k, q, Gam)
    assert np.all(np.isfinite(Ak[mask])) and np.all(np.isfinite(Aq[mask]))
    if kind == "saturated":  # the discarded triangle does overflow: masking must select
        assert not np.all(np.isfinite(Ak[~mask]))
    np.testing.assert_allclose(np.where(mask, Ak, 0.0), Ak_ref, rtol=0, atol=2e-6)
    np.testing.assert_allclose(np.where(mask, Aq, 0.0), Aq_ref, rtol=0, atol=2e-6)
    kp, qp, kh = _state_operands_fp32(k, q, Gam)
    for got, want in ((kp, k * np.exp(Gam)), (qp, q * np.exp(Gam)), (kh, k * np.exp(Gam[63] - Gam))):
        assert np.all(np.isfinite(got))
        np.testing.assert_allclose(got, want, rtol=2e-5, atol=1e-30)


def test_the_plain_factorisation_overflows_fp32_at_the_bound():
    """Why the tiles: K / gam alone is e^{315} at the last row when g = -5 everywhere."""
    Gam = _gam_cumsum(np.full((C, 4), -5.0)).astype(np.float32)
    with np.errstate(over="ignore"):
        inv = np.exp(-Gam)
    assert np.isinf(inv[-1]).all()
    # every factor of the tiled scheme stays within e^{+-80}
    assert (Gam[:HALF] - Gam[15]).max() <= 80 and (Gam[HALF:] - Gam[47]).min() >= -80
