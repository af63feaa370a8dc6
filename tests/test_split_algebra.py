"""The algebra behind the split along the sequence, in fp64 on the oracle (no GPU).

"Inside Kimi K3's Architecture", "Kimi Delta Attention: the linear core": the per-token
transition (I - beta k k^T) Diag(alpha) does not depend on the state, so over a segment that
starts from S_start

    S_t = M_t S_start + S_loc_t,      o_t = o_loc_t + S_start^T (M_t^T q_t),

with S_loc, o_loc the run from a zero state and M_t the product of the transitions. With v = 0
and the identity as the initial state the recurrence itself yields M_t (as its state) and
q~_t = M_t^T q_t (as its output). The split path computes these three runs and joins them; here
the join is checked against the unsplit run.
"""

import numpy as np
import pytest

import oracle


def _inputs(rng, T, H, d, decay):
    q = rng.standard_normal((1, T, H, d))
    k = rng.standard_normal((1, T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, d))
    g = -5.0 * decay / (1.0 + np.exp(-rng.standard_normal((1, T, H, d))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H))))
    return q, k, v, g, beta


@pytest.mark.parametrize("T,cuts,decay", [(40, [17], 1.0), (64, [16, 40], 0.02), (33, [1, 32], 0.1)])
def test_segments_join_to_the_unsplit_run(T, cuts, decay):
    rng = np.random.default_rng(T + len(cuts))
    H, d = 2, 8
    q, k, v, g, beta = _inputs(rng, T, H, d, decay)
    S0 = 0.1 * rng.standard_normal((1, H, d, d))
    o_ref, s_ref = oracle.recurrent(q, k, v, g, beta, initial_state=S0)
    eye = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    bounds = [0] + cuts + [T]
    S_start = S0
    o = np.zeros_like(o_ref)
    for a, b in zip(bounds[:-1], bounds[1:]):
        seg = [x[:, a:b] for x in (q, k, v, g, beta)]
        o_loc, s_loc = oracle.recurrent(*seg, initial_state=np.zeros_like(S0))         # local pass
        qt, M = oracle.recurrent(seg[0], seg[1], np.zeros_like(seg[2]), seg[3], seg[4],
                                 initial_state=eye)                                    # transition pass
        for h in range(H):
            o[0, a:b, h] = o_loc[0, :, h] + qt[0, :, h] @ S_start[0, h]                # q~ S_start
        S_start = np.einsum("hij,hjk->hik", M[0], S_start[0])[None] + s_loc           # scan step
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(S_start, s_ref, rtol=1e-10, atol=1e-10)


def test_transition_of_a_segment_is_the_product_of_the_token_transitions():
    """M from the v = 0 identity run equals the explicit product of (I - beta k k^T) Diag(alpha)."""
    rng = np.random.default_rng(5)
    T, H, d = 9, 1, 6
    q, k, v, g, beta = _inputs(rng, T, H, d, 1.0)
    eye = np.eye(d)[None, None]
    _, M = oracle.recurrent(q, k, np.zeros_like(v), g, beta, initial_state=eye)
    want = np.eye(d)
    for t in range(T):
        kt = k[0, t, 0]
        step = (np.eye(d) - beta[0, t, 0] * np.outer(kt, kt)) @ np.diag(np.exp(g[0, t, 0]))
        want = step @ want
    np.testing.assert_allclose(M[0, 0], want, rtol=1e-12, atol=1e-12)
