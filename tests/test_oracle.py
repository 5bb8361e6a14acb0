"""Pins for the CPU oracle, checked against what the pages and the mathematics fix.

Each test targets mistakes an oracle could plausibly make: a dropped or
inverted scale, a transposed operand (K Q^T instead of Q K^T, or V^T), a
wrong sign in the exponent, an off-by-one causal mask, a missing max shift,
a wrong LSE, a wrong normaliser.
"""
import math

import numpy as np
import pytest

import oracle
from oracle.tiled_model import tiled_attention
from conftest import read_golden


def one_head(q, k, v):
    """Wrap [N, d] matrices as [1, 1, N, d] float32 arrays."""
    return tuple(np.asarray(x, dtype=np.float32)[None, None] for x in (q, k, v))


def brute_force(q, k, v, scale, causal):
    """Materialise the full score matrix, softmax it, multiply by V (fp64).

    The plain "standard attention" that every page compares against, written
    independently of the oracle: exp of the max-shifted matrix, normalised
    by its row sums.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    s = np.einsum("bhid,bhjd->bhij", q, k) * scale
    if causal:
        nq, nk = s.shape[-2:]
        s = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None], s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    e = np.exp(s - mx)
    den = e.sum(axis=-1, keepdims=True)
    return np.einsum("bhij,bhjd->bhid", e / den, v), (mx + np.log(den))[..., 0]


# --------------------------------------------------------------------------
# Worked example: "Deep Learning - Flash Attention", "An Example"

WORKED_Q = np.array([[1, 2, 3, 4], [2, 1, 0, -1], [4, 3, 2, 1], [-1, 0, 1, 2]], dtype=np.float64)
WORKED_K = 2.0 * np.eye(4)
WORKED_V = np.eye(4)


def test_worked_example_scores_reproduced():
    g = read_golden("worked_example_4x4.txt")
    s = WORKED_Q @ WORKED_K.T * g["scale"][0]
    np.testing.assert_array_equal(s[0:2, 0:2].ravel(), g["S11"])
    np.testing.assert_array_equal(s[0:2, 2:4].ravel(), g["S12"])


def test_worked_example_oracle_rows():
    g = read_golden("worked_example_4x4.txt")
    dp = int(g["decimals"][0])
    o, lse = oracle.attention(*one_head(WORKED_Q, WORKED_K, WORKED_V), g["scale"][0])
    np.testing.assert_array_equal(np.round(o[0, 0, 0], dp), g["O_row1"])
    np.testing.assert_array_equal(np.round(o[0, 0, 1], dp), g["O_row2"])
    # V = I: each output row is a probability row, summing to 1
    np.testing.assert_allclose(o[0, 0].sum(axis=1), 1.0, rtol=0, atol=1e-15)
    # LSE of query 1 = ln(e^1 + e^2 + e^3 + e^4)
    assert abs(lse[0, 0, 0] - math.log(sum(math.exp(x) for x in (1, 2, 3, 4)))) < 1e-14


def test_worked_example_intermediates_of_tiled_model():
    g = read_golden("worked_example_4x4.txt")
    dp = int(g["decimals"][0])
    trace = []
    o, lse = tiled_attention(WORKED_Q, WORKED_K, WORKED_V, g["scale"][0], 2, 2, trace=trace)
    step1, step2 = trace[0], trace[1]
    assert (step1["q_block"], step1["k_block"], step2["k_block"]) == (0, 0, 1)
    np.testing.assert_array_equal(step1["S"].ravel(), g["S11"])
    np.testing.assert_array_equal(step1["m"], g["m_after_K1"])
    np.testing.assert_array_equal(step2["S"].ravel(), g["S12"])
    np.testing.assert_array_equal(step2["m"], g["m_after_K2"])
    np.testing.assert_array_equal(np.round(step2["alpha"], dp), g["alpha_K2"])
    # running denominators: after K_1 both rows hold 1 + e^-1; after K_2 row 1
    # holds (1 + e^-1) e^-2 + (e^-1 + 1) and row 2 holds 1 + e^-1 + e^-2 + e^-3
    e = math.exp
    np.testing.assert_allclose(step1["l"], [1 + e(-1), 1 + e(-1)], rtol=1e-15)
    np.testing.assert_allclose(step2["l"], [(1 + e(-1)) * e(-2) + e(-1) + 1,
                                            1 + e(-1) + e(-2) + e(-3)], rtol=1e-15)
    np.testing.assert_array_equal(np.round(o[0], dp), g["O_row1"])
    np.testing.assert_array_equal(np.round(o[1], dp), g["O_row2"])
    o_ref, lse_ref = oracle.attention(*one_head(WORKED_Q, WORKED_K, WORKED_V), g["scale"][0])
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lse_ref[0, 0], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# Closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_uniform_scores_give_mean_of_values(causal):
    rng = np.random.default_rng(11)
    N, d = 37, 8
    q = np.zeros((N, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    o, lse = oracle.attention(*one_head(q, k, v), 0.3, causal)
    v32 = v.astype(np.float32).astype(np.float64)
    for i in range(N):
        n_in = i + 1 if causal else N
        np.testing.assert_allclose(o[0, 0, i], v32[:n_in].mean(axis=0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(n_in)) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_identity_values_give_probability_rows(causal):
    """V = I: O[i, j] is the weight of key j, so O[i, j] / O[i, j'] must be
    exp(s_ij - s_ij') with s = scale * q_i . k_j, rows sum to 1, and under
    the causal mask every key after the query has weight 0."""
    rng = np.random.default_rng(12)
    N = d = 16
    q = rng.standard_normal((N, d)).astype(np.float32)
    k = rng.standard_normal((N, d)).astype(np.float32)
    scale = 0.37
    o, _ = oracle.attention(*one_head(q, k, np.eye(N)), scale, causal)
    o = o[0, 0]
    np.testing.assert_allclose(o.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    for i in range(N):
        for j in range(N):
            if causal and j > i:
                assert o[i, j] == 0.0
                continue
            sij = scale * sum(float(q[i, t]) * float(k[j, t]) for t in range(d))
            si0 = scale * sum(float(q[i, t]) * float(k[0, t]) for t in range(d))
            assert math.isclose(o[i, j] / o[i, 0], math.exp(sij - si0), rel_tol=1e-12)


def test_one_dominant_key_returns_its_value():
    """Query i scores 40 on key star[i] and 0 on every other key, so its
    output is v[star[i]] up to a weight error of (N-1) e^-40."""
    rng = np.random.default_rng(13)
    N = d = 16
    star = np.arange(N) * 7 % N          # a permutation of the keys
    q = np.eye(N)
    k = np.zeros((N, d))
    k[star] = 40.0 * np.eye(N)
    v = rng.standard_normal((N, d))
    o, _ = oracle.attention(*one_head(q, k, v), 1.0, False)
    v32 = v.astype(np.float32)
    for i in range(N):
        np.testing.assert_allclose(o[0, 0, i], v32[star[i]], rtol=0, atol=1e-14)


def test_single_key_returns_v0_and_its_score():
    rng = np.random.default_rng(14)
    q, k, v = (rng.standard_normal((1, 5)).astype(np.float32) for _ in range(3))
    o, lse = oracle.attention(*one_head(q, k, v), 0.5, False)
    np.testing.assert_array_equal(o[0, 0, 0], v[0].astype(np.float64))
    s = 0.5 * sum(float(a) * float(b) for a, b in zip(q[0], k[0]))
    assert abs(lse[0, 0, 0] - s) < 1e-15


# --------------------------------------------------------------------------
# Invariants

def test_constant_per_row_shift_leaves_output_unchanged():
    """Append a column c_i to Q and a ones column to K: every score of row i
    grows by scale * c_i, so O is unchanged and LSE moves by scale * c_i."""
    rng = np.random.default_rng(15)
    N, d, scale = 20, 6, 0.4
    q, k, v = (rng.standard_normal((N, d)).astype(np.float32) for _ in range(3))
    c = np.round(rng.uniform(-50, 50, N)).astype(np.float32)
    q2 = np.concatenate([q, c[:, None]], axis=1)
    k2 = np.concatenate([k, np.ones((N, 1), np.float32)], axis=1)
    v2 = np.concatenate([v, np.zeros((N, 1), np.float32)], axis=1)
    o1, l1 = oracle.attention(*one_head(q, k, v), scale)
    o2, l2 = oracle.attention(*one_head(q2, k2, v2), scale)
    np.testing.assert_allclose(o2[..., :d], o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, (scale * c.astype(np.float64))[None, None], rtol=0, atol=1e-12)


def test_permuting_keys_with_values_leaves_output_unchanged():
    rng = np.random.default_rng(16)
    N, d = 31, 7
    q, k, v = (rng.standard_normal((N, d)).astype(np.float32) for _ in range(3))
    perm = rng.permutation(N)
    o1, l1 = oracle.attention(*one_head(q, k, v), 0.5)
    o2, l2 = oracle.attention(*one_head(q, k[perm], v[perm]), 0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_output_is_linear_in_values():
    rng = np.random.default_rng(17)
    N, d = 19, 4
    q, k = (rng.standard_normal((N, d)).astype(np.float32) for _ in range(2))
    # quarter-integers, so that 2 v1 - v2 / 2 is exact in float32
    v1, v2 = (rng.integers(-16, 17, (N, d)) / 4.0 for _ in range(2))
    o1, _ = oracle.attention(*one_head(q, k, v1), 0.5)
    o2, _ = oracle.attention(*one_head(q, k, v2), 0.5)
    o3, _ = oracle.attention(*one_head(q, k, 2.0 * v1 - 0.5 * v2), 0.5)
    np.testing.assert_allclose(o3, 2.0 * o1 - 0.5 * o2, rtol=0, atol=1e-13)


def test_queries_are_independent():
    """Changing query row 5 changes output row 5 only."""
    rng = np.random.default_rng(18)
    N, d = 12, 4
    q, k, v = (rng.standard_normal((N, d)).astype(np.float32) for _ in range(3))
    o1, _ = oracle.attention(*one_head(q, k, v), 0.5)
    q[5] += 1.0
    o2, _ = oracle.attention(*one_head(q, k, v), 0.5)
    changed = np.abs(o1 - o2).max(axis=-1)[0, 0] > 0
    assert changed.tolist() == [i == 5 for i in range(N)]


# --------------------------------------------------------------------------
# Brute force and the tiled recurrence on small random inputs

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [False, True])
def test_matches_materialised_softmax(seed, causal):
    rng = np.random.default_rng(100 + seed)
    B, H = 1 + seed % 2, 1 + seed % 3
    N, d = int(rng.integers(1, 65)), int(rng.integers(1, 17))
    q, k, v = (rng.standard_normal((B, H, N, d)).astype(np.float32) for _ in range(3))
    scale = float(rng.uniform(0.05, 2.0))
    o, lse = oracle.attention(q, k, v, scale, causal)
    ob, lb = brute_force(q, k, v, scale, causal)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


@pytest.mark.parametrize("bq,bk", [(1, 1), (2, 3), (5, 4), (64, 64), (3, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_recurrence_reaches_three_pass_result(bq, bk, causal):
    rng = np.random.default_rng(bq * 10 + bk)
    N, d = 45, 6
    q, k, v = (rng.standard_normal((N, d)).astype(np.float32) for _ in range(3))
    o_t, l_t = tiled_attention(q, k, v, 0.6, bq, bk, causal)
    o, l = oracle.attention(*one_head(q, k, v), 0.6, causal)
    np.testing.assert_allclose(o_t, o[0, 0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l_t, l[0, 0], rtol=0, atol=1e-13)


def test_large_scores_do_not_overflow():
    """The max shift makes scores of several thousand safe (exp would overflow)."""
    q = np.array([[30.0, 30.0], [-30.0, 0.0]], dtype=np.float32)
    k = np.array([[40.0, 40.0], [39.0, 40.0], [0.0, 0.0]], dtype=np.float32)
    v = np.array([[1.0, 0.0], [0.0, 1.0], [2.0, 2.0]], dtype=np.float32)
    q3 = np.concatenate([q, q[:1]])
    o, lse = oracle.attention(*one_head(q3, k, v), 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    # row 0: scores 2400, 2370, 0 -> weight of key 0 is 1 / (1 + e^-30)
    w0 = 1.0 / (1.0 + math.exp(-30.0))
    w1 = math.exp(-30.0) / (1.0 + math.exp(-30.0))
    np.testing.assert_allclose(o[0, 0, 0], [w0, w1], rtol=1e-13)
    assert abs(lse[0, 0, 0] - (2400.0 + math.log1p(math.exp(-30.0)))) < 1e-10


# --------------------------------------------------------------------------
# The row-subset API and threading

def test_row_subset_and_thread_count_do_not_change_results():
    rng = np.random.default_rng(19)
    q, k, v = (rng.standard_normal((2, 3, 50, 8)).astype(np.float32) for _ in range(3))
    o_full, l_full = oracle.attention(q, k, v, 0.35, True, threads=1)
    rows = np.array([0, 49, 50, 123, 299, 7], dtype=np.int64)
    o_r, l_r = oracle.attention_rows(q, k, v, 0.35, True, rows, threads=4)
    np.testing.assert_array_equal(o_r, o_full.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(l_r, l_full.reshape(-1)[rows])
    o_m, _ = oracle.attention(q, k, v, 0.35, True, threads=7)
    np.testing.assert_array_equal(o_m, o_full)


def test_bad_rows_are_rejected():
    q = np.zeros((1, 1, 4, 2), np.float32)
    with pytest.raises(RuntimeError):
        oracle.attention_rows(q, q, q, 1.0, False, np.array([4]))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q[..., :1], q, 1.0, False, np.array([0]))


# --------------------------------------------------------------------------
# Cross-attention shapes: Nq != Nk and d_v != d_k ("Transformer Attention: A
# Mathematical Deep Dive", "The Attention Formula": Q (n, d_k), K (m, d_k),
# V (m, d_v))

@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [False, True])
def test_cross_shapes_match_materialised_softmax(seed, causal):
    rng = np.random.default_rng(200 + seed)
    B, H = 1 + seed % 2, 2
    nq, nk = int(rng.integers(1, 50)), int(rng.integers(1, 50))
    dk, dv = int(rng.integers(1, 12)), int(rng.integers(1, 12))
    q = rng.standard_normal((B, H, nq, dk)).astype(np.float32)
    k = rng.standard_normal((B, H, nk, dk)).astype(np.float32)
    v = rng.standard_normal((B, H, nk, dv)).astype(np.float32)
    o, lse = oracle.attention(q, k, v, 0.7, causal)
    assert o.shape == (B, H, nq, dv)
    ob, lb = brute_force(q, k, v, 0.7, causal)
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_cross_shapes_reduce_to_self_attention_pieces():
    """Queries 0..nq-1 against the first nk keys equal the self-attention of
    the padded problem restricted to those keys when causal (rows i < nk see
    only keys j <= i either way)."""
    rng = np.random.default_rng(300)
    n, d = 40, 6
    q, k, v = (rng.standard_normal((1, 1, n, d)).astype(np.float32) for _ in range(3))
    o_sq, l_sq = oracle.attention(q, k, v, 0.5, True)
    o_x, l_x = oracle.attention(q[:, :, :25], k[:, :, :30], v[:, :, :30], 0.5, True)
    np.testing.assert_array_equal(o_x, o_sq[:, :, :25])
    np.testing.assert_array_equal(l_x, l_sq[:, :, :25])


def test_values_wider_than_keys_are_column_independent():
    """Each output column depends on its own value column only: splitting V's
    columns splits O's."""
    rng = np.random.default_rng(301)
    q = rng.standard_normal((1, 1, 9, 3)).astype(np.float32)
    k = rng.standard_normal((1, 1, 13, 3)).astype(np.float32)
    v = rng.standard_normal((1, 1, 13, 10)).astype(np.float32)
    o, _ = oracle.attention(q, k, v, 0.8)
    o1, _ = oracle.attention(q, k, v[..., :4], 0.8)
    o2, _ = oracle.attention(q, k, v[..., 4:], 0.8)
    np.testing.assert_array_equal(o, np.concatenate([o1, o2], axis=-1))
