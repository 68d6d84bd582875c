"""Pins of the oracle's 19-tap WENO consumer against what the mathematics
fixes, independently of the oracle's own arithmetic.

The consumer (a reading: the pages name a 19-tap WENO consumer without its
formula) is the Godunov upwind squared gradient norm of a level set phi, built
from fifth-order WENO one-sided derivatives (Jiang & Shu 1996; Jiang & Peng
2000) at unit spacing, epsilon = 1e-6, in fp32.  What pins it:

- the WENO reconstruction rebuilt here from its definition: quadratic
  reconstructions matching three cell averages, ideal weights that reproduce
  the five-cell quartic reconstruction, smoothness indicators as integrals of
  the squared first and second derivatives over the reconstruction cell (all
  derived with numpy in fp64, not restated from the closed form);
- exact gradients of linear fields and of quadratics, and of a small quartic
  (where epsilon dominates the indicators and the ideal weights act alone);
- the upwind choice at a kink, outside and inside the level set;
- a constant field (background included) gives exactly 0;
- mirror and x<->y symmetry, bit for bit;
- the tap table against the brute-force neighbour lookup.
"""
import numpy as np
import pytest

import oracle
from tests import bruteforce

EPS = 1e-6


# ---------------------------------------------------------------------------
# WENO5 from its definition (fp64)
# ---------------------------------------------------------------------------

def _cell_average_rows(cells, degree):
    """Matrix M with M[i, p] = average of x**p over cells[i] = (lo, hi)."""
    M = np.zeros((len(cells), degree + 1))
    for i, (lo, hi) in enumerate(cells):
        for p in range(degree + 1):
            M[i, p] = (hi ** (p + 1) - lo ** (p + 1)) / ((p + 1) * (hi - lo))
    return M


def _weno_definition(v):
    """Left-biased WENO5 value at x=0 from the averages v[0..4] over the cells
    [-3,-2], [-2,-1], [-1,0], [0,1], [1,2]."""
    cells = [(-3, -2), (-2, -1), (-1, 0), (0, 1), (1, 2)]
    subs = [(0, 1, 2), (1, 2, 3), (2, 3, 4)]
    cand, beta, coef_at0 = [], [], []
    for sub in subs:
        M = _cell_average_rows([cells[i] for i in sub], 2)
        Minv = np.linalg.inv(M)                 # polynomial coefficients = Minv @ averages
        c = Minv @ np.array([v[i] for i in sub])
        P = np.polynomial.Polynomial(c)
        cand.append(P(0.0))
        b = 0.0
        for order in (1, 2):                    # integral over the cell [-1, 0] of (P^(l))^2
            Q = (P.deriv(order)) ** 2
            Qi = Q.integ()
            b += Qi(0.0) - Qi(-1.0)
        beta.append(b)
        row = np.zeros(5)                       # P_k(0) as a linear form in v
        row[list(sub)] = np.polynomial.polynomial.polyval(0.0, Minv)
        coef_at0.append(row)
    full = np.polynomial.polynomial.polyval(0.0, np.linalg.inv(_cell_average_rows(cells, 4)))
    A = np.array(coef_at0).T                    # 5 x 3: columns are the candidates' linear forms
    gamma, *_ = np.linalg.lstsq(A, full, rcond=None)
    assert np.allclose(A @ gamma, full, atol=1e-12)
    alpha = gamma / (EPS + np.array(beta)) ** 2
    return float(np.dot(alpha, cand) / alpha.sum()), gamma


def test_ideal_weights_from_the_definition():
    _, gamma = _weno_definition([1.0, 2.0, 3.0, 4.0, 5.0])
    np.testing.assert_allclose(gamma, [0.1, 0.6, 0.3], atol=1e-12)


def _line_grid(D, background_is_centre=True):
    """Voxels (k,0,0), k = -3..3, with phi(k) - phi(k-1) = D[k+2] for k = -2..3
    and phi(-3) = 0.  Returns (grid, phi rows, centre index)."""
    coords = np.array([[k, 0, 0] for k in range(-3, 4)], dtype=np.int32)
    g = oracle.OracleGrid(coords)
    vals = np.concatenate([[0.0], np.cumsum(D)]).astype(np.float32)   # phi at k = -3..3
    assert np.array_equal(np.diff(vals.astype(np.float64)), np.asarray(D, dtype=np.float64))
    phi = np.zeros(g.n + 1, dtype=np.float32)
    for k in range(-3, 4):
        phi[g.index(k, 0, 0)] = vals[k + 3]
    centre = g.index(0, 0, 0)
    phi[0] = vals[3] if background_is_centre else 0.0  # y and z taps then see no difference
    return g, phi, centre


def _godunov(minus, plus, outside):
    """Upwind rule (Osher & Fedkiw, the Godunov scheme for |grad phi|)."""
    if outside:
        return max(max(minus, 0.0) ** 2, min(plus, 0.0) ** 2)
    return max(min(minus, 0.0) ** 2, max(plus, 0.0) ** 2)


@pytest.mark.parametrize("seed", range(12))
def test_one_sided_derivatives_match_the_definition(seed):
    rng = np.random.default_rng(seed)
    # dyadic differences, so the partial sums are exact in fp32
    D = rng.integers(-256, 256, size=6) / 64.0
    if seed % 3 == 1:
        D[rng.integers(0, 6)] *= 40  # a jump: the nonlinear weights matter
    minus_def, _ = _weno_definition(D[0:5])
    plus_def, _ = _weno_definition(D[1:6][::-1])  # mirror image: cells read from the right
    g, phi, centre = _line_grid(D)
    c = float(phi[centre])
    scale = max(minus_def ** 2, plus_def ** 2)
    for outside in (True, False):
        got = g.weno_filter(phi, iso=c - 1.0 if outside else c + 1.0)[centre]
        want = _godunov(minus_def, plus_def, outside)
        assert abs(float(got) - want) <= 4e-5 * want + 1e-6 * scale, (outside, got, want, minus_def, plus_def)
    # both one-sided values are seen when each is the only candidate: make the
    # other side's contribution vanish by the sign rule
    if minus_def > 0 and plus_def > 0:
        np.testing.assert_allclose(np.sqrt(np.float64(g.weno_filter(phi, iso=c - 1.0)[centre])), minus_def,
                                   rtol=2e-5)
        np.testing.assert_allclose(np.sqrt(np.float64(g.weno_filter(phi, iso=c + 1.0)[centre])), plus_def,
                                   rtol=2e-5)


@pytest.mark.parametrize("seed", range(8))
def test_positive_differences_pin_each_side(seed):
    # all differences positive and without jumps: both derivatives are > 0, so
    # outside the result is minus^2 and inside plus^2 exactly by the rule
    rng = np.random.default_rng(100 + seed)
    D = rng.integers(32, 256, size=6) / 64.0
    minus_def, _ = _weno_definition(D[0:5])
    plus_def, _ = _weno_definition(D[1:6][::-1])
    assert minus_def > 0 and plus_def > 0
    g, phi, centre = _line_grid(D)
    c = float(phi[centre])
    np.testing.assert_allclose(np.sqrt(np.float64(g.weno_filter(phi, iso=c - 1.0)[centre])), minus_def, rtol=2e-5)
    np.testing.assert_allclose(np.sqrt(np.float64(g.weno_filter(phi, iso=c + 1.0)[centre])), plus_def, rtol=2e-5)


def _dense(lo, hi):
    r = np.arange(lo, hi + 1)
    return np.stack(np.meshgrid(r, r, r, indexing="ij"), -1).reshape(-1, 3).astype(np.int32)


def _interior(coords, lo, hi, margin=3):
    return np.all((coords >= lo + margin) & (coords <= hi - margin), axis=1)


@pytest.mark.parametrize("abc", [(1, 2, -2), (3, 0, 1), (-1, -1, 1)])
def test_linear_field_gives_its_gradient(abc):
    lo, hi = -5, 5
    g = oracle.OracleGrid(_dense(lo, hi))
    c = g.coords()
    a, b, d = abc
    phi = np.zeros(g.n + 1, dtype=np.float32)
    phi[1:] = a * c[:, 0] + b * c[:, 1] + d * c[:, 2] + 7
    out = g.weno_filter(phi, iso=0.0)[1:]
    inside = _interior(c, lo, hi)
    np.testing.assert_allclose(out[inside], a * a + b * b + d * d, rtol=1e-6)


def test_quadratic_field_gives_its_gradient():
    lo, hi = -6, 6
    g = oracle.OracleGrid(_dense(lo, hi))
    c = g.coords().astype(np.float64)
    phi = np.zeros(g.n + 1, dtype=np.float32)
    phi[1:] = (c ** 2).sum(1)
    for iso in (-1.0, 1000.0):  # everything outside, then everything inside
        out = g.weno_filter(phi, iso=iso)[1:]
        inside = _interior(c, lo, hi)
        np.testing.assert_allclose(out[inside], 4 * (c[inside] ** 2).sum(1), rtol=1e-5, atol=1e-5)


def test_small_quartic_uses_the_ideal_weights():
    # phi = s*x^4 with s tiny: the indicators are far below epsilon, so the
    # weights are the ideal ones and the scheme is exact for quartics.
    lo, hi = -6, 6
    s = 1e-8
    g = oracle.OracleGrid(_dense(lo, hi))
    c = g.coords().astype(np.float64)
    phi = np.zeros(g.n + 1, dtype=np.float32)
    phi[1:] = s * c[:, 0] ** 4
    inside = _interior(c, lo, hi) & (np.abs(c[:, 0]) >= 1)
    exact = 4 * s * np.abs(c[inside, 0]) ** 3
    for iso in (-1.0, 1.0):
        out = g.weno_filter(phi, iso=iso)[1:]
        np.testing.assert_allclose(np.sqrt(out[inside].astype(np.float64)), exact, rtol=1e-4)


@pytest.mark.parametrize("offset,expected", [(5.0, 0.0), (-5.0, 1.0)])
def test_upwind_choice_at_a_kink(offset, expected):
    # phi = |x| + offset: at x = 0 the left derivative is -1 and the right +1.
    # Outside (phi > 0) a minimum has no upwind gradient: exactly 0.  Inside,
    # both sides point away from the centre: 1.
    lo, hi = -4, 4
    g = oracle.OracleGrid(_dense(lo, hi))
    c = g.coords()
    phi = np.zeros(g.n + 1, dtype=np.float32)
    phi[1:] = np.abs(c[:, 0]) + offset
    phi[0] = 99.0
    centre = g.index(0, 0, 0)
    got = g.weno_filter(phi, iso=0.0)[centre]
    if expected == 0.0:
        assert got == 0.0
    else:
        np.testing.assert_allclose(got, expected, rtol=1e-6)


def _sparse_case(seed, n=600, side=9):
    rng = np.random.default_rng(seed)
    coords = np.unique(rng.integers(-side, side + 1, size=(n, 3)), axis=0).astype(np.int32)
    phi_of = {tuple(p): float(v) for p, v in zip(coords, rng.standard_normal(len(coords)).astype(np.float32))}
    return coords, phi_of


def _phi_rows(g, phi_of, background):
    phi = np.zeros(g.n + 1, dtype=np.float32)
    phi[0] = background
    for i, p in enumerate(g.coords(), start=1):
        phi[i] = phi_of[tuple(p)]
    return phi


@pytest.mark.parametrize("seed", range(3))
def test_constant_field_is_zero(seed):
    coords, _ = _sparse_case(seed)
    g = oracle.OracleGrid(coords)
    phi = np.full(g.n + 1, 2.5, dtype=np.float32)  # the background row too
    assert np.all(g.weno_filter(phi, iso=0.0) == 0.0)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("mirror", ["x", "y", "z", "swap_xy"])
def test_symmetries_bit_for_bit(seed, mirror):
    coords, phi_of = _sparse_case(seed)
    g = oracle.OracleGrid(coords)
    base = g.weno_filter(_phi_rows(g, phi_of, 0.25), iso=0.1)
    if mirror == "swap_xy":
        m = lambda p: (p[1], p[0], p[2])  # noqa: E731
    else:
        ax = "xyz".index(mirror)
        m = lambda p: tuple(-p[i] if i == ax else p[i] for i in range(3))  # noqa: E731
    coords2 = np.array([m(p) for p in coords], dtype=np.int32)
    phi2_of = {m(p): v for p, v in phi_of.items()}
    g2 = oracle.OracleGrid(coords2)
    other = g2.weno_filter(_phi_rows(g2, phi2_of, 0.25), iso=0.1)
    for i, p in enumerate(g.coords(), start=1):
        j = g2.index(*m(tuple(int(v) for v in p)))
        assert base[i].view(np.uint32) == other[j].view(np.uint32), (tuple(p), base[i], other[j])


def test_weno_taps_match_brute_force():
    coords, _ = _sparse_case(4, n=400, side=6)
    g = oracle.OracleGrid(coords)
    taps = g.taps(19)
    dense = bruteforce.Dense(bruteforce.tree_order(coords))
    offs = sorted({(k if a == 0 else 0, k if a == 1 else 0, k if a == 2 else 0)
                   for a in range(3) for k in range(-3, 4)})  # lexicographic (di, dj, dk)
    assert len(offs) == 19 and offs[9] == (0, 0, 0)
    want = np.stack([dense.neighbour(*d) for d in offs], axis=1)
    assert np.all(taps[0] == 0)
    np.testing.assert_array_equal(taps[1:].astype(np.int64), want)
