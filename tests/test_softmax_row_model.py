"""CPU model of one softmax row of the tensor-core attention kernel (attn_fwd_tc.cu).

The kernel walks a row's scores in tiles of 128 keys and keeps a running max m,
sum l and output O, built against the same m (the incremental form of the
max -> sum exp -> sum exp*v cascade).  Two rules decide when m moves:
  * the lazy rescale: m moves only when a tile's max exceeds it by more than
    2^8 (base-2 units), so every P stays <= 256;
  * speculation (non-causal D = 64): once m is finite, P is formed against it
    without scanning the tile.  A half row (64 keys) whose sum of P exceeds
    2^15 makes the kernel redo the row from the tile max (first half) or
    rescan the second half alone, with m + 15 bounding the first half.
This module restates both rules in numpy and checks, on rows built to take
every branch, that the result equals the plain softmax to rounding and that
no P ever exceeds the bound its rule promises.  The GPU tests check the kernel.
"""
import numpy as np
import pytest

THRESHOLD = 8.0      # lazy rescale, base-2 units
SPEC_LOG2 = 15.0     # speculation bound: every P <= 2^15
SPEC_MAX = 2.0 ** SPEC_LOG2
TILE, HALF = 128, 64


def row_forward(x2, v, speculate, skip_first_half_rescale=False):
    """x2: a row's scores in base-2 units (-inf = masked); v: [keys, d].
    Returns (O / l, lse in natural log, the largest P seen, the paths taken).
    skip_first_half_rescale plants a mistake for the test that the checks see it."""
    m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
    spec, pmax, paths = speculate, 0.0, []
    for t0 in range(0, len(x2), TILE):
        s, vt = x2[t0:t0 + TILE], v[t0:t0 + TILE]
        exact = not spec or m == -np.inf
        m_new = m
        while True:
            if exact:
                mt = s.max()
                m_new = mt if mt > m + THRESHOLD else m
            m_use = 0.0 if m_new == -np.inf else m_new
            p = np.exp2(s - m_use)
            if exact:
                paths.append("exact")
                break
            if not p[:HALF].sum() <= SPEC_MAX:   # a first half too large: redo from the tile max
                exact, spec = True, False
                continue
            if not p[HALF:].sum() <= SPEC_MAX:   # only the second half: rescan it alone
                spec = False
                m_new = max(s[HALF:].max(), m + SPEC_LOG2)
                if not skip_first_half_rescale:
                    p[:HALF] *= np.exp2(m - m_new)
                p[HALF:] = np.exp2(s[HALF:] - m_new)
                paths.append("second half rescanned")
            else:
                paths.append("speculated")
            break
        pmax = max(pmax, float(p.max()))
        alpha = np.exp2(m - m_new) if (m_new != m and m_new != -np.inf) else 1.0
        l = l * alpha + p.sum()
        o = o * alpha + p @ vt
        m = m_new
    return o / l, (m + np.log2(l)) * np.log(2.0), pmax, paths


def plain_softmax(x2, v):
    w = np.exp2(x2 - x2.max())
    return (w @ v) / w.sum(), (x2.max() + np.log2(w.sum())) * np.log(2.0)


def rows():
    rng = np.random.default_rng(0)
    n = 5 * TILE
    out = []
    # levels per half tile (natural-log units, as in the GPU test of rising scores)
    for levels in ([[0, 0], [0, 14], [30, 30], [31, 29], [5, 60]], [[0, 0], [1, 0], [20, 20], [20, 21], [40, 40]]):
        sc = np.repeat(np.asarray(levels, dtype=np.float64).reshape(-1), HALF) + 0.5 * rng.standard_normal(n)
        out.append(sc)
    out.append(rng.standard_normal(n))                    # random scores: speculation never fails
    out.append(np.linspace(0, 400, n))                    # rising in every tile
    out.append(np.linspace(400, 0, n))                    # falling: the first tile holds the max
    masked = rng.standard_normal(n) * 3
    masked[:200] = -np.inf                                # a fully masked first tile, then keys
    out.append(masked)
    return out


@pytest.mark.parametrize("speculate", [False, True])
@pytest.mark.parametrize("k", range(6))
def test_row_matches_plain_softmax(speculate, k):
    x = rows()[k]
    x2 = x * np.log2(np.e)
    v = np.random.default_rng(k).standard_normal((len(x), 8))
    o, lse, pmax, _ = row_forward(x2, v, speculate)
    ro, rlse = plain_softmax(x2, v)
    np.testing.assert_allclose(o, ro, rtol=1e-9, atol=1e-12)
    assert abs(lse - rlse) <= 1e-9 * max(1.0, abs(rlse))
    assert pmax <= (SPEC_MAX if speculate else 2.0 ** THRESHOLD)


def test_every_branch_is_taken():
    seen = set()
    for x in rows():
        seen.update(row_forward(x * np.log2(np.e), np.ones((len(x), 1)), True)[3])
    assert seen == {"exact", "speculated", "second half rescanned"}
    # the first-half failure shows as an exact tile after speculation began
    paths = row_forward(rows()[1] * np.log2(np.e), np.ones((5 * TILE, 1)), True)[3]
    assert paths[0] == "exact" and "exact" in paths[1:]


def test_a_planted_mistake_is_caught():
    """Leaving the first half's P against the old m when only the second half is
    rescanned must break the match with the plain softmax."""
    # second tile: a first half that passes (sum of P about 2^14.7) beside a
    # second half that does not, so both halves carry weight in the result
    rng = np.random.default_rng(3)
    x = np.repeat(np.asarray([0, 0, 6, 8], dtype=np.float64), HALF) + 0.3 * rng.standard_normal(2 * TILE)
    x2 = x * np.log2(np.e)
    v = rng.standard_normal((len(x2), 8))
    o_ok, _, _, _ = row_forward(x2, v, True)
    o, _, _, paths = row_forward(x2, v, True, skip_first_half_rescale=True)
    assert "second half rescanned" in paths
    ro, _ = plain_softmax(x2, v)
    np.testing.assert_allclose(o_ok, ro, rtol=1e-9, atol=1e-12)
    assert np.abs(o - ro).max() > 1e-2
