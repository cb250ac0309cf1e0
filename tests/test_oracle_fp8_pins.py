"""Pins of the oracle's opt-in E4M3 indexer (CPU only).

The E4M3 rounding is pinned to the format's definition (closed-form values:
the largest finite value, the subnormal spacing, ties to even, saturation) and
to a library conversion (torch's float8_e4m3fn cast) on every code point, on
random values and on every halfway point between neighbouring codes.  The
per-row quantiser is pinned by what its definition fixes: each row's largest
magnitude lands on +-448, codes are E4M3 values, the dequantisation error is
within half a code spacing, scaling a row by a power of two changes only its
scale, and all-zero rows stay zero.  The E4M3 scores reduce exactly to the
bf16 scores when the operands are E4M3 values with unit scales.  A planted
mistake in each piece makes one of these pins fail.
"""
import numpy as np
import pytest

from oracle import v4_oracle as O

torch = pytest.importorskip("torch")


def _e4m3_code_values():
    """Every finite E4M3 value, decoded by torch from the 256 bit patterns."""
    v = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return np.unique(v[np.isfinite(v)])


def test_e4m3_code_points_and_range():
    v = _e4m3_code_values()
    assert len(v) == 253                      # 254 finite patterns, +0 and -0 are one value
    assert v.max() == 448.0 and v.min() == -448.0
    assert np.min(np.abs(v[v != 0])) == 2.0 ** -9
    np.testing.assert_array_equal(O.round_to_e4m3(v), v)


def test_e4m3_matches_library_cast_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-460, 460, 20000), rng.normal(0, 1, 20000),
                        rng.normal(0, 2.0 ** -7, 5000)]).astype(np.float32).astype(np.float64)
    v = _e4m3_code_values()
    mids = (v[1:] + v[:-1]) / 2                 # every halfway point (exact in float32)
    mids = mids[np.abs(mids) < 448]
    for arr in (x, mids):
        ref = torch.from_numpy(arr).float().to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
        np.testing.assert_array_equal(O.round_to_e4m3(arr), ref)


def test_e4m3_saturates():
    got = O.round_to_e4m3(np.array([464.0, 470.0, 1.0e6, -500.0, -449.0]))
    np.testing.assert_array_equal(got, [448.0, 448.0, 448.0, -448.0, -448.0])


@pytest.mark.parametrize("x,want", [
    (448.0, 448.0), (464.0, 448.0), (470.0, 448.0), (1.0e6, 448.0), (-500.0, -448.0),
    (2.0 ** -9, 2.0 ** -9), (2.0 ** -10, 0.0), (3 * 2.0 ** -10, 2.0 ** -8),
    (1.0625, 1.0), (1.1875, 1.25), (1.0 + 2.0 ** -5, 1.0), (0.0, 0.0),
    (240.0, 240.0), (17.0, 16.0), (19.0, 20.0), (2.0 ** -6 + 2.0 ** -10, 2.0 ** -6),
])
def test_e4m3_closed_forms(x, want):
    assert O.round_to_e4m3(np.array([x]))[0] == want


def _rows(seed=1):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 1, (64, 128))
    x[3] *= 1e-3
    x[5, 17] = 40.0                             # one dominant value
    x[7] = 0.0                                  # all-zero row
    x[9] = np.abs(x[9])                         # positive row
    return O.round_to_bf16(x)


def test_quantizer_row_maximum_lands_on_448():
    x = _rows()
    codes, scales = O.quantize_e4m3_rows(x)
    nz = np.abs(x).max(axis=1) > 0
    np.testing.assert_array_equal(np.abs(codes[nz]).max(axis=1), 448.0)
    assert scales[7] == 0 and np.all(codes[7] == 0)
    v = _e4m3_code_values()
    assert np.all(np.isin(codes, v))
    np.testing.assert_allclose(scales[nz], np.abs(x[nz]).max(axis=1) / 448.0, rtol=2.0 ** -23)


def test_quantizer_error_within_half_spacing():
    x = _rows(2)
    codes, scales = O.quantize_e4m3_rows(x)
    err = np.abs(codes * scales[:, None] - x)
    # half a spacing: 2^-4 relative for normal codes, 2^-10 * scale for
    # subnormal ones; the float32 steps add a few units of 2^-24
    bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * scales[:, None] + 4 * 2.0 ** -24 * np.abs(x)
    assert np.all(err <= bound)


def test_quantizer_power_of_two_scaling():
    x = _rows(3)
    c1, s1 = O.quantize_e4m3_rows(x)
    c2, s2 = O.quantize_e4m3_rows(x * 2.0 ** 5)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(s2, s1 * 2.0 ** 5)


def test_e4m3_scores_exact_on_representable_operands():
    rng = np.random.default_rng(4)
    v = _e4m3_code_values()
    B, S, Hi, Di, r = 1, 24, 4, 16, 4
    N = S // r
    q = rng.choice(v, (B, S, Hi, Di))
    k = rng.choice(v, (B, N, Di))
    q[..., 0] = 448.0                          # amax exactly 448: unit scales
    k[..., 0] = 448.0
    w = rng.normal(0, 1, (B, S, Hi))
    qc, qs = O.quantize_e4m3_rows(q)
    kc, ks = O.quantize_e4m3_rows(k)
    assert np.all(qs == 1.0) and np.all(ks == 1.0)
    np.testing.assert_array_equal(qc, q)
    got = O.indexer_scores_e4m3(qc, qs, kc, ks, w, r)
    np.testing.assert_array_equal(got, O.indexer_scores(q, k, w, r))
    # and a plain loop over the definition, on a few (t, s)
    c = O.indexer_scale(Hi, Di)
    for t, s in ((23, 5), (7, 0), (15, 3)):
        ref = sum(w[0, t, h] * c * max(0.0, float(np.dot(q[0, t, h], k[0, s]))) for h in range(Hi))
        assert abs(got[0, t, s] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_e4m3_selection_close_to_bf16_on_gaussian_rows():
    # quantisation moves scores by a few percent; most of the top-k survives
    rng = np.random.default_rng(5)
    B, S, Hi, Di, r, K = 1, 256, 8, 64, 4, 16
    N = S // r
    q = O.round_to_bf16(rng.normal(0, 1, (B, S, Hi, Di)))
    k = O.round_to_bf16(rng.normal(0, 1, (B, N, Di)))
    w = rng.normal(0, 1, (B, S, Hi))
    ref = O.indexer_topk(q, k, w, None, r, K, prepared=True)["idx"]
    qc, qs = O.quantize_e4m3_rows(q)
    kc, ks = O.quantize_e4m3_rows(k)
    got = O.indexer_topk_e4m3(qc, qs, kc, ks, w, r, K)["idx"]
    kept = [len(set(a[a >= 0]) & set(b[b >= 0])) / max(1, (a >= 0).sum()) for a, b in zip(ref[0], got[0])]
    assert np.mean(kept) > 0.85
