"""The CPU oracle against its pins (no GPU)."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def lib():
    return oracle.default_lib()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    pin(lib)


def test_error_metrics_definition():
    import numpy as np
    ref = np.array([1.0, -2.0, 0.0, 4.0])
    y = np.array([1.5, -2.0, 0.25, 3.0])
    mx, mean = oracle.error_metrics(y, ref)
    assert mx == pytest.approx(1.0 / 4.0)
    assert mean == pytest.approx(1.75 / 7.0)


def test_heads_subset_matches_full(lib):
    import numpy as np
    rng = np.random.default_rng(3)
    x, dt, A, B, C, D, h0 = oracle_pins._rand_inputs(rng, b=2, L=9, H=4, G=2)
    y, hT = oracle.scan(x, dt, A, B, C, D, h0, lib=lib)
    heads = [(1, 3), (0, 0), (1, 1)]
    ys, hs = oracle.scan(x, dt, A, B, C, D, h0, heads=heads, lib=lib)
    for i, (b, h) in enumerate(heads):
        assert np.array_equal(ys[i], y[b, :, h, :])
        assert np.array_equal(hs[i], hT[b, h])


def test_chunked_stages_consistent():
    """The chunked oracle's staged intermediates recombine into its own outputs."""
    import numpy as np
    rng = np.random.default_rng(4)
    x, dt, A, B, C, D, h0 = oracle_pins._rand_inputs(rng, b=1, L=20, H=2, G=1)
    y, hT, st = oracle.chunked(x, dt, A, B, C, D, h0, chunk_size=8, keep_stages=True)
    for (b, h, c), s in st.items():
        lo, hi = c * 8, min(20, c * 8 + 8)
        yc = (s["Ydiag"] + s["Yoff"])[: hi - lo] + D[h] * x[b, lo:hi, h, :]
        assert np.allclose(yc, y[b, lo:hi, h, :], rtol=1e-12, atol=1e-12)
