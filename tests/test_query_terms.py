"""The bounds stated for the fp8 kernel's query operand, checked on the CPU.

A bf16 query row is scaled by 2^a so that its largest |x| lies in [128, 256),
and split into e4m3 terms T1 + T2/16 + T3/256 + ..., each term the e4m3
rounding (to nearest, ties to even) of the previous residual times 16; the
kernel uses 4 terms with up to 8 query rows per KV head and 2 with 16. The
stated bounds: with 2 terms every scaled element of magnitude >= 2^-6 (down
to 2^-14 of the row maximum) is exact and the others are within 2^-14; with
4 terms the same holds from 2^-14 on, the others within 2^-22. The split is
restated here with torch's e4m3 conversion, independently of the CUDA path;
the residuals are exact in float64 as they are in the kernel's float32."""
import numpy as np
import pytest
import torch

import synth


def _e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _terms_sum(x: np.ndarray, terms: int) -> np.ndarray:
    """Sum of the e4m3 terms of x (each the rounding of the residual x 16)."""
    total = np.zeros_like(x)
    r = x.copy()
    w = 1.0
    for _ in range(terms):
        t = _e4m3(r)
        total += t * w
        r = (r - t) * 16.0
        w /= 16.0
    return total


def _scaled_rows(seed: int, rows: int = 512, dims: int = 128) -> np.ndarray:
    """bf16 rows with an outlier and elements log-uniform over 2^-30 .. 1 of
    it, scaled as the kernel scales them (max |x| in [128, 256))."""
    r = np.random.default_rng(seed)
    q = np.where(r.random((rows, dims)) < 0.5, -1.0, 1.0) * 2.0 ** r.uniform(-30.0, 0.0, (rows, dims))
    q[:, 0] *= 2.0 ** r.uniform(0.0, 8.0, rows)
    bits = synth.round_to_bf16_bits(q.astype(np.float32))
    qb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    amax = np.abs(qb).max(axis=1, keepdims=True)
    _, ex = np.frexp(amax)
    a = np.clip(8 - ex, -126, 126)
    x = qb * np.exp2(a)
    assert np.all((np.abs(x).max(axis=1) >= 128) & (np.abs(x).max(axis=1) < 256))
    return x


@pytest.mark.parametrize("terms,exact_from,err_below", [(2, 2.0 ** -6, 2.0 ** -14), (4, 2.0 ** -14, 2.0 ** -22)])
def test_query_terms_bounds(terms, exact_from, err_below):
    x = _scaled_rows(11 + terms)
    err = np.abs(_terms_sum(x, terms) - x)
    big = np.abs(x) >= exact_from
    assert big.any() and (~big).any()
    assert np.all(err[big] == 0.0), "an element above the bound is not exact"
    assert err[~big].max() <= err_below, f"error below the bound {err[~big].max():.3g} > {err_below:.3g}"


def test_two_terms_are_not_exact_for_all_elements():
    """The bound is tight in the sense that it matters: 2 terms do lose small
    elements that 4 terms keep (so the 16-row kernel's query is not claimed
    exact everywhere)."""
    x = _scaled_rows(7)
    e2 = np.abs(_terms_sum(x, 2) - x)
    e4 = np.abs(_terms_sum(x, 4) - x)
    assert e2.max() > 0.0
    assert e4.max() < e2.max()
