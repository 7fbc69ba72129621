"""Pins for the FP8 (E4M3) weight quantisation oracle (oracle/fp8_ref.py).

What fixes it outside the oracle: the E4M3 format definition (an exhaustive
code table built from sign/exponent/mantissa fields, ties to even, the
largest finite value 448), the error bound of rounding to 3 mantissa bits,
and the scale's defining property (each row's largest magnitude maps to 448).
"""
import numpy as np
import pytest

import oracle.fp8_ref as F
from workload import get_config, make_weights
from workload.gen import bf16_bits_to_f32


def _decode(code):
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return np.nan
    return s * (2.0 ** -6 * m / 8 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8))


def test_grid_is_the_format_table():
    vals = sorted({abs(_decode(c)) for c in range(256) if not np.isnan(_decode(c))})
    assert np.array_equal(np.array(vals), F.e4m3_grid())
    assert F.e4m3_grid()[-1] == 448.0 and F.e4m3_grid()[1] == 2.0 ** -9


def test_every_code_round_trips_and_ties_go_to_even():
    g = F.e4m3_grid()
    assert np.array_equal(F.round_e4m3(g), g) and np.array_equal(F.round_e4m3(-g), -g)
    mid = (g[:-1] + g[1:]) / 2
    r = F.round_e4m3(mid)
    even = np.where(np.arange(len(mid)) % 2 == 0, g[:-1], g[1:])  # codes i, i+1: the even one
    assert np.array_equal(r, even)
    # just off the midpoints the nearest value wins
    assert np.array_equal(F.round_e4m3(mid * (1 - 1e-9)), g[:-1])
    assert np.array_equal(F.round_e4m3(mid * (1 + 1e-9)), g[1:])


def test_saturation_and_error_bound():
    assert F.round_e4m3(np.array([1e6, -500.0, 464.0]))[0] == 448.0
    assert F.round_e4m3(np.array([-500.0]))[0] == -448.0
    rng = np.random.default_rng(0)
    y = rng.uniform(2.0 ** -6, 448, 100000) * rng.choice([-1, 1], 100000)
    r = F.round_e4m3(y)
    assert np.all(np.abs(r - y) <= 2.0 ** -4 * np.abs(y) * (1 + 1e-12))  # half an ulp of 3 mantissa bits


def test_row_scales_map_the_row_maximum_to_448():
    cfg = get_config("tiny")
    w = bf16_bits_to_f32(make_weights(cfg)["layers"][0]["wqkv"]).astype(np.float64)
    q, s = F.quantize_rows(w)
    assert s.dtype == np.float32
    assert np.allclose(np.max(np.abs(q), -1), 448.0, rtol=2 ** -3)
    dq = F.dequantize_rows(w)
    assert np.all(np.abs(dq - w) <= 2.0 ** -4 * np.abs(w) + 2.0 ** -10 * s[:, None])
    rel = np.linalg.norm(dq - w) / np.linalg.norm(w)
    assert 0.005 < rel < 0.04


def test_planted_mistake_bias_or_no_ties_is_caught(monkeypatch):
    # rounding half away from zero instead of to even changes some midpoints
    g = F.e4m3_grid()

    def away(y):
        y = np.asarray(y, dtype=np.float64)
        a = np.minimum(np.abs(y), 448.0)
        i = np.clip(np.searchsorted(g, a), 1, len(g) - 1)
        r = np.where(g[i] - a <= a - g[i - 1], g[i], g[i - 1])
        return np.copysign(np.where(a == 0, 0, r), y)
    monkeypatch.setattr(F, "round_e4m3", away)
    with pytest.raises(AssertionError):
        test_every_code_round_trips_and_ties_go_to_even()


def test_fp8_model_uses_the_dequantised_weights():
    import oracle as O
    cfg = get_config("tiny")
    w = make_weights(cfg)
    m8 = O.OracleModel(cfg, w, fp8=True)
    m16 = O.OracleModel(cfg, w)
    for name in ("wqkv", "wo", "w_gate_up", "w_down"):
        assert np.array_equal(m8.w(name, 1), F.dequantize_rows(m16.w(name, 1)))
    assert np.array_equal(m8.w("in_norm", 0), m16.w("in_norm", 0))          # gains stay exact
    ids = np.array([0, 7, cfg.vocab - 1])
    assert np.array_equal(m8.embed_rows(ids), F.dequantize_rows(m16.embed_rows(ids)))
    h = np.random.default_rng(1).normal(size=(3, cfg.hidden))
    ref = O.rmsnorm(h, m8.w("final_norm"), cfg.rms_eps) @ F.dequantize_rows(O.bf16_to_f64(w["embed"])).T
    assert np.allclose(O.lm_head_logits(m8, h), ref, atol=1e-12)


def test_rounding_equals_the_library_cast_within_range():
    """Inside the finite range, rounding onto the E4M3 grid equals PyTorch's own
    float8_e4m3fn cast (an independent implementation of the same format);
    beyond 448 the library gives NaN where the reading taken here saturates."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    rng = np.random.default_rng(1)
    g = F.e4m3_grid()
    mid = ((g[:-1] + g[1:]) / 2).astype(np.float32)
    for arr in (rng.uniform(-448, 448, 100000).astype(np.float32), mid, -mid,
                rng.uniform(-2 ** -5, 2 ** -5, 20000).astype(np.float32)):
        lib = torch.from_numpy(arr).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        assert np.array_equal(F.round_e4m3(arr.astype(np.float64)), lib)
