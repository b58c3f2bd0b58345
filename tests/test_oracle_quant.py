"""Pins of the oracle's number formats and quantiser (QEvict §4.3 "Migration-Stable Quantization").

Each check compares the oracle with something other than itself: torch's own
format conversions, an exhaustive search over the code lattice, hand-built
groups whose correct codes are known, and the quantisation error bound.
"""
import numpy as np
import pytest
import torch

from oracle import qevict_oracle as O


def _special_f32(rng, n):
    x = rng.standard_normal(n).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, n).astype(np.float32)
    ties = (rng.integers(0, 1 << 16, n).astype(np.uint32) << 16) | np.uint32(0x8000)   # exact bf16 ties
    return np.concatenate([x, ties.view(np.float32), np.array([0.0, -0.0, 1e-40, -3e-39, 3.0e38, -3.3e38,
                                                              np.inf, -np.inf], np.float32)])


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(0)
    x = _special_f32(rng, 20000)
    x = x[np.isfinite(x) | np.isinf(x)]
    ours = O.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


def test_fp16_round_matches_torch():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000).astype(np.float32)
    ours = O.fp16_round(x)
    ref = torch.from_numpy(x).to(torch.float16).numpy()
    assert np.array_equal(ours.view(np.uint16), ref.view(np.uint16))


def _bf16_values(rng, shape, scale=1.0):
    return O.bf16_round((rng.standard_normal(shape) * scale).astype(np.float32))


@pytest.mark.parametrize("bits", [2, 4])
def test_codes_minimise_error_exhaustively(bits):
    """code = argmin_c |x - (c*s + m)| over the whole lattice (up to float32 rounding of the quotient)."""
    rng = np.random.default_rng(bits)
    x = _bf16_values(rng, (400, 32), scale=3.0)              # 400 groups of 32 along axis 1
    code, s16, m16 = O.quantize_groups(x, axis=1, bits=bits)
    s = s16.astype(np.float64)[:, None]
    m = m16.astype(np.float64)[:, None]
    lattice = np.arange(1 << bits, dtype=np.float64)
    err_all = np.abs(x.astype(np.float64)[..., None] - (lattice * s[..., None] + m[..., None]))
    best = err_all.min(axis=-1)
    chosen = np.take_along_axis(err_all, code.astype(np.int64)[..., None], axis=-1)[..., 0]
    assert code.max() <= (1 << bits) - 1
    assert np.all(chosen <= best + 1e-6 * s + 1e-30)
    # the scale covers the group's range in (2^bits - 1) steps, up to fp16 rounding
    rng_ = x.max(axis=1) - x.min(axis=1)
    assert np.allclose(s16.astype(np.float64), rng_ / ((1 << bits) - 1), rtol=2 ** -10, atol=1e-7)
    assert np.array_equal(m16, x.min(axis=1).astype(np.float16))


def test_hand_cases_lattice_constant_ties():
    # exact lattice {m, m+s, m+2s, m+3s} -> codes 0..3
    lat = np.array([[1.0, 1.5, 2.0, 2.5, 2.5, 1.0]], np.float32)
    c, s, m = O.quantize_groups(lat, axis=1, bits=2)
    assert s[0] == np.float16(0.5) and m[0] == np.float16(1.0)
    assert c.tolist() == [[0, 1, 2, 3, 3, 0]]
    # constant group -> s = 0, codes 0, reconstruction = m
    const = np.full((1, 8), 0.75, np.float32)
    c, s, m = O.quantize_groups(const, axis=1, bits=2)
    assert s[0] == 0 and np.all(c == 0)
    assert np.all(O.dequantize_groups(c, s, m, axis=1) == np.float32(0.75))
    # ties at 0.5 s, 1.5 s, 2.5 s round half to even -> 0, 2, 2  (m = 0, s = 1)
    ties = np.array([[0.0, 3.0, 0.5, 1.5, 2.5]], np.float32)
    c, s, m = O.quantize_groups(ties, axis=1, bits=2)
    assert s[0] == 1 and m[0] == 0
    assert c[0, 2:].tolist() == [0, 2, 2]


def test_key_and_value_groups_run_along_the_right_axes():
    """Keys: one group per (head, channel) across tokens.  Values: one group per (head, token) across channels."""
    W, H, d = 32, 2, 128
    K = np.broadcast_to(np.arange(d, dtype=np.float32)[None, None, :], (W, H, d)).copy()   # constant per channel
    V = np.broadcast_to(np.arange(W, dtype=np.float32)[:, None, None], (W, H, d)).copy()   # constant per token
    led = O.quantize_window(K, V, bits=2)
    assert led.s_k.shape == (H, d) and led.s_v.shape == (H, W)
    assert np.all(led.s_k == 0) and np.all(led.s_v == 0)
    Kh, Vh = led.dequantize()
    assert np.array_equal(Kh, K) and np.array_equal(Vh, V)


@pytest.mark.parametrize("bits", [2, 4])
def test_reconstruction_error_bound(bits):
    """|x - x_hat| <= s/2 (nearest lattice point) + fp16/bf16 rounding of the parameters and result."""
    rng = np.random.default_rng(10 + bits)
    K = _bf16_values(rng, (32, 2, 128))
    V = _bf16_values(rng, (32, 2, 128))
    led = O.quantize_window(K, V, bits)
    Kh, Vh = led.dequantize()
    sk = led.s_k.astype(np.float32).transpose(0, 1)[None]           # [1][H][d]
    sv = led.s_v.astype(np.float32).transpose(1, 0)[:, :, None]     # [W][H][1]
    eps = 2 ** -8
    assert np.all(np.abs(K - Kh) <= 0.5 * sk * (1 + 2 ** -9) + eps * np.abs(K) + 2 ** -10 * np.abs(sk) + 1e-6)
    assert np.all(np.abs(V - Vh) <= 0.5 * sv * (1 + 2 ** -9) + eps * np.abs(V) + 2 ** -10 * np.abs(sv) + 1e-6)


def test_dequantize_is_bf16_of_one_rounded_sum():
    """x_hat is a bf16 value and equals bf16(float32(c*s+m)) evaluated with torch's fused multiply-add."""
    rng = np.random.default_rng(7)
    x = _bf16_values(rng, (64, 32), 2.0)
    c, s, m = O.quantize_groups(x, axis=1, bits=2)
    ours = O.dequantize_groups(c, s, m, axis=1)
    ref = torch.addcmul(torch.from_numpy(m.astype(np.float32))[:, None], torch.from_numpy(c.astype(np.float32)),
                        torch.from_numpy(s.astype(np.float32))[:, None]).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours, ref)


def _golden_groups():
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "quant_groups.txt")
    out = []
    for ln in open(path):
        if ln.strip() and not ln.startswith("#"):
            f = [p.split() for p in ln.split("|")]
            out.append((int(f[0][0]), [float(v) for v in f[1]], float(f[2][0]), float(f[3][0]),
                        [int(v) for v in f[4]], [float(v) for v in f[5]]))
    return out


@pytest.mark.parametrize("bits,x,s,m,codes,xhat", _golden_groups())
def test_groups_worked_by_hand(bits, x, s, m, codes, xhat):
    """Groups whose parameters, codes and reconstructions were worked by hand
    (tests/golden/quant_groups.txt, QEvict §4.3 "Migration-Stable Quantization")."""
    xa = np.array([x], np.float32)
    assert np.array_equal(O.bf16_round(xa), xa)
    c, s16, m16 = O.quantize_groups(xa, axis=1, bits=bits)
    assert float(s16[0]) == s and float(m16[0]) == m
    assert c[0].tolist() == codes
    assert O.dequantize_groups(c, s16, m16, axis=1)[0].tolist() == xhat
