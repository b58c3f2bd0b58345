"""Pins of the oracle's RoPE-domain keys (QEvict §4.3: quantized keys are kept in the pre-RoPE
domain with their absolute positions and RoPE is re-applied after dequantisation).

Checks:
- the rotation is the rotate-half RoPE: pairing (i, i + 64) as the complex number x_i + j x_{i+64},
  a forward rotation multiplies it by exp(j pos theta_i) (numpy complex arithmetic);
- the inverse undoes the forward rotation (to float32 rounding);
- rotated queries and keys give dot products that depend only on the relative position;
- quantisation happens in the pre-RoPE domain: keys constant across tokens before rotation form
  groups whose scales stay at rounding size although the rotated keys differ token by token, and the
  re-rotated dequantised keys reproduce the given post-RoPE keys;
- a promoted window holds the same re-rotated keys attention uses.
"""
import numpy as np

from oracle import qevict_oracle as O
from recoverable_quantized_kv_gb300 import synth


def test_rotation_is_complex_multiplication():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 128)).astype(np.float32)
    cs = synth.rope_table(64, 10000.0)[[3, 17, 29, 40, 63]]
    got = O.rope_rotate(x, cs)
    z = (x[:, :64].astype(np.float64) + 1j * x[:, 64:].astype(np.float64))
    rot = z * (cs[..., 0].astype(np.float64) + 1j * cs[..., 1].astype(np.float64))
    want = np.concatenate([rot.real, rot.imag], axis=-1)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-5)


def test_inverse_undoes_the_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 128)).astype(np.float32)
    cs = synth.rope_table(4096, 500000.0)[rng.integers(0, 4096, 9)]
    back = O.rope_rotate(O.rope_rotate(x, cs), cs, inverse=True)
    assert np.allclose(back, x, rtol=1e-5, atol=1e-6)


def test_dot_products_depend_on_relative_position():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    table = synth.rope_table(300, 10000.0).astype(np.float64)

    def dot(pq, pk):
        return float(O.rope_rotate(q, table[pq]).astype(np.float64) @ O.rope_rotate(k, table[pk]).astype(np.float64))
    for delta in (0, 5, 77):
        assert abs(dot(100, 100 - delta) - dot(200, 200 - delta)) < 1e-3 * (1 + abs(dot(100, 100 - delta)))


def test_keys_are_quantized_before_rotation():
    cfg = O.Config(h_q=4, h_kv=2, d_head=128, n_sink=2, n_recent=64, window=32, bits=2, omega=8,
                   prompt_len=200, max_len=260, budget_num=60, rope_base=10000.0)
    rng = np.random.default_rng(3)
    table = synth.rope_table(cfg.max_len, cfg.rope_base)
    pre = O.bf16_round(rng.integers(-8, 8, (cfg.h_kv, 128)).astype(np.float32) / 4)   # exact in fp16 and bf16
    lo = cfg.n_sink
    cs = table[lo:lo + cfg.window]
    post = O.bf16_round(O.rope_rotate(np.broadcast_to(pre, (cfg.window, cfg.h_kv, 128)), cs[:, None, :, :]))
    assert not np.all(post == post[0])                  # the rotated keys differ token by token
    led = O.quantize_window(post, post, cfg.bits, cs)
    flat = O.quantize_window(post, post, cfg.bits)      # the same keys quantised after rotation
    # back in the pre-RoPE domain every key channel is the same across the tokens, up to the bf16
    # rounding of the post-RoPE inputs: the group offsets are the pre-RoPE keys and the scales stay
    # at rounding size, while quantising the rotated keys needs scales of the keys' own size
    # (positions n_s .. n_s + W rotate the fast channels by up to W radians)
    assert np.max(np.abs(led.m_k.astype(np.float32) - pre)) <= 2 ** -5 * np.max(np.abs(pre))
    assert np.max(led.s_k.astype(np.float32)) <= 2 ** -6 * np.max(np.abs(pre))
    assert np.max(flat.s_k.astype(np.float32)) >= 0.25 * np.max(np.abs(pre))
    kh, _ = led.dequantize(cs)
    kf, _ = flat.dequantize()
    assert np.max(np.abs(kh - post)) <= 2 ** -5 * np.max(np.abs(post))
    assert np.max(np.abs(kf - post)) >= 8 * np.max(np.abs(kh - post))


def test_promotion_keeps_the_attended_keys():
    cfg = O.Config(h_q=4, h_kv=2, d_head=128, n_sink=2, n_recent=64, window=32, bits=2, omega=8,
                   prompt_len=400, max_len=600, budget_num=60, q_num=50, rope_base=10000.0)
    rng = np.random.default_rng(4)
    u = O.Unit(cfg)
    u.set_rope_table(synth.rope_table(cfg.max_len, cfg.rope_base))
    P = cfg.prompt_len
    k = O.bf16_round(rng.standard_normal((P, cfg.h_kv, 128)).astype(np.float32))
    u.prefill_route(k, k, rng.random(O.prompt_windows(cfg)))
    for s in range(1, 41):
        q = O.bf16_round(rng.standard_normal((cfg.h_q, 128)).astype(np.float32))
        u.decode_step(q, k[s % P], k[s % P])
        if s % cfg.omega == 0:
            u.route(rng.random(len(u.S)) * 10)
    promoted = [w for w, led in u.ledger.items() if led.status == O.DORMANT]
    assert promoted
    for w in promoted:
        Kf, _ = u.full[w]
        Kq, _ = u.ledger[w].dequantize(u.window_cs(w))
        assert np.array_equal(Kf, Kq)
