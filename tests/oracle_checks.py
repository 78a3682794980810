"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on oracle builds with one planted mistake
each and requires that some check fails.

What pins what (sources: vllm_omni/edge/spark_export.py for the Spark decode
step, vllm/models/hy_v4/nvidia/flashmla_sparse.py for the sink):
  bf16 rounding      hand-built ties, torch's float->bf16 cast on binary32 inputs,
                     the half-quantum bound
  rotary table       position 0, closed-form entries (frequency 1 and theta^-1/2),
                     the angle addition identity, geometric frequency spacing
  rotation           identity at 0, pass-through, unit vectors, complex product,
                     relative-position property
  attention          scipy softmax/logsumexp, one-key closed form, equal keys,
                     weight sum = sigmoid(lse - sink), -inf sink, permutation
  layer / GQA        expanded-head MHA brute force with scipy
  windows / layouts  sliding == full inside the window, ring == roll, and a
                     token-by-token history model (a plain list of every past
                     token) that the cache bookkeeping must reproduce
  footprint          the page's 4k-context KV figures (tests/golden)
  output gate        scipy expit per head; exact values at +inf, 0 and -inf
  fp8 e4m3 (R14)     all 256 codes against torch's float8_e4m3fn cast, round trip,
                     brute-force nearest-even on random and midpoint doubles,
                     saturation; FP8 layers against a scipy brute force on the
                     dequantised cache, against the bf16 layer on values both
                     formats hold exactly, and against the history model
  multi-token (R15)  T tokens per step against a brute force over positions:
                     token t's key set is every position of its window up to
                     c+t, and the caches end holding the extended history
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.special as sps
import torch

SLIDING, FULL = 0, 1
RING, ROLL = 1, 2
NAN_BITS = np.uint16(0x7FC0)
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16_bits_random(rng, shape, std=1.0):
    x = (rng.standard_normal(size=shape) * std).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _bits_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _f32_ulp(x):
    return np.spacing(np.abs(np.float32(x)).astype(np.float32)).astype(np.float64)


# --------------------------------------------------------------------- bf16 --

def check_bf16_hand_ties(orc):
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (1.0)
        (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (1 + 2^-6)
        (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),    # just above the tie: up (no double rounding)
        (-(1.0 + 2.0 ** -8 + 2.0 ** -40), 0xBF81),
        (1.0 + 2.0 ** -8 - 2.0 ** -40, 0x3F80),    # just below the tie: down
        (2.0 ** -133, 0x0001),                     # smallest subnormal
        (2.0 ** -134, 0x0000),                     # tie between 0 and 2^-133 -> even (0)
        (1.5 * 2.0 ** -134, 0x0001),
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie above the largest finite -> inf
        (float("inf"), 0x7F80),
        (float("-inf"), 0xFF80),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (3.140625, 0x4049),
    ]
    for x, want in cases:
        got = int(orc.lib.orc_f64_to_bf16(x))
        assert got == want, f"bf16({x!r}) = {got:#06x}, want {want:#06x}"
    assert (int(orc.lib.orc_f64_to_bf16(float("nan"))) & 0x7FFF) > 0x7F80


def check_bf16_matches_torch_on_binary32(orc):
    rng = np.random.default_rng(1)
    mant = rng.standard_normal(4000)
    expo = rng.integers(-140, 126, size=4000)
    x = (mant * np.exp2(expo.astype(np.float64))).astype(np.float32)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.lib.orc_f64_to_bf16(float(v)) for v in x], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} mismatches vs torch, first x={x[bad[0]]!r}"


def check_bf16_nearest_on_doubles(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(3000) * np.exp2(rng.integers(-20, 20, size=3000).astype(np.float64))
    for v in x:
        b = int(orc.lib.orc_f64_to_bf16(float(v)))
        r = orc.lib.orc_bf16_to_f64(b)
        lo = orc.lib.orc_bf16_to_f64((b - 1) & 0xFFFF) if (b & 0x7FFF) else r
        hi = orc.lib.orc_bf16_to_f64((b + 1) & 0xFFFF)
        err = abs(v - r)
        assert err <= abs(v - lo) and err <= abs(v - hi), f"bf16({v!r}) is not the nearest"


def check_bf16_to_f64_matches_torch(orc):
    bits = np.arange(0, 0x10000, 7, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    want = _bits_to_f64(bits)
    got = np.array([orc.lib.orc_bf16_to_f64(int(b)) for b in bits])
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ rotary --

def check_angles_position_zero(orc):
    for rot, theta in ((256, 1e4), (64, 5e6), (8, 1e4)):
        c, s = orc.rope_angles(0, rot, theta)
        assert np.all(c == 1.0) and np.all(s == 0.0)


def check_angles_closed_form_entries(orc):
    # Entry 0 has frequency 1; entry rot/4 has frequency theta^(-1/2); the last
    # entry has frequency theta^(-(rot-2)/rot).
    for rot, theta in ((256, 1e4), (64, 5e6)):
        for p in (1, 7, 4096, 131072):
            c, s = orc.rope_angles(p, rot, theta)
            for i, w in ((0, 1.0), (rot // 4, 1.0 / math.sqrt(theta)),
                         (rot // 2 - 1, theta ** (-(rot - 2) / rot))):
                a = p * w
                assert abs(c[i] - math.cos(a)) <= _f32_ulp(math.cos(a)) + 1e-12 * p, (rot, p, i)
                assert abs(s[i] - math.sin(a)) <= _f32_ulp(math.sin(a)) + 1e-12 * p, (rot, p, i)


def check_angles_addition_identity(orc):
    for rot, theta in ((256, 1e4), (64, 5e6)):
        for p, q in ((3, 5), (100, 411), (2000, 2096)):
            cp, sp = orc.rope_angles(p, rot, theta)
            cq, sq = orc.rope_angles(q, rot, theta)
            cpq, spq = orc.rope_angles(p + q, rot, theta)
            cp, sp, cq, sq = (a.astype(np.float64) for a in (cp, sp, cq, sq))
            assert np.allclose(cpq, cp * cq - sp * sq, atol=4e-7, rtol=0)
            assert np.allclose(spq, sp * cq + cp * sq, atol=4e-7, rtol=0)


def check_angles_frequency_spacing(orc):
    # At position 1 the angle is the frequency itself; consecutive frequencies
    # fall by theta^(-2/rot).
    for rot, theta in ((256, 1e4), (64, 5e6)):
        c, s = orc.rope_angles(1, rot, theta)
        w = np.arctan2(s.astype(np.float64), c.astype(np.float64))
        ratio = w[1:] / w[:-1]
        assert np.allclose(ratio, theta ** (-2.0 / rot), rtol=2e-6), (rot, ratio[:3])


def check_rope_identity_and_passthrough(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(256)
    c, s = orc.rope_angles(0, 64, 5e6)
    assert np.array_equal(orc.rope(x, 64, c, s), x)
    c, s = orc.rope_angles(12345, 64, 5e6)
    y = orc.rope(x, 64, c, s)
    assert np.array_equal(y[64:], x[64:])
    assert not np.array_equal(y[:64], x[:64])


def check_rope_unit_vectors(orc):
    for rot, theta, D in ((256, 1e4, 256), (64, 5e6, 256)):
        half = rot // 2
        c, s = orc.rope_angles(777, rot, theta)
        for i in (0, 1, half - 1):
            e = np.zeros(D)
            e[i] = 1.0
            y = orc.rope(e, rot, c, s)
            want = np.zeros(D)
            want[i], want[i + half] = c[i], s[i]
            assert np.array_equal(y, want), (rot, i)
            e = np.zeros(D)
            e[i + half] = 1.0
            y = orc.rope(e, rot, c, s)
            want = np.zeros(D)
            want[i], want[i + half] = -s[i], c[i]
            assert np.array_equal(y, want), (rot, i, "second half")


def check_rope_is_complex_product(orc):
    rng = np.random.default_rng(4)
    for rot, theta in ((256, 1e4), (64, 5e6)):
        half = rot // 2
        x = rng.standard_normal(256)
        c, s = orc.rope_angles(4096, rot, theta)
        y = orc.rope(x, rot, c, s)
        z = (x[:half] + 1j * x[half:rot]) * (c.astype(np.float64) + 1j * s.astype(np.float64))
        tol = 1e-15 * np.max(np.abs(x))
        assert np.allclose(y[:half], z.real, rtol=0, atol=tol)
        assert np.allclose(y[half:rot], z.imag, rtol=0, atol=tol)


def check_rope_relative_position(orc):
    rng = np.random.default_rng(5)
    for rot, theta in ((256, 1e4), (64, 5e6)):
        q, k = rng.standard_normal(256), rng.standard_normal(256)
        for m, n in ((10, 3), (700, 189), (5000, 4999)):
            cm, sm = orc.rope_angles(m, rot, theta)
            cn, sn = orc.rope_angles(n, rot, theta)
            cd, sd = orc.rope_angles(m - n, rot, theta)
            lhs = orc.rope(q, rot, cm, sm) @ orc.rope(k, rot, cn, sn)
            rhs = orc.rope(q, rot, cd, sd) @ k
            assert abs(lhs - rhs) <= 2e-5 * np.linalg.norm(q) * np.linalg.norm(k), (rot, m, n)


# --------------------------------------------------------------- attention --

def check_attend_vs_scipy(orc):
    rng = np.random.default_rng(6)
    for D in (4, 8, 16):
        for n in (1, 2, 5, 20):
            q = rng.standard_normal(D) * 3
            K = rng.standard_normal((n, D))
            V = rng.standard_normal((n, D))
            for sink in (None, 0.3, -2.0):
                out, lse = orc.attend(q, K, V, sink)
                sc = K @ q / math.sqrt(D)
                want = sps.softmax(sc) @ V
                want_lse = sps.logsumexp(sc)
                if sink is not None:
                    want = want * sps.expit(want_lse - sink)
                assert np.allclose(out, want, rtol=1e-12, atol=1e-12), (D, n, sink)
                assert abs(lse - want_lse) < 1e-12, (D, n)


def check_attend_one_key(orc):
    rng = np.random.default_rng(7)
    q, k, v = rng.standard_normal((3, 256))
    s = float(q @ k) / 16.0
    for sink in (None, 0.0, 1.5, -3.0):
        out, lse = orc.attend(q, k[None], v[None], sink)
        f = 1.0 if sink is None else 1.0 / (1.0 + math.exp(sink - s))
        assert abs(lse - s) < 1e-13
        assert np.allclose(out, v * f, rtol=1e-14, atol=1e-15)


def check_attend_equal_keys_mean(orc):
    rng = np.random.default_rng(8)
    q, k = rng.standard_normal((2, 64))
    V = rng.standard_normal((9, 64))
    out, lse = orc.attend(q, np.tile(k, (9, 1)), V)
    assert np.allclose(out, V.mean(0), rtol=1e-13, atol=1e-14)
    assert abs(lse - (float(q @ k) / 8.0 + math.log(9))) < 1e-12


def check_attend_weight_sum(orc):
    rng = np.random.default_rng(9)
    n = D = 12
    q = rng.standard_normal(D) * 2
    K = rng.standard_normal((n, D))
    V = np.eye(n)  # out then equals the attention weights
    for sink in (-1.0, 0.0, 2.5):
        out, lse = orc.attend(q, K, V, sink)
        assert np.all(out >= 0)
        assert abs(out.sum() - math.exp(lse) / (math.exp(lse) + math.exp(sink))) < 1e-13


def check_attend_neg_inf_sink(orc):
    rng = np.random.default_rng(10)
    q, K, V = rng.standard_normal(32), rng.standard_normal((7, 32)), rng.standard_normal((7, 32))
    a, la = orc.attend(q, K, V, None)
    b, lb = orc.attend(q, K, V, float("-inf"))
    assert np.array_equal(a, b) and la == lb


def check_attend_permutation(orc):
    rng = np.random.default_rng(11)
    q, K, V = rng.standard_normal(32), rng.standard_normal((30, 32)), rng.standard_normal((30, 32))
    a, la = orc.attend(q, K, V, 0.5)
    p = rng.permutation(30)
    b, lb = orc.attend(q, K[p], V[p], 0.5)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14) and abs(la - lb) < 1e-13


# ------------------------------------------------------------ decode layer --

def _rope_complex(x, rot, c, s):
    half = rot // 2
    z = (x[..., :half] + 1j * x[..., half:rot]) * (c.astype(np.float64) + 1j * s.astype(np.float64))
    return np.concatenate([z.real, z.imag, x[..., rot:]], axis=-1)


def _layer(orc, **kw):
    return orc.decode_layer(**kw)


def check_layer_gqa_vs_expanded_mha(orc):
    """Full layer vs an MHA brute force with K/V expanded per query head."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, D, rot, theta = 2, 8, 2, 16, 8, 5e6
    g = Hq // Hkv
    ctx = np.array([5, 9], np.int32)
    cap = 12
    kc = _bf16_bits_random(rng, (B, Hkv, cap, D))
    vc = _bf16_bits_random(rng, (B, Hkv, cap, D))
    for b in range(B):
        kc[b, :, ctx[b]:] = NAN_BITS
        vc[b, :, ctx[b]:] = NAN_BITS
    q = _bf16_bits_random(rng, (B, Hq, D))
    k = _bf16_bits_random(rng, (B, Hkv, D))
    v = _bf16_bits_random(rng, (B, Hkv, D))
    sink = rng.standard_normal(Hq).astype(np.float32)
    kc0, vc0 = kc.copy(), vc.copy()
    r = _layer(orc, layer_type=FULL, layout=0, window=512, rotary_dim=rot, rope_theta=theta,
               context=ctx, q=q, k=k, v=v, kcache=kc, vcache=vc, sink=sink)
    for b in range(B):
        c_, s_ = orc.rope_angles(int(ctx[b]), rot, theta)
        qr = _rope_complex(_bits_to_f64(q[b]), rot, c_, s_)            # [Hq, D]
        kr = _rope_complex(_bits_to_f64(k[b]), rot, c_, s_)            # [Hkv, D]
        kw = np.array([[orc.lib.orc_f64_to_bf16(float(t)) for t in row] for row in kr], np.uint16)
        assert np.array_equal(r["k_written"][b], kw), "written key"
        assert np.allclose(r["qrot"][b], qr, rtol=0, atol=0)
        n = int(ctx[b])
        keys = np.concatenate([_bits_to_f64(kc0[b, :, :n]), _bits_to_f64(kw)[:, None]], axis=1)
        vals = np.concatenate([_bits_to_f64(vc0[b, :, :n]), _bits_to_f64(v[b])[:, None]], axis=1)
        keys_e = np.repeat(keys, g, axis=0)   # [Hq, n+1, D]: head h reads kv head h // g
        vals_e = np.repeat(vals, g, axis=0)
        sc = np.einsum("hd,hnd->hn", qr, keys_e) / math.sqrt(D)
        w = sps.softmax(sc, axis=-1)
        lse = sps.logsumexp(sc, axis=-1)
        out = np.einsum("hn,hnd->hd", w, vals_e) * sps.expit(lse - sink)[:, None]
        assert np.allclose(r["out"][b], out, rtol=1e-12, atol=1e-12)
        assert np.allclose(r["lse"][b], lse, rtol=0, atol=1e-12)
        # append: the new entry lands at index c, nothing else changes
        assert np.array_equal(kc[b, :, n], kw) and np.array_equal(vc[b, :, n], v[b])
        assert np.array_equal(kc[b, :, :n], kc0[b, :, :n])


def check_sliding_equals_full_inside_window(orc):
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D, rot, theta = 1, 4, 2, 32, 16, 5e6
    for c in (0, 1, 100, 510):
        ring_k = _bf16_bits_random(rng, (B, Hkv, 511, D))
        ring_v = _bf16_bits_random(rng, (B, Hkv, 511, D))
        ring_k[:, :, c:] = NAN_BITS
        ring_v[:, :, c:] = NAN_BITS
        full_k = np.full((B, Hkv, 600, D), NAN_BITS, np.uint16)
        full_v = full_k.copy()
        full_k[:, :, :511] = ring_k
        full_v[:, :, :511] = ring_v
        q = _bf16_bits_random(rng, (B, Hq, D))
        k = _bf16_bits_random(rng, (B, Hkv, D))
        v = _bf16_bits_random(rng, (B, Hkv, D))
        args = dict(window=512, rotary_dim=rot, rope_theta=theta, context=np.array([c], np.int32),
                    q=q, k=k, v=v, sink=None)
        a = _layer(orc, layer_type=SLIDING, layout=RING, kcache=ring_k, vcache=ring_v, **args)
        b = _layer(orc, layer_type=FULL, layout=0, kcache=full_k, vcache=full_v, **args)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"]), c


def _history_caches(rng, n_pos, Hkv, D):
    hk = _bf16_bits_random(rng, (n_pos, Hkv, D))
    hv = _bf16_bits_random(rng, (n_pos, Hkv, D))
    return hk, hv


def check_ring_equals_roll(orc):
    rng = np.random.default_rng(14)
    Hq, Hkv, D, W = 4, 2, 32, 512
    for c in (1, 300, 511, 512, 513, 700, 1100):
        hk, hv = _history_caches(rng, c, Hkv, D)
        ring_k = np.full((1, Hkv, W - 1, D), NAN_BITS, np.uint16)
        ring_v = ring_k.copy()
        for p in range(max(0, c - (W - 1)), c):
            ring_k[0, :, p % (W - 1)] = hk[p]
            ring_v[0, :, p % (W - 1)] = hv[p]
        roll_k = np.full((1, Hkv, W, D), NAN_BITS, np.uint16)
        roll_v = roll_k.copy()
        lo = max(0, c - W)
        for i, p in enumerate(range(lo, c)):
            roll_k[0, :, i] = hk[p]
            roll_v[0, :, i] = hv[p]
        q = _bf16_bits_random(rng, (1, Hq, D))
        k = _bf16_bits_random(rng, (1, Hkv, D))
        v = _bf16_bits_random(rng, (1, Hkv, D))
        sink = rng.standard_normal(Hq).astype(np.float32)
        args = dict(layer_type=SLIDING, window=W, rotary_dim=32, rope_theta=1e4,
                    context=np.array([c], np.int32), q=q, k=k, v=v, sink=sink)
        a = _layer(orc, layout=RING, kcache=ring_k, vcache=ring_v, **args)
        b = _layer(orc, layout=ROLL, kcache=roll_k, vcache=roll_v, **args)
        assert np.allclose(a["out"], b["out"], rtol=1e-12, atol=1e-13), c
        assert np.allclose(a["lse"], b["lse"], rtol=0, atol=1e-12), c


def check_history_model(orc):
    """Run many steps from an empty cache; every step must equal brute force over
    the window of a plain list of all past tokens."""
    rng = np.random.default_rng(15)
    Hq, Hkv, D, rot = 4, 2, 16, 8
    g = Hq // Hkv
    for layer_type, layout, window, steps in ((SLIDING, RING, 8, 30), (SLIDING, ROLL, 8, 30),
                                              (FULL, 0, 8, 20), (SLIDING, RING, 512, 515)):
        if layer_type == SLIDING:
            cap = window - 1 if layout == RING else window
        else:
            cap = steps + 1
        kc = np.full((1, Hkv, cap, D), NAN_BITS, np.uint16)
        vc = kc.copy()
        past_k, past_v = [], []
        for c in range(steps):
            q = _bf16_bits_random(rng, (1, Hq, D))
            k = _bf16_bits_random(rng, (1, Hkv, D))
            v = _bf16_bits_random(rng, (1, Hkv, D))
            sink = rng.standard_normal(Hq).astype(np.float32)
            r = _layer(orc, layer_type=layer_type, layout=layout, window=window, rotary_dim=rot,
                       rope_theta=1e4, context=np.array([c], np.int32), q=q, k=k, v=v,
                       kcache=kc, vcache=vc, sink=sink)
            past_k.append(r["k_written"][0])
            past_v.append(v[0])
            lo = max(0, c - window + 1) if layer_type == SLIDING else 0
            keys = _bits_to_f64(np.stack(past_k[lo:c + 1], axis=1))   # [Hkv, n, D]
            vals = _bits_to_f64(np.stack(past_v[lo:c + 1], axis=1))
            for h in range(Hq):
                sc = keys[h // g] @ r["qrot"][0, h] / math.sqrt(D)
                lse = sps.logsumexp(sc)
                out = sps.softmax(sc) @ vals[h // g] * sps.expit(lse - sink[h])
                assert np.allclose(r["out"][0, h], out, rtol=1e-12, atol=1e-12), (layer_type, layout, c, h)
                assert abs(r["lse"][0, h] - lse) < 1e-12, (layer_type, layout, c, h)


def check_output_gate(orc):
    """The output gate scales each head by sigmoid(logit) (scipy expit), leaves
    lse alone, is exactly a no-op at +inf, halves at 0 and zeroes at -inf."""
    rng = np.random.default_rng(16)
    B, Hq, Hkv, D = 2, 4, 2, 16
    ctx = np.array([5, 0], np.int32)
    base = dict(layer_type=FULL, layout=0, window=512, rotary_dim=8, rope_theta=1e4, context=ctx)
    kc = _bf16_bits_random(rng, (B, Hkv, 8, D))
    vc = _bf16_bits_random(rng, (B, Hkv, 8, D))
    q = _bf16_bits_random(rng, (B, Hq, D))
    k = _bf16_bits_random(rng, (B, Hkv, D))
    v = _bf16_bits_random(rng, (B, Hkv, D))
    sink = rng.standard_normal(Hq).astype(np.float32)
    plain = _layer(orc, kcache=kc.copy(), vcache=vc.copy(), q=q, k=k, v=v, sink=sink, **base)
    logits = rng.standard_normal((B, Hq)).astype(np.float32) * 3
    gated = orc.decode_layer(kcache=kc.copy(), vcache=vc.copy(), q=q, k=k, v=v, sink=sink, gate=logits, **base)
    want = plain["out"] * sps.expit(logits.astype(np.float64))[:, :, None]
    assert np.allclose(gated["out"], want, rtol=1e-14, atol=1e-15)
    assert np.array_equal(gated["lse"], plain["lse"])
    special = np.array([[np.inf, 0.0, -np.inf, np.inf]] * B, np.float32)
    g2 = orc.decode_layer(kcache=kc.copy(), vcache=vc.copy(), q=q, k=k, v=v, sink=sink, gate=special, **base)
    assert np.array_equal(g2["out"][:, 0], plain["out"][:, 0])
    assert np.array_equal(g2["out"][:, 1], plain["out"][:, 1] * 0.5)
    assert np.all(g2["out"][:, 2] == 0.0)


# --------------------------------------------------------------- fp8 e4m3 --

NAN_CODE = np.uint8(0x7F)


def _e4m3_table():
    """All 256 codes decoded by torch's float8_e4m3fn -> float32 cast."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().double().numpy()


def _e4m3_nearest(x, table):
    """Brute force: the code of x's sign whose value is nearest to x, ties to the
    code with an even mantissa; beyond the largest finite value, that value."""
    if np.isnan(x):
        return 0x7F
    sign = 0x80 if np.signbit(x) else 0
    if abs(x) > 448.0:
        return sign | 0x7E
    codes = [c for c in range(sign, sign + 128) if not np.isnan(table[c])]
    dist = [abs(x - table[c]) for c in codes]
    best = min(dist)
    ties = [c for c, d_ in zip(codes, dist) if d_ == best]
    if len(ties) > 1:
        ties = [c for c in ties if c % 2 == 0]
    assert len(ties) == 1, (x, ties)
    return ties[0]


def _random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C  # no NaN codes among written entries
    return c


def check_e4m3_decode_matches_torch(orc):
    want = _e4m3_table()
    got = orc.e4m3_to_f64(np.arange(256))
    nan = np.isnan(want)
    assert nan.sum() == 2 and want[0x7E] == 448.0 and want[0x01] == 2.0 ** -9
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def check_e4m3_round_trip(orc):
    table = _e4m3_table()
    finite = np.array([c for c in range(256) if not np.isnan(table[c])], np.uint8)
    assert np.array_equal(orc.f64_to_e4m3(orc.e4m3_to_f64(finite)), finite)


def check_e4m3_nearest_even_brute_force(orc):
    table = _e4m3_table()
    rng = np.random.default_rng(17)
    mags = np.exp2(rng.uniform(-12.0, 9.2, size=1500))
    xs = list(mags * np.where(rng.random(1500) < 0.5, -1.0, 1.0))
    pos = np.sort(np.unique(table[:0x7F]))                 # +0 .. 448
    mids = (pos[:-1] + pos[1:]) / 2                        # exact ties in fp64
    xs += list(mids) + list(-mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, 1e9))
    xs += [0.0, -0.0, 448.0, 449.0, 464.0, 464.0001, 480.0, 1e30, -1e30, 2.0 ** -10, 2.0 ** -11,
           3 * 2.0 ** -11, 1e-300]
    got = orc.f64_to_e4m3(np.array(xs))
    want = np.array([_e4m3_nearest(x, table) for x in xs], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"e4m3 rounding differs at {xs[bad[0]]!r}: {got[bad[0]]:#x} vs {want[bad[0]]:#x}"
    assert list(orc.f64_to_e4m3(np.array([np.inf, -np.inf]))) == [0x7E, 0xFE]
    assert (orc.f64_to_e4m3(np.array([np.nan]))[0] & 0x7F) == 0x7F


def check_e4m3_matches_torch_on_binary32(orc):
    rng = np.random.default_rng(18)
    x = (np.exp2(rng.uniform(-11.0, 8.8, size=4000)) * np.where(rng.random(4000) < 0.5, -1, 1)).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.f64_to_e4m3(x.astype(np.float64)), want)


def _fp8_case(rng, B, Hkv, cap, D, written):
    kc = np.full((B, Hkv, cap, D), NAN_CODE, np.uint8)
    vc = kc.copy()
    for b in range(B):
        n = written[b]
        kc[b, :, :n] = _random_codes(rng, (Hkv, n, D))
        vc[b, :, :n] = _random_codes(rng, (Hkv, n, D))
    return kc, vc


def check_fp8_layer_vs_brute_force(orc):
    """FP8 full and ring layers: written codes are the brute-force nearest codes of
    the fp64 rotated key / scale (and value / scale); out and lse are a scipy
    brute force over the dequantised key set."""
    table = _e4m3_table()
    rng = np.random.default_rng(19)
    B, Hq, Hkv, D, rot, theta = 2, 4, 2, 16, 8, 1e4
    g = Hq // Hkv
    for layer_type, layout, cap, ctx in ((FULL, 0, 12, np.array([5, 11], np.int32)),
                                         (SLIDING, RING, 7, np.array([3, 12], np.int32))):
        written = np.minimum(ctx, cap)
        kc, vc = _fp8_case(rng, B, Hkv, cap, D, written)
        q = _bf16_bits_random(rng, (B, Hq, D))
        k = _bf16_bits_random(rng, (B, Hkv, D), std=3.0)
        v = _bf16_bits_random(rng, (B, Hkv, D), std=3.0)
        ks = rng.uniform(0.004, 0.02, Hkv).astype(np.float32)
        vs = rng.uniform(0.004, 0.02, Hkv).astype(np.float32)
        sink = rng.standard_normal(Hq).astype(np.float32)
        kc0, vc0 = kc.copy(), vc.copy()
        r = _layer(orc, layer_type=layer_type, layout=layout, window=8, rotary_dim=rot, rope_theta=theta,
                   context=ctx, q=q, k=k, v=v, kcache=kc, vcache=vc, sink=sink, k_scale=ks, v_scale=vs)
        for b in range(B):
            c_, s_ = orc.rope_angles(int(ctx[b]), rot, theta)
            qr = _rope_complex(_bits_to_f64(q[b]), rot, c_, s_)
            kr = _rope_complex(_bits_to_f64(k[b]), rot, c_, s_)
            kq = np.array([[_e4m3_nearest(t / float(ks[h]), table) for t in kr[h]] for h in range(Hkv)], np.uint8)
            vf = _bits_to_f64(v[b])
            vq = np.array([[_e4m3_nearest(t / float(vs[h]), table) for t in vf[h]] for h in range(Hkv)], np.uint8)
            assert np.array_equal(r["k_written"][b], kq), "written key codes"
            if layer_type == FULL:
                slots, lo = [int(ctx[b])], 0
                idx = list(range(int(ctx[b])))
            else:
                c = int(ctx[b])
                idx = [p % cap for p in range(max(0, c - cap), c)]
                slots = [c % cap]
            kd = table[kc0[b][:, idx]] * ks[:, None, None]
            vd = table[vc0[b][:, idx]] * vs[:, None, None]
            keys = np.concatenate([kd, table[kq][:, None] * ks[:, None, None]], axis=1)
            vals = np.concatenate([vd, table[vq][:, None] * vs[:, None, None]], axis=1)
            for h in range(Hq):
                sc = keys[h // g] @ qr[h] / math.sqrt(D)
                lse = sps.logsumexp(sc)
                out = sps.softmax(sc) @ vals[h // g] * sps.expit(lse - sink[h])
                assert np.allclose(r["out"][b, h], out, rtol=1e-12, atol=1e-12), (layer_type, b, h)
                assert abs(r["lse"][b, h] - lse) < 1e-12
            assert np.array_equal(kc[b][:, slots[0]], kq) and np.array_equal(vc[b][:, slots[0]], vq)


def check_fp8_equals_bf16_on_shared_values(orc):
    """With a power-of-two scale and values both formats hold exactly (and no
    rotation), the FP8 layer and the bf16 layer compute bit-identical results and
    write the same values."""
    rng = np.random.default_rng(20)
    B, Hq, Hkv, D = 2, 4, 2, 16
    scale = np.float32(2.0 ** -5)
    table = _e4m3_table()
    ctx = np.array([6, 9], np.int32)
    for layer_type, layout, cap in ((FULL, 0, 10), (SLIDING, RING, 7), (SLIDING, ROLL, 8)):
        written = np.minimum(ctx, cap)
        kc, vc = _fp8_case(rng, B, Hkv, cap, D, written)
        to_bf16 = lambda codes: torch.from_numpy(table[codes] * float(scale)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16).copy()
        kb = np.where(kc == NAN_CODE, NAN_BITS, to_bf16(np.where(kc == NAN_CODE, 0, kc)))
        vb = np.where(vc == NAN_CODE, NAN_BITS, to_bf16(np.where(vc == NAN_CODE, 0, vc)))
        knew_codes = _random_codes(rng, (B, Hkv, D))
        vnew_codes = _random_codes(rng, (B, Hkv, D))
        q = _bf16_bits_random(rng, (B, Hq, D))
        sink = rng.standard_normal(Hq).astype(np.float32)
        args = dict(layer_type=layer_type, layout=layout, window=8, rotary_dim=0, rope_theta=1e4,
                    context=ctx, q=q, k=to_bf16(knew_codes), v=to_bf16(vnew_codes), sink=sink)
        a = _layer(orc, kcache=kc, vcache=vc, k_scale=np.full(Hkv, scale), v_scale=np.full(Hkv, scale), **args)
        b = _layer(orc, kcache=kb, vcache=vb, **args)
        assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"]), layer_type
        assert np.array_equal(a["k_written"], knew_codes)
        assert np.array_equal(b["k_written"], to_bf16(knew_codes))
        for fp8_cache, bf16_cache in ((kc, kb), (vc, vb)):
            held = fp8_cache != NAN_CODE
            assert np.array_equal(to_bf16(np.where(held, fp8_cache, 0))[held], bf16_cache[held])
            assert np.all(bf16_cache[~held] == NAN_BITS)


def check_fp8_history_model(orc):
    """FP8 ring, roll and full caches over many steps from empty against a plain
    list of every past token's codes (brute-force quantised)."""
    table = _e4m3_table()
    rng = np.random.default_rng(21)
    Hq, Hkv, D, rot = 4, 2, 16, 8
    g = Hq // Hkv
    ks = np.array([0.01, 0.02], np.float32)
    vs = np.array([0.015, 0.005], np.float32)
    for layer_type, layout, window, steps in ((SLIDING, RING, 8, 24), (SLIDING, ROLL, 8, 24), (FULL, 0, 8, 14)):
        cap = (window - 1 if layout == RING else window) if layer_type == SLIDING else steps + 1
        kc = np.full((1, Hkv, cap, D), NAN_CODE, np.uint8)
        vc = kc.copy()
        past_k, past_v = [], []
        for c in range(steps):
            q = _bf16_bits_random(rng, (1, Hq, D))
            k = _bf16_bits_random(rng, (1, Hkv, D))
            v = _bf16_bits_random(rng, (1, Hkv, D))
            r = _layer(orc, layer_type=layer_type, layout=layout, window=window, rotary_dim=rot,
                       rope_theta=1e4, context=np.array([c], np.int32), q=q, k=k, v=v,
                       kcache=kc, vcache=vc, k_scale=ks, v_scale=vs)
            past_k.append(r["k_written"][0])
            vf = _bits_to_f64(v[0])
            past_v.append(np.array([[_e4m3_nearest(t / float(vs[h]), table) for t in vf[h]]
                                    for h in range(Hkv)], np.uint8))
            lo = max(0, c - window + 1) if layer_type == SLIDING else 0
            keys = table[np.stack(past_k[lo:c + 1], axis=1)] * ks[:, None, None]
            vals = table[np.stack(past_v[lo:c + 1], axis=1)] * vs[:, None, None]
            for h in range(Hq):
                sc = keys[h // g] @ r["qrot"][0, h] / math.sqrt(D)
                out = sps.softmax(sc) @ vals[h // g]
                assert np.allclose(r["out"][0, h], out, rtol=1e-12, atol=1e-12), (layer_type, layout, c, h)
                assert abs(r["lse"][0, h] - sps.logsumexp(sc)) < 1e-12


# -------------------------------------------------------------- multi-token --

def _layout_cache(hist_k, hist_v, layer_type, layout, window, cap, upto, Hkv, D):
    """Cache [1, Hkv, cap, D] holding positions < upto of a history list as the
    layout keeps them (NaN elsewhere): full at index p, ring at slot p mod cap,
    roll the last `window` positions in order."""
    kc = np.full((1, Hkv, cap, D), NAN_BITS, np.uint16)
    vc = kc.copy()
    if layer_type == FULL:
        idx = {p: p for p in range(upto)}
    elif layout == RING:
        idx = {p: p % cap for p in range(max(0, upto - cap), upto)}
    else:
        lo = max(0, upto - window)
        idx = {p: p - lo for p in range(lo, upto)}
    for p, i in idx.items():
        kc[0, :, i] = hist_k[p]
        vc[0, :, i] = hist_v[p]
    return kc, vc


def check_decode_tokens_brute_force(orc):
    """T tokens in one step: token t (position c+t) attends to every position of its
    window up to c+t -- cached history and the new tokens 0..t -- with its own RoPE;
    the caches end holding the history extended by the T written entries."""
    rng = np.random.default_rng(22)
    Hq, Hkv, D, rot, theta, W = 4, 2, 16, 8, 1e4, 8
    g = Hq // Hkv
    for layer_type, layout in ((FULL, 0), (SLIDING, RING), (SLIDING, ROLL)):
        for c, T in ((3, 4), (6, 5), (13, 6), (0, 3)):
            cap = (W - 1 if layout == RING else W) if layer_type == SLIDING else c + T + 2
            hist_k = [_bf16_bits_random(rng, (Hkv, D)) for _ in range(c)]
            hist_v = [_bf16_bits_random(rng, (Hkv, D)) for _ in range(c)]
            kc, vc = _layout_cache(hist_k, hist_v, layer_type, layout, W, cap, c, Hkv, D)
            q = _bf16_bits_random(rng, (1, T, Hq, D))
            k = _bf16_bits_random(rng, (1, T, Hkv, D))
            v = _bf16_bits_random(rng, (1, T, Hkv, D))
            sink = rng.standard_normal(Hq).astype(np.float32)
            gate = rng.standard_normal((1, T, Hq)).astype(np.float32)
            r = orc.decode_tokens(layer_type=layer_type, layout=layout, window=W, rotary_dim=rot,
                                  rope_theta=theta, context=np.array([c], np.int32), q=q, k=k, v=v,
                                  kcache=kc, vcache=vc, sink=sink, gate=gate)
            for t in range(T):
                pos = c + t
                cs, sn = orc.rope_angles(pos, rot, theta)
                kr = _rope_complex(_bits_to_f64(k[0, t]), rot, cs, sn)
                hist_k.append(np.array([[orc.lib.orc_f64_to_bf16(float(x)) for x in row] for row in kr], np.uint16))
                hist_v.append(v[0, t])
                lo = max(0, pos - W + 1) if layer_type == SLIDING else 0
                keys = _bits_to_f64(np.stack(hist_k[lo:pos + 1], axis=1))   # [Hkv, n, D]
                vals = _bits_to_f64(np.stack(hist_v[lo:pos + 1], axis=1))
                qr = _rope_complex(_bits_to_f64(q[0, t]), rot, cs, sn)
                for h in range(Hq):
                    sc = keys[h // g] @ qr[h] / math.sqrt(D)
                    lse = sps.logsumexp(sc)
                    out = sps.softmax(sc) @ vals[h // g] * sps.expit(lse - float(sink[h])) * sps.expit(float(gate[0, t, h]))
                    assert np.allclose(r["out"][0, t, h], out, rtol=1e-12, atol=1e-12), (layer_type, layout, c, t, h)
                    assert abs(r["lse"][0, t, h] - lse) < 1e-12, (layer_type, layout, c, t, h)
            ek, ev = _layout_cache(hist_k, hist_v, layer_type, layout, W, cap, c + T, Hkv, D)
            assert np.array_equal(kc, ek) and np.array_equal(vc, ev), (layer_type, layout, c, T)


# -------------------------------------------------------------- footprint --

def check_kv_cache_bytes_golden(orc):
    with open(os.path.join(GOLDEN, "spark_kv_cache_bytes_4k.json")) as f:
        gold = json.load(f)
    types = [SLIDING, SLIDING, SLIDING, FULL] * 7
    hyb, uni = orc.kv_cache_bytes(types, RING, 512, gold["num_kv_heads"], gold["head_dim"],
                                  gold["context"], gold["bytes_per_elem"])
    assert round(hyb / 1e6) == gold["printed_hybrid"], hyb
    assert round(uni / 1e6) == gold["printed_uniform"], uni
    assert hyb == gold["hybrid_bytes"] and uni == gold["uniform_bytes"]


def check_cache_len_cases(orc):
    for c in (0, 1, 510, 511, 512, 513, 4096):
        assert orc.cache_len(SLIDING, RING, 512, c) == min(c, 511)
        assert orc.cache_len(SLIDING, ROLL, 512, c) == min(c, 512)
        assert orc.cache_len(FULL, 0, 512, c) == c


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
