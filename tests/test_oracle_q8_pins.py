"""Pins for the oracle's quantised KV (Q8_0, one of the kv_type choices of "How to
Implement Long Context Inference (Up to 139K Tokens) with KTransformers", Step 1).

Reading under test: a 128-channel row of K or V is cut into 4 groups of 32; a
group keeps a binary16 scale and 32 signed 8-bit codes; with amax the group's
largest |x| (binary32), dd = amax / 127 and id = 1 / dd (binary32), a code is
round-half-away-from-zero(x * id) and the scale is dd rounded to binary16; a
dequantised value is scale * code.

The pins do not retype that formula: the binary16 encoder is checked against
numpy's, codes are checked where quantisation must be exact (values on each
group's own grid of 127 steps), against error and sign bounds that hold for
any input, and attention over exactly quantisable KV must equal attention over
the fp16 KV (so a scale applied to the wrong row or group fails).
"""
import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(4321)


def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _dec(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_binary16_encoder_matches_numpy():
    vals = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32) * s
        for s in (1e-7, 1e-5, 1e-3, 0.1, 1.0, 30.0, 1e3, 3e4)] + [
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 7e4, -7e4, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25], dtype=np.float32),
        # exact halfway cases between neighbouring binary16 values (ties to even)
        (np.arange(1024, 2048, dtype=np.float32) + 0.5) * np.float32(2.0 ** -10),
        (np.arange(1, 1024, dtype=np.float32) + 0.5) * np.float32(2.0 ** -24)])
    with np.errstate(over="ignore"):  # values past 65520 round to infinity on purpose
        want = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(want[i])) for i in bad[:5]]


def _grid_rows(rows, rng):
    """Rows whose every 32-channel group lies on its own grid: values m * 2^-e
    with integers |m| <= 127, one of them at +-127 (the group's amax)."""
    x = np.zeros((rows, 128))
    e = rng.integers(0, 11, size=(rows, 4))
    m = rng.integers(-127, 128, size=(rows, 128))
    for r in range(rows):
        for g in range(4):
            j = g * 32 + int(rng.integers(0, 32))
            m[r, j] = 127 if rng.random() < 0.5 else -127
    for r in range(rows):
        for g in range(4):
            x[r, g * 32:(g + 1) * 32] = m[r, g * 32:(g + 1) * 32] * 2.0 ** -float(e[r, g])
    return x, m, e


def test_codes_exact_on_group_grids():
    x, m, e = _grid_rows(300, RNG)
    code, scale = oracle.quantize_q8_0(_f16(x))
    assert np.array_equal(code.astype(np.int64), m)
    assert np.array_equal(_dec(scale), 2.0 ** -e.astype(np.float64))


def test_zero_group_and_bounds_on_random_rows():
    x = RNG.standard_normal((400, 128)) * RNG.choice([1e-3, 1.0, 50.0], size=(400, 1))
    x[7, 32:64] = 0.0                       # an all-zero group
    bits = _f16(x)
    code, scale = oracle.quantize_q8_0(bits)
    xv = _dec(bits)
    assert np.all(code[7, 32:64] == 0) and scale[7, 1] == 0
    c = code.astype(np.float64).reshape(400, 4, 32)
    xs = xv.reshape(400, 4, 32)
    amax = np.abs(xs).max(axis=2, keepdims=True)
    deq = c * _dec(scale)[:, :, None]
    # |x - scale*code| <= half a step plus 127 times the binary16 rounding of
    # the step (half an ulp: 2^-11 relative, or 2^-25 for subnormal steps)
    step = amax / 127
    rnd = np.maximum(step * 2.0 ** -11, 2.0 ** -25)
    assert np.all(np.abs(xs - deq) <= 0.5 * step * (1 + 1e-6) + 127 * rnd)
    assert np.all(np.abs(c) <= 127)
    assert np.all(np.sign(c) * np.sign(xs) >= 0)          # never the wrong sign
    top = np.abs(xs) == amax                               # the largest |x| maps to +-127
    assert np.all(np.abs(c[top & (amax > 0)]) == 127)
    # codes are monotone in x within a group
    for r in range(0, 400, 37):
        for g in range(4):
            o = np.argsort(xs[r, g], kind="stable")
            assert np.all(np.diff(c[r, g][o]) >= 0)


def _grid_kv(seed, lens, H_kv=2):
    """A paged KV (permuted pages) whose K and V rows lie on per-group grids."""
    rng = np.random.default_rng(seed)
    w = synth.custom(seed, lens, num_q_heads=2 * H_kv, num_kv_heads=H_kv, rep=synth.REP_QUEST,
                     top_k=3, permute_pages=True)
    P = w.num_pages
    xk, _, _ = _grid_rows(P * H_kv * 128, rng)
    xv, _, _ = _grid_rows(P * H_kv * 128, rng)
    w.k_pool = _f16(xk).reshape(P, H_kv, 128, 128)
    w.v_pool = _f16(xv).reshape(P, H_kv, 128, 128)
    return w


def test_attention_over_exact_q8_equals_fp16_attention():
    w = _grid_kv(61, [128 * 9 + 70, 128 * 5])
    kv = oracle.KV.of(w)
    kvq = oracle.KVQ(kv)
    ref = oracle.sparse_step(kv, w.q, w.params)
    got = oracle.attend_selection_q8(kvq, w.q, w.params, ref["sel"], ref["cnt"])
    want = oracle.attend_selection(kv, w.q, w.params, ref["sel"], ref["cnt"])
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14)
    assert np.allclose(want, ref["out"], rtol=1e-12, atol=1e-14)


def test_attention_over_random_q8_is_close_to_fp16():
    # quantisation error of ~half a step per element moves the output by far
    # less than the values themselves
    w = synth.custom(62, [128 * 12 + 3], num_q_heads=4, num_kv_heads=2, rep=synth.REP_QUEST,
                     top_k=4)
    kv = oracle.KV.of(w)
    ref = oracle.sparse_step(kv, w.q, w.params)
    got = oracle.attend_selection_q8(oracle.KVQ(kv), w.q, w.params, ref["sel"], ref["cnt"])
    err = np.abs(got - ref["out"]).max(-1) / np.abs(ref["out"]).max(-1)
    assert 0 < err.max() < 0.1
