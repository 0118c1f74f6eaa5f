"""Pins of the CPU oracle: checks against what the pages and mathematics fix.

Each pin takes an ``oracle.Oracle`` and a scratch directory and raises
``AssertionError`` when the oracle disagrees with a printed value, a closed
form, an invariant or an exact computation.  ``test_oracle_pins.py`` runs them
on the oracle itself; ``test_oracle_mutants.py`` runs them on copies of the
oracle with one planted mistake each and requires that some pin fails.

None of the pins re-types the oracle's own formula: they use the pages'
printed numbers (``golden/``), closed forms that follow from the definitions
(t = 1, constant gradient, zero gradient), exact sums (``math.fsum``),
Pythagorean triples, and the checkpoint's byte layout read back by hand.
"""
from __future__ import annotations

import json
import math
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
B1, B2, EPS = 0.9, 0.999, 1e-8


def read_golden(name):
    inputs, expects, other = {}, {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "input":
                inputs[parts[1]] = float(parts[2])
            elif parts[0] == "expect":
                expects[parts[1]] = (float(parts[2]), float(parts[3]))
            else:
                other[parts[0]] = parts[1:]
    return inputs, expects, other


# --- the pages' worked example ---------------------------------------------

def pin_example1(o, tmp):
    """Example 1: m, v, bias-corrected moments, decayed and final weight."""
    inp, exp, _ = read_golden("example1.txt")
    s = o.clip_scale(abs(inp["g"]), inp["clip"])
    r = o.adamw_element(inp["w"], inp["g"], 0.0, 0.0, s, int(inp["t"]),
                        inp["lr"], inp["wd"])
    r["scale"] = s
    for k, (val, tol) in exp.items():
        assert abs(r[k] - val) <= tol, (k, r[k], val, tol)


def pin_example1_float32_state(o, tmp):
    """Example 1 through the float32 vector step: same printed values after
    one rounding to float32."""
    inp, exp, _ = read_golden("example1.txt")
    w = np.array([inp["w"]], np.float32)
    g = np.array([inp["g"]], np.float32)
    m = np.zeros(1, np.float32)
    v = np.zeros(1, np.float32)
    st, norm = o.adamw_clip_step(w, g, m, v, 1, inp["lr"], inp["wd"], inp["clip"])
    assert st == 0 and norm == 0.5
    for k, arr in (("w", w), ("m", m), ("v", v)):
        val, tol = exp[k]
        # one float32 rounding of the exact value, plus the printed tolerance
        assert abs(float(arr[0]) - val) <= tol + abs(val) * 2.0 ** -24, (k, arr[0])


def _scalar_step(o, state, g, clip, lr, wd):
    w, m, v, t = state
    s = o.clip_scale(abs(g), clip)
    r = o.adamw_element(w, g, m, v, s, t + 1, lr, wd)
    return [r["w"], r["m"], r["v"], t + 1]


def pin_worked_code_resume(o, tmp):
    """The worked code's three assertions (first step, exact resume from the
    full state after a JSON round trip, weights-only resume diverges)."""
    _, _, g = read_golden("worked_code_resume.txt")
    w0 = float(g["w0"][0])
    grads = [float(x) for x in g["grads"]]
    clip, lr, wd = float(g["clip"][0]), float(g["lr"][0]), float(g["wd"][0])
    state = [w0, 0.0, 0.0, 0]
    first = _scalar_step(o, state, grads[0], clip, lr, wd)
    assert abs(first[0] - float(g["first_w"][0])) < float(g["first_w"][1])
    cont = state
    for x in grads:
        cont = _scalar_step(o, cont, x, clip, lr, wd)
    prefix = state
    for x in grads[:2]:
        prefix = _scalar_step(o, prefix, x, clip, lr, wd)
    resumed = _scalar_step(o, json.loads(json.dumps(prefix)), grads[2], clip, lr, wd)
    assert cont == resumed
    wrong = _scalar_step(o, [prefix[0], 0.0, 0.0, 0], grads[2], clip, lr, wd)
    assert abs(wrong[0] - cont[0]) > float(g["weights_only_min_gap"][0])


def pin_second_step_moments(o, tmp):
    """Step 2 of the worked example (gradient -0.25): the moments are the
    exponential averages 0.9*0.05 + 0.1*(-0.25) = 0.02 and
    0.999*0.00025 + 0.001*0.0625 = 0.00031225 (hand arithmetic)."""
    s1 = _scalar_step(o, [2.0, 0.0, 0.0, 0], 0.5, 1.0, 0.1, 0.01)
    s2 = _scalar_step(o, s1, -0.25, 1.0, 0.1, 0.01)
    assert abs(s2[1] - 0.02) < 1e-15 and abs(s2[2] - 0.00031225) < 1e-15
    # bias-corrected: 0.02/(1-0.81) and 0.00031225/(1-0.998001)
    r = o.adamw_element(s1[0], -0.25, s1[1], s1[2], 1.0, 2, 0.1, 0.01)
    assert abs(r["m_hat"] - 0.02 / 0.19) < 1e-14
    assert abs(r["v_hat"] - 0.00031225 / 0.001999) < 1e-13


# --- AdamW closed forms ------------------------------------------------------

def pin_t1_closed_form(o, tmp):
    """At t = 1 from zero moments, m_hat = g_hat and v_hat = g_hat^2 for any
    betas, so the update is lr*g_hat/(|g_hat| + eps)."""
    rng = np.random.default_rng(1)
    for b1, b2 in ((0.9, 0.999), (0.5, 0.7), (0.8, 0.95)):
        for gh in list(rng.normal(0, 1, 8)) + [1e-8, -3e-9, 250.0]:
            w, lr, wd = 0.75, 0.01, 0.1
            r = o.adamw_element(w, gh, 0.0, 0.0, 1.0, 1, lr, wd, b1, b2, EPS)
            want_upd = lr * gh / (abs(gh) + EPS)
            assert math.isclose(r["m_hat"], gh, rel_tol=1e-14)
            assert math.isclose(r["v_hat"], gh * gh, rel_tol=1e-14)
            assert math.isclose(r["update"], want_upd, rel_tol=1e-13), (gh, r)
            assert math.isclose(r["w"], w * (1 - lr * wd) - want_upd,
                                rel_tol=1e-13, abs_tol=1e-15)


def pin_eps_position(o, tmp):
    """eps is added to sqrt(v_hat): a gradient equal to eps at t = 1 moves the
    weight by exactly lr/2 (no decay)."""
    r = o.adamw_element(1.0, EPS, 0.0, 0.0, 1.0, 1, 0.2, 0.0)
    assert math.isclose(r["update"], 0.1, rel_tol=1e-12), r
    assert math.isclose(r["w"], 0.9, rel_tol=1e-12)


def pin_constant_gradient(o, tmp):
    """A constant gradient gamma gives m_t = gamma (1-b1^t) and
    v_t = gamma^2 (1-b2^t), so m_hat = gamma and v_hat = gamma^2 at every t:
    each update is lr*gamma/(|gamma|+eps) and
    w_t = w0 d^t - u (1 - d^t)/(1 - d) with d = 1 - lr wd."""
    gamma, lr, wd, w0 = -0.3, 0.05, 0.2, 1.5
    d = 1 - lr * wd
    u = lr * gamma / (abs(gamma) + EPS)
    state = [w0, 0.0, 0.0, 0]
    for t in range(1, 41):
        r = o.adamw_element(state[0], gamma, state[1], state[2], 1.0, t, lr, wd)
        state = [r["w"], r["m"], r["v"], t]
        assert math.isclose(r["m"], gamma * (1 - B1 ** t), rel_tol=1e-12)
        assert math.isclose(r["v"], gamma * gamma * (1 - B2 ** t), rel_tol=1e-12)
        assert math.isclose(r["m_hat"], gamma, rel_tol=1e-12), (t, r)
        assert math.isclose(r["v_hat"], gamma * gamma, rel_tol=1e-12), (t, r)
        want = w0 * d ** t - u * (1 - d ** t) / (1 - d)
        assert math.isclose(r["w"], want, rel_tol=1e-12), (t, r["w"], want)


def pin_zero_gradient(o, tmp):
    """A zero gradient decays the weight only and shrinks the moments by the
    betas: w' = w (1 - lr wd), m' = b1 m, v' = b2 v (with v > 0 the update
    is lr m_hat/(sqrt(v_hat)+eps) of the shrunk moments)."""
    r = o.adamw_element(3.0, 0.0, 0.0, 0.0, 1.0, 5, 0.01, 0.5)
    assert r["update"] == 0.0 and math.isclose(r["w"], 3.0 * (1 - 0.005), rel_tol=1e-15)
    r = o.adamw_element(3.0, 0.0, 0.2, 0.04, 1.0, 1, 0.01, 0.0)
    assert math.isclose(r["m"], B1 * 0.2, rel_tol=1e-15)
    assert math.isclose(r["v"], B2 * 0.04, rel_tol=1e-15)


def pin_decay_on_every_parameter(o, tmp):
    """Weight decay is decoupled and multiplies the OLD weight: with lr = 1e-3
    and wd = 1, the decay term is w*lr*wd independent of the update."""
    for w in (-2.0, 0.5, 4.0):
        r = o.adamw_element(w, 0.25, 0.0, 0.0, 1.0, 1, 1e-3, 1.0)
        assert math.isclose(r["w_decayed"], w * (1 - 1e-3), rel_tol=1e-15)
        assert math.isclose(r["w"] - r["w_decayed"], -r["update"], rel_tol=1e-12)


def pin_update_ranges_compose_to_the_step(o, tmp):
    """Updating disjoint ranges that cover [0, n), each with the clip factor
    of the whole gradient, is the full step bit for bit (the update of one
    element depends on that element and s only)."""
    rng = np.random.default_rng(23)
    n = 1001
    w0 = rng.normal(0, 0.05, n).astype(np.float32)
    g = rng.normal(0, 0.3, n).astype(np.float32)
    m0 = rng.normal(0, 0.01, n).astype(np.float32)
    v0 = np.abs(rng.normal(0, 1e-3, n)).astype(np.float32)
    wa, ma, va = w0.copy(), m0.copy(), v0.copy()
    _, norm = o.adamw_clip_step(wa, g, ma, va, 5, 2e-3, 0.05, 1.0)
    s = o.clip_scale(norm, 1.0)
    assert s < 1.0
    wb, mb, vb = w0.copy(), m0.copy(), v0.copy()
    for lo, hi in ((700, 1001), (0, 1), (1, 333), (333, 333), (333, 700)):
        o.adamw_update_range(wb, g, mb, vb, lo, hi, s, 5, 2e-3, 0.05)
    assert wa.tobytes() == wb.tobytes() and ma.tobytes() == mb.tobytes()
    assert va.tobytes() == vb.tobytes()
    wc = w0.copy()
    o.adamw_update_range(wc, g, m0.copy(), v0.copy(), 10, 20, s, 5, 2e-3, 0.05)
    assert wc[:10].tobytes() == w0[:10].tobytes() and wc[20:].tobytes() == w0[20:].tobytes()
    assert np.all(wc[10:20] != w0[10:20])


# --- per-group weight decay ---------------------------------------------------

_MASK_SIZES = (5, 3, 8, 1, 13, 4, 7, 2)
_MASK_FLAGS = (1, 0, 0, 1, 0, 1, 1, 0)


def _mask_table():
    num = np.array(_MASK_SIZES, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    return off, num, int(num.sum())


def pin_decay_mask_partition(o, tmp):
    """A per-tensor decay flag splits the step: every element of a flagged
    tensor is bit for bit the plain step with wd, every element of an exempt
    one the plain step with wd = 0, and the norm (hence the clip) stays
    global.  The flags are not shift-symmetric, so an index slip shows."""
    off, num, n = _mask_table()
    rng = np.random.default_rng(21)
    w0 = rng.normal(0, 0.5, n).astype(np.float32)
    g = rng.normal(0, 0.6, n).astype(np.float32)
    m0 = rng.normal(0, 0.01, n).astype(np.float32)
    v0 = np.abs(rng.normal(0, 1e-3, n)).astype(np.float32)
    lr, wd = 0.05, 0.3
    outs = []
    for mode in ("mask", "wd", "zero"):
        w, m, v = w0.copy(), m0.copy(), v0.copy()
        if mode == "mask":
            _, norm = o.adamw_clip_step_masked(w, g, m, v, off, num, _MASK_FLAGS, 3, lr, wd, 1.0)
        else:
            _, norm = o.adamw_clip_step(w, g, m, v, 3, lr, wd if mode == "wd" else 0.0, 1.0)
        outs.append((w, m, v, norm))
    (wm, mm, vm, nm), (wa, ma, va, na), (wb, mb, vb, nb) = outs
    assert nm == na == nb and o.clip_scale(nm, 1.0) < 1.0
    assert mm.tobytes() == ma.tobytes() and vm.tobytes() == va.tobytes()
    for k, flag in enumerate(_MASK_FLAGS):
        sl = slice(off[k], off[k] + num[k])
        ref = wa if flag else wb
        assert wm[sl].tobytes() == ref[sl].tobytes(), (k, flag)
        other = wb if flag else wa
        assert np.all(wm[sl] != other[sl]), (k, flag)  # wd changes every weight here


def pin_decay_mask_closed_forms(o, tmp):
    """Example 1 with its one tensor exempt: at t = 1, m_hat = g_hat and
    sqrt(v_hat) = |g_hat|, so w = 2 - 0.1 * 0.5 / (0.5 + 1e-8) (no 1 - lr wd
    factor).  With all flags set the masked step is the plain step bit for
    bit.  A zero gradient leaves an exempt weight exactly as it was and
    decays a flagged one by exactly float32(w (1 - lr wd))."""
    inp, _, _ = read_golden("example1.txt")
    w = np.array([inp["w"]], np.float32)
    m = np.zeros(1, np.float32)
    v = np.zeros(1, np.float32)
    o.adamw_clip_step_masked(w, np.array([inp["g"]], np.float32), m, v, [0], [1], [0],
                             1, inp["lr"], inp["wd"], inp["clip"])
    want = 2.0 - 0.1 * 0.5 / (0.5 + 1e-8)
    assert abs(float(w[0]) - want) <= 2.0 ** -22, (w[0], want)
    assert abs(float(w[0]) - 1.898) > 1e-3  # the decayed value is not reached

    off, num, n = _mask_table()
    rng = np.random.default_rng(22)
    w0 = rng.normal(0, 1.0, n).astype(np.float32)
    g = rng.normal(0, 0.1, n).astype(np.float32)
    wa, ma, va = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    wm, mm, vm = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    o.adamw_clip_step(wa, g, ma, va, 2, 1e-2, 0.1, 1.0)
    o.adamw_clip_step_masked(wm, g, mm, vm, off, num, np.ones(len(num)), 2, 1e-2, 0.1, 1.0)
    assert wa.tobytes() == wm.tobytes() and ma.tobytes() == mm.tobytes()

    z = np.zeros(n, np.float32)
    wz, mz, vz = w0.copy(), z.copy(), z.copy()
    o.adamw_clip_step_masked(wz, z, mz, vz, off, num, _MASK_FLAGS, 1, 0.25, 0.5, 1.0)
    for k, flag in enumerate(_MASK_FLAGS):
        sl = slice(off[k], off[k] + num[k])
        if flag:
            want = (w0[sl].astype(np.float64) * (1.0 - 0.25 * 0.5)).astype(np.float32)
            assert wz[sl].tobytes() == want.tobytes(), k
        else:
            assert wz[sl].tobytes() == w0[sl].tobytes(), k


def pin_decay_mask_rejects_bad_table(o, tmp):
    """The tensors must tile [0, n) in order: a gap, an overlap or a short
    cover is refused and leaves the state untouched."""
    n = 10
    for off, num in (([0, 6], [5, 4]), ([0, 4], [5, 5]), ([0, 5], [5, 4])):
        w = np.ones(n, np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        try:
            o.adamw_clip_step_masked(w, np.ones(n, np.float32), m, v, off, num, [1, 0],
                                     1, 0.1, 0.1, 1.0)
        except Exception:  # noqa: BLE001 - the refusal is the expected outcome
            pass
        else:
            raise AssertionError(f"table {off} {num} accepted")
        assert np.all(w == 1.0) and np.all(m == 0.0)


# --- norm and clip -----------------------------------------------------------

def pin_norm_pythagorean(o, tmp):
    for vec, want in (([3, 4], 5.0), ([1, 2, 2], 3.0), ([2, 3, 6], 7.0),
                      ([-3, -4], 5.0), ([0, 0, 0], 0.0), ([8, 9, 12], 17.0)):
        assert o.global_norm(np.array(vec, np.float32)) == want, vec


def pin_norm_constant(o, tmp):
    """g = k everywhere: ||g|| = |k| sqrt(n), exact for k = 0.5, n = 4096."""
    assert o.global_norm(np.full(4096, 0.5, np.float32)) == 32.0
    assert o.global_norm(np.full(10000, -0.25, np.float32)) == 25.0


def pin_norm_exact_sum(o, tmp):
    """Squares of float32 values are exact in double, so math.fsum of them is
    the correctly rounded sum of squares; the index-order sum stays within
    n ulps of it."""
    rng = np.random.default_rng(2)
    for n in (1, 7, 1000, 65537):
        g = (rng.standard_normal(n) * rng.choice([1e-3, 1.0, 40.0], n)).astype(np.float32)
        exact = math.fsum(float(x) * float(x) for x in g)
        got = o.sumsq(g)
        assert abs(got - exact) <= n * 2.3e-16 * exact, (n, got, exact)
        assert math.isclose(o.global_norm(g), math.sqrt(exact), rel_tol=n * 2.3e-16)


def pin_tensor_norms(o, tmp):
    """Per-tensor sums: Pythagorean tensors give 25, 169 and 0; the tensor
    sums add up to the global sum exactly for small integers; a one-tensor
    table gives the global sum."""
    g = np.array([3, 4, 5, 12, 0, 0, 0, 1, 2, 2], np.float32)
    got = o.tensor_sumsq(g, [0, 2, 4, 7], [2, 2, 3, 3])
    assert list(got) == [25.0, 169.0, 0.0, 9.0]
    assert got.sum() == o.sumsq(g)
    rng = np.random.default_rng(13)
    h = rng.integers(-50, 51, 1000).astype(np.float32)
    bounds = [0, 1, 2, 10, 500, 999]
    off = bounds
    num = [b - a for a, b in zip(bounds, bounds[1:] + [1000])]
    assert o.tensor_sumsq(h, off, num).sum() == o.sumsq(h)
    assert o.tensor_sumsq(h, [0], [1000])[0] == o.sumsq(h)


def pin_norm_homogeneous(o, tmp):
    """||2^k g|| = 2^k ||g|| exactly (power-of-two scaling is exact)."""
    g = np.random.default_rng(3).standard_normal(999).astype(np.float32)
    base = o.global_norm(g)
    assert o.global_norm(g * np.float32(4.0)) == 4.0 * base
    assert o.global_norm(g * np.float32(0.125)) == 0.125 * base


def pin_clip_closed_forms(o, tmp):
    """clip(g) has norm <= c, keeps the direction, and is g itself when
    ||g|| <= c (strict '>' in the threshold test)."""
    assert o.clip_scale(5.0, 5.0) == 1.0          # ||g|| == c: unchanged
    assert o.clip_scale(0.0, 1.0) == 1.0          # zero gradient: no division
    assert o.clip_scale(10.0, 5.0) == 0.5         # [6, 8] with c = 5
    rng = np.random.default_rng(4)
    for c in (0.1, 1.0, 30.0):
        g = rng.standard_normal(500) * rng.uniform(0.01, 5)
        norm = o.global_norm(g.astype(np.float32))
        s = o.clip_scale(norm, c)
        clipped = g.astype(np.float32).astype(np.float64) * s
        assert np.linalg.norm(clipped) <= c * (1 + 1e-12) or s == 1.0
        if norm <= c:
            assert s == 1.0
        else:
            assert math.isclose(np.linalg.norm(clipped), c, rel_tol=1e-12)
        assert s > 0


def pin_clipped_vector_step(o, tmp):
    """First vector step with clipping: m = (1-b1) s g, v = (1-b2) (s g)^2
    and w = w d - lr sign(g) |s g|/(|s g| + eps), each rounded to float32
    once, with s = c/||g|| from the Pythagorean vector [30, 40] (norm 50)."""
    g = np.array([30.0, 40.0, 0.0], np.float32)
    w = np.array([1.0, -1.0, 0.5], np.float32)
    m = np.zeros(3, np.float32)
    v = np.zeros(3, np.float32)
    lr, wd, c = 0.01, 0.1, 1.0
    st, norm = o.adamw_clip_step(w, g, m, v, 1, lr, wd, c)
    assert st == 0 and norm == 50.0
    s = c / 50.0
    gh = np.array([30.0 * s, 40.0 * s, 0.0])
    want_m = (1 - B1) * gh
    want_v = (1 - B2) * gh * gh
    upd = np.where(gh != 0, lr * gh / (np.abs(gh) + EPS), 0.0)
    want_w = np.array([1.0, -1.0, 0.5]) * (1 - lr * wd) - upd
    for got, want in ((m, want_m), (v, want_v), (w, want_w)):
        assert np.all(np.abs(got.astype(np.float64) - want)
                      <= np.abs(want) * 2.0 ** -24 + 1e-30), (got, want)


def pin_nonfinite_gradient(o, tmp):
    """An inf or nan gradient gives a non-finite norm: status ENONFINITE and
    the state is left bit-for-bit unchanged."""
    for bad in (np.inf, -np.inf, np.nan):
        g = np.array([0.1, bad, 0.2], np.float32)
        w = np.array([1.0, 2.0, 3.0], np.float32)
        m = np.array([0.1, 0.2, 0.3], np.float32)
        v = np.array([0.01, 0.02, 0.03], np.float32)
        before = (w.copy(), m.copy(), v.copy())
        st, norm = o.adamw_clip_step(w, g, m, v, 3, 0.1, 0.01, 1.0,
                                     raise_on_error=False)
        assert st == 6 and not math.isfinite(norm)
        for a, b in zip((w, m, v), before):
            assert a.tobytes() == b.tobytes()


def pin_step_matches_elements(o, tmp):
    """The vector step equals, element by element, the scalar update fed the
    vector's clip factor (the composition norm -> clip -> AdamW)."""
    rng = np.random.default_rng(5)
    n = 257
    w = rng.normal(0, 0.02, n).astype(np.float32)
    g = rng.normal(0, 0.2, n).astype(np.float32)
    m = rng.normal(0, 0.01, n).astype(np.float32)
    v = np.abs(rng.normal(0, 1e-4, n)).astype(np.float32)
    w0, m0, v0 = w.copy(), m.copy(), v.copy()
    st, norm = o.adamw_clip_step(w, g, m, v, 4, 3e-3, 0.01, 1.0)
    s = o.clip_scale(norm, 1.0)
    assert s < 1.0
    ws, ms, vs = o.adamw_at(np.arange(n), w0, g, m0, v0, s, 4, 3e-3, 0.01)
    assert w.tobytes() == ws.tobytes() and m.tobytes() == ms.tobytes()
    assert v.tobytes() == vs.tobytes()


def pin_scaled_step_power_of_two(o, tmp):
    """Scaling the gradient by 2^-k is exact: the scaled step equals the
    plain step on g * 2^-k, bit for bit (norm, state)."""
    rng = np.random.default_rng(9)
    n = 300
    g = rng.normal(0, 3.0, n).astype(np.float32)
    for gs in (0.5, 0.25, 2.0 ** -7):
        a = [rng.normal(0, 0.02, n).astype(np.float32), np.zeros(n, np.float32),
             np.zeros(n, np.float32)]
        b = [x.copy() for x in a]
        _, n1 = o.adamw_clip_step_scaled(*a[:1], g, *a[1:], 1, 3e-3, 0.01, 1.0, gs)
        _, n2 = o.adamw_clip_step(b[0], g * np.float32(gs), b[1], b[2], 1, 3e-3, 0.01, 1.0)
        assert n1 == n2
        for x, y in zip(a, b):
            assert x.tobytes() == y.tobytes()


def pin_scaled_step_clips_the_scaled_norm(o, tmp):
    """The clip sees the averaged gradient: [3, 4] scaled by 1/4 has norm
    1.25 < 2 (no clip, m = 0.1 * 0.75 at t = 1); [30, 40] scaled by 1/2 has
    norm 25 > 1 (factor 1/25: g_hat = [0.6, 0.8])."""
    for g, gs, c, want_norm, want_m in (([3, 4], 0.25, 2.0, 1.25, [0.075, 0.1]),
                                        ([30, 40], 0.5, 1.0, 25.0, [0.06, 0.08])):
        w = np.zeros(2, np.float32)
        m = np.zeros(2, np.float32)
        v = np.zeros(2, np.float32)
        _, norm = o.adamw_clip_step_scaled(w, np.array(g, np.float32), m, v, 1, 0.1, 0.0, c, gs)
        assert norm == want_norm
        assert np.allclose(m, np.array(want_m, np.float32), rtol=2 ** -23, atol=0)


def pin_micro_batch_average(o, tmp):
    """Accumulating k micro-batch gradients and scaling by 1/k is the step on
    their mean (small integers: the sums and the 1/4 are exact)."""
    rng = np.random.default_rng(10)
    parts = [rng.integers(-8, 9, 64).astype(np.float32) for _ in range(4)]
    acc = np.sum(parts, axis=0).astype(np.float32)
    mean = (acc / np.float32(4)).astype(np.float32)
    a = [np.full(64, 0.5, np.float32), np.zeros(64, np.float32), np.zeros(64, np.float32)]
    b = [x.copy() for x in a]
    o.adamw_clip_step_scaled(a[0], acc, a[1], a[2], 2, 0.01, 0.1, 5.0, 0.25)
    o.adamw_clip_step(b[0], mean, b[1], b[2], 2, 0.01, 0.1, 5.0)
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()


# --- 16-bit formats of the mixed-precision step ------------------------------

def pin_decode16_values(o, tmp):
    """Hand-decoded bit patterns: bfloat16 is the top half of a binary32;
    binary16 has bias 15, 10 fraction bits, subnormals at 2^-24 steps."""
    for h, want in ((0x3F80, 1.0), (0xC000, -2.0), (0x3EAB, 0.333984375), (0x0001, 2.0 ** -133),
                    (0x7F7F, 3.3895313892515355e38), (0x7F80, math.inf)):
        assert o.decode16(h, 1) == want, hex(h)
    for h, want in ((0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24),
                    (0x0400, 2.0 ** -14), (0x7BFF, 65504.0), (0xC000, -2.0),
                    (0x3555, 0.333251953125), (0x7C00, math.inf), (0xFC00, -math.inf)):
        assert o.decode16(h, 2) == want, hex(h)
    assert math.isnan(o.decode16(0x7E00, 2)) and math.isnan(o.decode16(0x7FC0, 1))
    assert math.copysign(1.0, o.decode16(0x8000, 2)) == -1.0


def pin_encode_f16_matches_numpy(o, tmp):
    """binary16 rounding equals numpy's float16 conversion (nearest, ties to
    even) bit for bit, across subnormals, normals, ties and overflow."""
    rng = np.random.default_rng(14)
    x = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)).astype(np.float32),
        np.array([65504, 65519.99, 65520, 70000, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                  2.0 ** -14 - 2.0 ** -25, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.0, -0.0,
                  np.inf, -np.inf], np.float32)])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = np.array([o.encode16(v, 2) for v in x], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], want[bad[:5]])


def pin_encode_bf16_nearest_even(o, tmp):
    """bfloat16 rounding picks the nearer of the two neighbouring bfloat16
    values (distances compared in double), ties to the even pattern."""
    rng = np.random.default_rng(15)
    x = (rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000)).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 5 * 2.0 ** -8)], np.float32)
    for v in np.concatenate([x, ties]):
        bits = int(np.float32(v).view(np.uint32))
        lo = bits >> 16
        cands = [(lo, o.decode16(lo, 1)), (lo + 1, o.decode16(lo + 1, 1))]
        d = [abs(c - float(v)) for _, c in cands]
        if d[0] != d[1]:
            want = cands[0][0] if d[0] < d[1] else cands[1][0]
        else:
            want = cands[0][0] if cands[0][0] % 2 == 0 else cands[1][0]
        assert o.encode16(float(v), 1) == want, (v, hex(want))
    assert [o.encode16(float(t), 1) for t in ties] == [0x3F80, 0x3F82, 0xBF82]


def pin_mixed_step_equals_float32_step(o, tmp):
    """Gradients exactly representable in 16 bits give the float32 step bit
    for bit; the 16-bit weight copy is the rounding of the new weights."""
    rng = np.random.default_rng(16)
    n = 512
    g32 = rng.integers(-64, 65, n).astype(np.float32) / np.float32(256)
    g_bf = (g32.view(np.uint32) >> 16).astype(np.uint16)
    g_f16 = g32.astype(np.float16).view(np.uint16)
    for dt, g16 in ((1, g_bf), (2, g_f16)):
        a = [rng.normal(0, 0.02, n).astype(np.float32), np.zeros(n, np.float32),
             np.zeros(n, np.float32)]
        b = [x.copy() for x in a]
        _, n1, w_lp = o.adamw_clip_step_mixed(a[0], g16, dt, a[1], a[2], 1, 3e-3, 0.01, 1.0,
                                              0.5, w_lp_dtype=dt)
        _, n2 = o.adamw_clip_step_scaled(b[0], g32, b[1], b[2], 1, 3e-3, 0.01, 1.0, 0.5)
        assert n1 == n2
        for x, y in zip(a, b):
            assert x.tobytes() == y.tobytes()
        assert list(w_lp) == [o.encode16(float(x), dt) for x in a[0]]


# --- checkpoint format -----------------------------------------------------

def pin_ckpt_printed_sizes(o, tmp):
    """8 + 12 n bytes; the pages print 154 MB for 12.8M parameters and about
    1.44 GB for ~120M."""
    _, _, _ = read_golden("ckpt_sizes.txt")
    with open(os.path.join(GOLDEN, "ckpt_sizes.txt")) as f:
        rows = [l.split() for l in f if l.startswith("params")]
    for _, n, size, unit, digits in rows:
        scale = {"MB": 1e6, "GB": 1e9}[unit]
        got = o.ckpt_size(int(n))
        assert got == 8 + 12 * int(n)
        assert round(got / scale, int(digits)) == float(size), (n, got)
    assert o.ckpt_size(12_800_000) == 153_600_008


def pin_pack_layout(o, tmp):
    """Header = little-endian int32 step then int32 n; then w, m, v as
    contiguous little-endian float32 regions, in that order."""
    n = 5
    w = np.arange(1, 6, dtype=np.float32)
    m = -np.arange(1, 6, dtype=np.float32)
    v = np.arange(1, 6, dtype=np.float32) / 8
    img = o.pack(100, w, m, v)
    assert img.size == 8 + 12 * n
    b = img.tobytes()
    assert struct.unpack("<ii", b[:8]) == (100, n)
    floats = struct.unpack("<%df" % (3 * n), b[8:])
    assert list(floats[:n]) == list(w) and list(floats[n:2 * n]) == list(m)
    assert list(floats[2 * n:]) == list(v)


def pin_write_read_roundtrip(o, tmp):
    """The file is named step_%06d.bin, holds the pack image byte for byte,
    leaves no .tmp behind and reads back to identical arrays and step."""
    rng = np.random.default_rng(6)
    n = 1001
    w, m, v = (rng.standard_normal(n).astype(np.float32) for _ in range(3))
    path = o.ckpt_write(str(tmp), 100, w, m, v)
    assert os.path.basename(path) == "step_000100.bin"
    assert not os.path.exists(path + ".tmp")
    with open(path, "rb") as f:
        data = f.read()
    assert data == o.pack(100, w, m, v).tobytes()
    st, step, w2, m2, v2 = o.ckpt_read(path, n)
    assert st == 0 and step == 100
    assert w2.tobytes() == w.tobytes() and m2.tobytes() == m.tobytes()
    assert v2.tobytes() == v.tobytes()
    p2 = o.ckpt_write(str(tmp), 1234567, w, m, v)
    assert os.path.basename(p2) == "step_1234567.bin"


def pin_read_rejects_bad_files(o, tmp):
    """Refuse loudly ("Three failure modes"): truncated file, extra bytes,
    a parameter count that differs from the caller's, a negative header
    field, a file shorter than the header, a missing file."""
    n = 16
    z = np.zeros(n, np.float32)
    good = o.ckpt_write(str(tmp), 7, z + 1, z + 2, z + 3)
    data = open(good, "rb").read()

    def case(name, payload):
        p = os.path.join(str(tmp), name)
        with open(p, "wb") as f:
            f.write(payload)
        return o.ckpt_read(p, n)[0]

    assert case("trunc.bin", data[:-4]) == 4          # ESIZE
    assert case("extra.bin", data + b"\0") == 4       # ESIZE
    assert case("short.bin", data[:5]) == 4           # ESIZE
    assert case("other_n.bin", struct.pack("<ii", 7, n + 1) + data[8:]) == 5  # EMISMATCH
    assert case("neg_n.bin", struct.pack("<ii", 7, -1) + data[8:]) == 3       # EFORMAT
    assert case("neg_step.bin", struct.pack("<ii", -2, n) + data[8:]) == 3    # EFORMAT
    assert o.ckpt_read(os.path.join(str(tmp), "absent.bin"), n)[0] == 2      # EIO
    assert o.ckpt_read(good, n - 1)[0] == 5


def pin_float32_resume_bit_exact(o, tmp):
    """Saving m and v makes resume bit-equivalent: 3 float32 steps without a
    break equal 2 steps, write, read, 1 step ("Why save m & v"); resuming
    from the weights alone does not."""
    rng = np.random.default_rng(8)
    n = 333
    w0 = rng.normal(0, 0.02, n).astype(np.float32)
    gs = [rng.normal(0, 0.5, n).astype(np.float32) for _ in range(3)]

    def run(w, m, v, t0, steps):
        for k in steps:
            o.adamw_clip_step(w, gs[k], m, v, t0 + k + 1, 3e-3, 0.01, 1.0)

    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run(w, m, v, 0, range(3))
    w2, m2, v2 = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    run(w2, m2, v2, 0, range(2))
    path = o.ckpt_write(str(tmp), 2, w2, m2, v2)
    st, step, w3, m3, v3 = o.ckpt_read(path, n)
    assert st == 0 and step == 2
    o.adamw_clip_step(w3, gs[2], m3, v3, step + 1, 3e-3, 0.01, 1.0)
    assert w3.tobytes() == w.tobytes() and m3.tobytes() == m.tobytes()
    assert v3.tobytes() == v.tobytes()
    w4 = w3.copy()
    w4[:] = o.ckpt_read(path, n)[2]
    mz, vz = np.zeros(n, np.float32), np.zeros(n, np.float32)
    o.adamw_clip_step(w4, gs[2], mz, vz, 1, 3e-3, 0.01, 1.0)
    assert np.max(np.abs(w4.astype(np.float64) - w)) > 1e-4




# --- sharded checkpoint ------------------------------------------------------

def _shards(n_per, world, seed=12):
    rng = np.random.default_rng(seed)
    return [tuple(rng.standard_normal(n_per).astype(np.float32) for _ in range(3))
            for _ in range(world)]


def pin_sharded_manifest_schema(o, tmp):
    """The oracle's manifest has the page's keys, nesting, order and types,
    and equal 65,536-element shards start at R x 65,536 (golden example)."""
    from oracle import sharded
    with open(os.path.join(GOLDEN, "manifest_example.json")) as f:
        page = json.load(f)
    shards = _shards(65536, 4)
    d = sharded.save_sharded(str(tmp), 1234, shards, [0, 65536, 131072, 196608], 4521)
    with open(os.path.join(d, "manifest.json")) as f:
        ours = json.load(f)
    assert list(ours) == list(page)
    assert ours["schema_version"] == page["schema_version"] == 1
    assert (ours["world_size"], ours["step"]) == (page["world_size"], page["step"])
    for a, b in zip(ours["shards"], page["shards"]):
        assert list(a) == list(b)
        for k in ("rank", "path", "param_shard_offset", "param_shard_numel"):
            assert a[k] == b[k], k
        assert len(a["sha256"]) == 64


def pin_sharded_roundtrip_and_guards(o, tmp):
    """4 shard files + manifest, reloaded byte for byte ("Ship it"); a
    different world size, a dropped shard and a truncated or corrupted shard
    are refused ("Three failure modes")."""
    import shutil

    from oracle import sharded
    shards = _shards(1000, 4)
    d = sharded.save_sharded(str(tmp), 7, shards, [0, 1000, 2000, 3000])
    assert sorted(os.listdir(d)) == ["manifest.json", "rank0.bin", "rank1.bin", "rank2.bin",
                                     "rank3.bin"]
    step, got = sharded.load_sharded(d, 4)
    assert step == 7
    for (off, k, w, m, v), (w0, m0, v0), r in zip(got, shards, range(4)):
        assert (off, k) == (1000 * r, 1000)
        assert w.tobytes() == w0.tobytes() and m.tobytes() == m0.tobytes()
        assert v.tobytes() == v0.tobytes()

    def refused(kind, mutate):
        bad = os.path.join(str(tmp), f"bad_{kind}_{len(os.listdir(str(tmp)))}")
        shutil.copytree(d, bad)
        world = mutate(bad)
        try:
            sharded.load_sharded(bad, world)
        except sharded.ShardedCheckpointError as e:
            assert e.kind == kind, (e.kind, kind)
            return
        raise AssertionError(f"{kind} not refused")

    refused("world_size", lambda b: 2)

    def drop_shard(b):
        p = os.path.join(b, "manifest.json")
        man = json.load(open(p))
        man["shards"] = man["shards"][:3]
        json.dump(man, open(p, "w"))
        return 4
    refused("shard_count", drop_shard)

    def truncate(b):
        p = os.path.join(b, "rank2.bin")
        data = open(p, "rb").read()
        open(p, "wb").write(data[:-12])
        return 4
    refused("partial_write", truncate)

    def flip(b):
        p = os.path.join(b, "rank1.bin")
        data = bytearray(open(p, "rb").read())
        data[100] ^= 1
        open(p, "wb").write(bytes(data))
        return 4
    refused("partial_write", flip)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
