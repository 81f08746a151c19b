"""Pins of the fp64 oracle to facts fixed outside it.

Each check takes a loaded oracle build and raises AssertionError when the
oracle disagrees with a closed form, a hand-derived golden value, a library
routine on a special case, or an invariant the pages state. test_oracle_pins
runs them all against the real oracle; test_oracle_mutations shows that every
planted mistake in the oracle fails at least one of them.

Passages (page title, section):
  * vllm-omni commits, score-space join commit: cache and new token scored
    separately, scores concatenated; ring of window-1 slots, order-free, masked
    unwritten slots; a test pins ring and roll to the same output on a shared
    history.
  * vllm-omni commits, Spark model commit: per-layer-type RoPE; head-wise
    sigmoid output gate.
  * vllm-omni commits, talker export commit: GQA by reshaping the query.
  * TensorFold PR #608: verify windows under tree masks; drafted == serial;
    concurrent == alone.
"""
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NAN = 0x7FC0


def bf16(x):
    """bf16 bits of values exactly representable in bf16 (test constants)."""
    a = torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return a.view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(x):
    return float(np.float32(x))


def sigmoid(g):
    return 1.0 / (1.0 + math.exp(-g))


def close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


def _parse_pow2(expr: str) -> float:
    """Evaluate the small arithmetic used in the golden file (powers of 2)."""
    return float(eval(expr.replace("^", "**"), {"__builtins__": {}}, {}))


# ------------------------------------------------------------------ numbers

def pin_bf16_rounding_golden(o):
    cases = json.load(open(os.path.join(GOLDEN, "bf16_rounding.json")))["cases"]
    for c in cases:
        x = _parse_pow2(c["x"])
        got = o.bf16_round(x)
        assert got == int(c["bits"], 16), f"bf16({c['x']}) = {got:#06x}, want {c['bits']} ({c['why']})"


def pin_bf16_rounding_matches_fp32_conversion(o):
    """For values exactly representable in fp32, one-step rounding from fp64
    equals the library's fp32 -> bf16 round-to-nearest-even conversion."""
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4000, generator=g) * torch.exp(torch.randn(4000, generator=g) * 8)
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.bf16_round(float(v)) for v in x.numpy()], np.uint16)
    assert np.array_equal(got, want), f"{np.sum(got != want)} of 4000 differ"


# ------------------------------------------------------------------ RoPE

def _golden_sym(expr: str) -> float:
    env = {"c": lambda a: math.cos(a), "s": lambda a: math.sin(a)}
    return float(eval(expr, {"__builtins__": {}}, env))


# The oracle's cos and sin are fp32 values within COS_SIN_TOL of the cosine and
# sine of the exact angle for |pos| <= 2^21 (fixed-point phase, fp32 Taylor
# polynomial on [-pi/4, pi/4]); a pair rotated by them is within twice that
# times the pair's magnitude.
COS_SIN_TOL = 1.5e-7


def pin_rope_cos_sin_accuracy(o):
    """cos/sin of pos * theta^(-2i/r) against 40-digit values, over both layer
    types, every quadrant, angles at quarter turns and negative positions."""
    mpmath = __import__("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(3)
    positions = list(range(0, 33)) + [-1, -77, 511, 4095, 8192, 1 << 20, (1 << 21) - 1]
    positions += [int(p) for p in rng.integers(0, 1 << 21, 24)]
    for r, theta in ((256, 1e4), (64, 5e6), (2, 1.0)):
        for pos in positions:
            for i in range(r // 2):
                c, s = o.rope_cos_sin(r, theta, pos, i)
                assert c == f32(c) and s == f32(s), "cos/sin are fp32 values"
                a = mpmath.mpf(pos) * mpmath.power(mpmath.mpf(theta), mpmath.mpf(-2 * i) / r)
                close([c, s], [float(mpmath.cos(a)), float(mpmath.sin(a))], COS_SIN_TOL,
                      f"cos/sin r={r} theta={theta} pos={pos} i={i}")
    # r = 2, theta irrelevant (frequency 1): angles 0, 1, ..., and near k pi/4
    for k in range(-9, 10):
        pos = round(k * math.pi / 4)
        c, s = o.rope_cos_sin(2, 1.0, pos, 0)
        close([c, s], [math.cos(pos), math.sin(pos)], COS_SIN_TOL, f"pos {pos}")


def pin_rope_golden(o):
    cases = json.load(open(os.path.join(GOLDEN, "rope_cases.json")))["cases"]
    for c in cases:
        D = c["D"]
        x = np.zeros(D, np.float32)
        for k, val in c["x"].items():
            x[int(k)] = val
        want = x.astype(np.float64)
        for k in c["x"]:
            if k not in c["expect"]:
                want[int(k)] = 0.0
        for k, e in c["expect"].items():
            want[int(k)] = _golden_sym(e)
        got = o.rope_f64(bf16(x), c["r"], c["theta"], c["pos"])
        close(got, want, 2 * COS_SIN_TOL * max(1.0, np.abs(x).max()), f"rope golden ({c['why']})")


def pin_rope_r2_is_complex_multiplication(o):
    """r = 2: the single pair turns like (x0 + i x1) * exp(i pos)."""
    x = rand_bf16(2, 11)
    xv = bf16_val(x)
    for pos in (1, 2, 7, 100, 4097, 1 << 20):
        z = complex(xv[0], xv[1]) * complex(math.cos(pos), math.sin(pos))
        got = o.rope_f64(x, 2, 12345.0, pos)
        close(got, [z.real, z.imag], 2 * COS_SIN_TOL * abs(z), f"r=2 pos={pos}")


def pin_rope_norm_and_relative_position(o):
    """Rotation keeps the norm, and <R(m) q, R(n) k> depends only on m - n
    (up to the fp32 rounding of cos and sin)."""
    q = rand_bf16(64, 12)
    k = rand_bf16(64, 13)
    nq = np.linalg.norm(bf16_val(q))
    for r, theta in ((64, 1e4), (16, 5e6)):
        for m in (0, 5, 300, 70000):
            close([np.linalg.norm(o.rope_f64(q, r, theta, m))], [nq], 1e-5 * nq, "norm")
        base = np.dot(o.rope_f64(q, r, theta, 40), o.rope_f64(k, r, theta, 10))
        for shift in (1, 17, 1000):
            other = np.dot(o.rope_f64(q, r, theta, 40 + shift), o.rope_f64(k, r, theta, 10 + shift))
            close([other], [base], 1e-4, f"relative position shift {shift}")


def _bf16_of_fraction(v):
    """bf16 bits of the Fraction v rounded to nearest, ties to even (8
    significant bits, exponent range of fp32, subnormal grid 2^-133)."""
    from fractions import Fraction
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    spacing = Fraction(2) ** (max(e, -126) - 7)
    units = a / spacing
    k = units.numerator // units.denominator
    rem = units - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    val = k * spacing
    if val >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = int(np.array([float(val)], np.float32).view(np.uint32)[0]) >> 16
    return sign | bits


def _f32_bits_value(bits):
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def pin_bf16_dot2_exact_against_fractions(o):
    """The K entry's rounding: the bf16 nearest to the exact x*c + y*s, checked
    against rational arithmetic on random operands of every scale, products
    that land on rounding ties, and tiny second products."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    cases = []
    for _ in range(3000):
        xb = int(rng.integers(0, 1 << 16)) & 0xFFFF
        yb = int(rng.integers(0, 1 << 16)) & 0xFFFF
        if (xb & 0x7F80) == 0x7F80 or (yb & 0x7F80) == 0x7F80:
            continue
        cb = int(rng.integers(0, 1 << 32))
        sb = int(rng.integers(0, 1 << 32))
        if (cb & 0x7F800000) == 0x7F800000 or (sb & 0x7F800000) == 0x7F800000:
            continue
        cases.append((xb, cb, yb, sb))
    for _ in range(2000):  # ordinary magnitudes, like rotated N(0,1) keys
        x = float(rng.standard_normal())
        y = float(rng.standard_normal())
        ang = float(rng.uniform(-7, 7))
        xb = int(np.array([x], np.float32).view(np.uint32)[0]) >> 16
        yb = int(np.array([y], np.float32).view(np.uint32)[0]) >> 16
        cb = int(np.array([math.cos(ang)], np.float32).view(np.uint32)[0])
        sb = int(np.array([math.sin(ang)], np.float32).view(np.uint32)[0])
        cases.append((xb, cb, yb, sb))
    # x*c on a bf16 tie, y*s far below it (on either side), or exactly zero
    for k in range(1, 127, 2):
        c = 1.0 + k * 2.0 ** -8
        cb = int(np.array([c], np.float32).view(np.uint32)[0])
        for yb in (67 << 7, (67 << 7) | 0x8000, 0):
            cases.append((0x3F80, cb, yb, 0x3F800000))
    for xb, cb, yb, sb in cases:
        c, s = _f32_bits_value(cb), _f32_bits_value(sb)
        want = (_bf16_of_fraction(Fraction(bf16_val(xb)[()]) * Fraction(c) + Fraction(bf16_val(yb)[()]) * Fraction(s))
                if not (c == 0 and s == 0) else None)
        got = o.bf16_dot2(xb, c, yb, s)
        if want is None:
            continue
        if want == 0 and got == 0x8000:
            got = 0  # the sign of an exact zero is IEEE's; only the value is pinned here
        assert got == want, f"bf16({bf16_val(xb)[()]}*{c} + {bf16_val(yb)[()]}*{s}) = {got:#06x}, want {want:#06x}"


def pin_rope_entry_matches_rotation(o):
    """The K entry is the rotation of the key rounded to bf16: away from bf16
    rounding ties it equals the fp64 rotation rounded once."""
    for seed, (r, theta, pos) in enumerate(((256, 1e4, 300), (64, 5e6, 4096), (128, 1e6, 77777))):
        x = rand_bf16(256, 40 + seed)
        ent = o.rope_bf16(x, r, theta, pos)
        rot = o.rope_f64(x, r, theta, pos)
        want = np.array([o.bf16_round(v) for v in rot], np.uint16)
        assert np.array_equal(ent, want), f"r={r}: {np.sum(ent != want)} entries differ"


def _mpf_fraction(x):
    """The exact rational value of an mpmath number (a binary float)."""
    from fractions import Fraction
    sign, man, exp, _ = x._mpf_
    f = Fraction(int(man)) * (Fraction(2) ** exp if exp >= 0 else Fraction(1, 2 ** (-exp)))
    return -f if sign else f


def _bf16_midpoint_distance(v):
    """|v| minus its nearest bf16 rounding boundary (a midpoint between two
    neighbouring bf16 values), as a float; v is a Fraction."""
    from fractions import Fraction
    a = abs(v)
    if a == 0:
        return float("inf")
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    spacing = Fraction(2) ** (max(e, -126) - 7)
    units = a / spacing
    frac = units - units.numerator // units.denominator
    return float(abs(frac - Fraction(1, 2)) * spacing)


def pin_rope_entry_is_rounded_exact_rotation(o):
    """The K entry against its plain definition: the bf16 nearest (ties to
    even) to the exact rotation x cos(a) - y sin(a), y cos(a) + x sin(a) with
    a = pos * theta^(-2i/r), cos and sin to 40 digits (mpmath), the rounding in
    rational arithmetic. The oracle turns by fp32 cos/sin within COS_SIN_TOL of
    the exact ones, so an element may differ only where the exact value lies
    within (|x| + |y|) * COS_SIN_TOL of a bf16 rounding boundary; those
    exceptions are counted and must stay rare. Covers both layer types and the
    paged batch's RoPE (r = 256, theta 1e4; r = 64, theta 5e6; r = 128, theta
    1e6), positions up to 2^21 - 1 and negative ones; dims >= r pass through."""
    mpmath = __import__("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(17)
    D = 256
    positions = [0, 1, 2, 3, 7, 299, 300, 511, 4095, 4096, 65535, -5, (1 << 21) - 1]
    positions += [int(p) for p in rng.integers(0, 1 << 21, 12)]
    checked = near = 0
    for cfg, (r, theta) in enumerate(((256, 1e4), (64, 5e6), (128, 1e6))):
        half = r // 2
        inv = [mpmath.power(mpmath.mpf(theta), mpmath.mpf(-2 * i) / r) for i in range(half)]
        for n, pos in enumerate(positions):
            x = rand_bf16(D, 1000 + 100 * cfg + n)
            xv = bf16_val(x)
            ent = o.rope_bf16(x, r, theta, pos)
            assert np.array_equal(ent[r:], x[r:]), f"r={r}: dims past r must pass through"
            for i in range(half):
                a = mpmath.mpf(pos) * inv[i]
                c, s = mpmath.cos(a), mpmath.sin(a)
                px, py = mpmath.mpf(float(xv[i])), mpmath.mpf(float(xv[i + half]))
                bound = (abs(float(xv[i])) + abs(float(xv[i + half]))) * COS_SIN_TOL
                for d, exact in ((i, px * c - py * s), (i + half, py * c + px * s)):
                    v = _mpf_fraction(exact)
                    checked += 1
                    if _bf16_midpoint_distance(v) <= bound:
                        near += 1  # within the cos/sin error of a rounding boundary
                        continue
                    want = _bf16_of_fraction(v)
                    got = int(ent[d])
                    if want == 0 and got == 0x8000:
                        got = 0
                    assert got == want, (f"r={r} theta={theta} pos={pos} dim {d}: entry {got:#06x}, "
                                         f"exact rotation rounds to {want:#06x}")
    assert near <= max(3, checked // 200), f"{near} of {checked} elements near a rounding boundary"


def pin_append_ring_places_entries(o):
    """Bulk append into rings, against a hand-derived slot layout. R = 5 slots,
    three ring rows, call rows mapped to ring rows 2 and 0. Call row 0 writes
    tokens 0..3 at indices 3..6, i.e. slots 3, 4, 0, 1 of ring row 2; call row 1
    writes tokens 0..4 at indices 7..11, i.e. slots 2, 3, 4, 0, 1 of ring row 0
    (a whole ring, wrapping). Keys are turned at start_pos + t (or copied when
    rotate is off); every other slot keeps its NaN."""
    Hkv, D, R, n_rows = 2, 8, 5, 3
    Kr = np.full((n_rows, Hkv, R, D), NAN, np.uint16)
    Vr = Kr.copy()
    k = rand_bf16((2, 5, Hkv, D), 950)
    v = rand_bf16((2, 5, Hkv, D), 951)
    where = {(2, 3): (0, 0), (2, 4): (0, 1), (2, 0): (0, 2), (2, 1): (0, 3),
             (0, 2): (1, 0), (0, 3): (1, 1), (0, 4): (1, 2), (0, 0): (1, 3), (0, 1): (1, 4)}
    start_pos = [10, 0]
    for rotate in (True, False):
        Ko, Vo = o.append_ring(Kr, Vr, [3, 7], start_pos, [4, 5], k, v, 8, 1e4, rotate=rotate,
                               stream_rows=[2, 0])
        for row in range(n_rows):
            for slot in range(R):
                if (row, slot) not in where:
                    assert np.all(Ko[row, :, slot] == NAN) and np.all(Vo[row, :, slot] == NAN), \
                        f"slot ({row}, {slot}) was written"
                    continue
                b, t = where[(row, slot)]
                for j in range(Hkv):
                    want_k = o.rope_bf16(k[b, t, j], 8, 1e4, start_pos[b] + t) if rotate else k[b, t, j]
                    assert np.array_equal(Ko[row, j, slot], want_k), f"K at ({row}, {slot}) rotate={rotate}"
                    assert np.array_equal(Vo[row, j, slot], v[b, t, j]), f"V at ({row}, {slot})"


def pin_rope_entry_identity(o):
    """At position 0, and with no rotary dims, the K entry is the key itself."""
    x = rand_bf16(256, 14)
    assert np.array_equal(o.rope_bf16(x, 256, 1e4, 0), x)
    assert np.array_equal(o.rope_bf16(x, 0, 1e4, 999), x)


# ------------------------------------------------------------------ decode helpers

def ring_decode(o, K, V, head, count, q, kn, vn, pos, r=0, theta=1e4, gate=None):
    """K, V: [R, Hkv, D] float data for one stream, laid out per slot."""
    Kb = bf16(K).transpose(1, 0, 2)[None].copy()
    Vb = bf16(V).transpose(1, 0, 2)[None].copy()
    out, ke, ve = o.decode_ring(Kb, Vb, [head], [count], bf16(q)[None], bf16(kn)[None],
                                bf16(vn)[None], [pos], r, theta,
                                gate=None if gate is None else bf16(gate)[None])
    return out[0], ke[0], ve[0]


def _nan_ring(R, Hkv, D):
    K = np.full((R, Hkv, D), np.nan, np.float32)
    V = np.full((R, Hkv, D), np.nan, np.float32)
    return K, V


# ------------------------------------------------------------------ closed forms

def pin_empty_cache_is_gated_v_new(o):
    """No cached token: the softmax has one entry, out = sigmoid(g) * v_new."""
    D, Hq, Hkv, R = 8, 4, 2, 5
    K, V = _nan_ring(R, Hkv, D)
    q = bf16_val(rand_bf16((Hq, D), 21)).astype(np.float32)
    kn = bf16_val(rand_bf16((Hkv, D), 22)).astype(np.float32)
    vn = bf16_val(rand_bf16((Hkv, D), 23)).astype(np.float32)
    g = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    out, _, _ = ring_decode(o, K, V, 3, 0, q, kn, vn, 17, r=8, theta=1e4, gate=g)
    want = np.stack([sigmoid(float(g[h])) * vn[h // 2].astype(np.float64) for h in range(Hq)])
    close(out, want, 1e-15, "empty cache")


def pin_two_keys_logistic(o):
    """One cached key: the two-way softmax is the logistic function of the score
    difference. q = a e0, cached key e0, new key 0, position 0 (no turn):
    s_cache = a / sqrt(D), s_new = 0."""
    for D in (4, 16):
        Hq = Hkv = 1
        R = 3
        K, V = _nan_ring(R, Hkv, D)
        K[1, 0] = 0.0
        K[1, 0, 0] = 1.0
        V[1, 0] = bf16_val(rand_bf16(D, 31 + D))
        vn = bf16_val(rand_bf16((1, D), 41 + D)).astype(np.float32)
        a = 3.0
        q = np.zeros((Hq, D), np.float32)
        q[0, 0] = a
        kn = np.zeros((Hkv, D), np.float32)
        out, _, _ = ring_decode(o, K, V, 2, 1, q, kn, vn, 0, r=D)
        p1 = 1.0 / (1.0 + math.exp(-a / math.sqrt(D)))
        want = p1 * V[1, 0].astype(np.float64) + (1 - p1) * vn[0].astype(np.float64)
        close(out[0], want, 1e-14, f"two-key logistic D={D}")


def pin_uniform_weights_when_q_is_zero(o):
    """q = 0 gives every key the same score: out = mean of the attended values."""
    D, Hq, Hkv, R = 8, 2, 1, 9
    K, V = _nan_ring(R, Hkv, D)
    head, count = 4, 6
    slots = [(head - 1 - i) % R for i in range(count)]
    for s in slots:
        K[s] = bf16_val(rand_bf16((Hkv, D), 50 + s))
        V[s] = bf16_val(rand_bf16((Hkv, D), 60 + s))
    vn = bf16_val(rand_bf16((Hkv, D), 70)).astype(np.float32)
    kn = bf16_val(rand_bf16((Hkv, D), 71)).astype(np.float32)
    out, _, _ = ring_decode(o, K, V, head, count, np.zeros((Hq, D), np.float32), kn, vn, 33, r=8)
    want = (sum(V[s, 0].astype(np.float64) for s in slots) + vn[0]) / (count + 1)
    close(out, np.stack([want, want]), 1e-15, "q = 0 mean")


def pin_ring_valid_slots_onehot(o):
    """A ring's valid slots are the `count` slots before `head` (cyclically).
    With q = 0 and V[slot] = e_slot, the output spells out the set that was
    attended; unwritten slots hold NaN. Hand-derived: R = 5, head = 1, count = 3
    attends slots {0, 4, 3}; head = 0, count = 5 attends all five."""
    D, R = 8, 5
    for head, count, want_slots in ((1, 3, [0, 4, 3]), (0, 5, [0, 1, 2, 3, 4]), (3, 1, [2])):
        K, V = _nan_ring(R, 1, D)
        for s in want_slots:
            K[s, 0] = 0.0
            V[s, 0] = 0.0
            V[s, 0, s] = 1.0
        vn = np.zeros((1, D), np.float32)
        vn[0, 7] = 1.0
        out, _, _ = ring_decode(o, K, V, head, count, np.zeros((1, D), np.float32),
                                np.zeros((1, D), np.float32), vn, 9, r=8)
        want = np.zeros(D)
        want[want_slots] = 1.0 / (count + 1)
        want[7] = 1.0 / (count + 1)
        close(out[0], want, 1e-15, f"ring slots head={head} count={count}")


def pin_paged_traversal_onehot(o):
    """Token t of a stream lives at offset t % P of page block_table[t // P].
    With q = 0 and V = e_t at token t, the output is the uniform mix of the
    first seq_len tokens and the new one; the free slot holds NaN."""
    D, P, Hkv = 8, 2, 1
    bt = np.array([[2, 0, 1]], np.int32)
    n = 5
    Kp = np.full((3, Hkv, P, D), np.nan, np.float32)
    Vp = np.full((3, Hkv, P, D), np.nan, np.float32)
    for t in range(n):
        pg, off = bt[0, t // P], t % P
        Kp[pg, 0, off] = 0.0
        Vp[pg, 0, off] = 0.0
        Vp[pg, 0, off, t] = 1.0
    vn = np.zeros((1, 1, D), np.float32)
    vn[0, 0, 7] = 1.0
    out, _, _ = o.decode_paged(bf16(Kp), bf16(Vp), bt, [n], bf16(np.zeros((1, 1, D))),
                               bf16(np.zeros((1, 1, D))), bf16(vn), [n], 8, 1e4)
    want = np.zeros(D)
    want[:n] = 1.0 / (n + 1)
    want[7] = 1.0 / (n + 1)
    close(out[0, 0], want, 1e-15, "paged traversal")


def pin_gqa_contiguous_groups(o):
    """Query head h reads KV head h // G (the query is reshaped into groups)."""
    D, Hq, Hkv, R = 4, 4, 2, 3
    K = np.zeros((R, Hkv, D), np.float32)
    V = np.zeros((R, Hkv, D), np.float32)
    V[:, 0] = 1.0
    V[:, 1] = -1.0
    vn = np.array([[1.0] * D, [-1.0] * D], np.float32)
    q = bf16_val(rand_bf16((Hq, D), 80)).astype(np.float32)
    out, _, _ = ring_decode(o, K, V, 0, 3, q, np.zeros((Hkv, D), np.float32), vn, 4, r=4)
    close(out, np.array([[1.0] * D, [1.0] * D, [-1.0] * D, [-1.0] * D]), 1e-15, "gqa map")


def pin_gate_scales_by_sigmoid(o):
    """out_gated = sigmoid(g) * out_ungated; g = 0 halves the output."""
    D, Hq, Hkv, R = 8, 2, 1, 6
    K = bf16_val(rand_bf16((R, Hkv, D), 90)).astype(np.float32)
    V = bf16_val(rand_bf16((R, Hkv, D), 91)).astype(np.float32)
    q = bf16_val(rand_bf16((Hq, D), 92)).astype(np.float32)
    kn = bf16_val(rand_bf16((Hkv, D), 93)).astype(np.float32)
    vn = bf16_val(rand_bf16((Hkv, D), 94)).astype(np.float32)
    base, _, _ = ring_decode(o, K, V, 2, 6, q, kn, vn, 20, r=8)
    g = np.array([0.0, 2.0], np.float32)
    gated, _, _ = ring_decode(o, K, V, 2, 6, q, kn, vn, 20, r=8, gate=g)
    close(gated, base * np.array([[0.5], [sigmoid(2.0)]]), 1e-15, "gate")


# ------------------------------------------------------------------ invariants

def pin_score_space_join_equals_key_concat(o):
    """Scoring the cache and the new token separately and concatenating the
    score vectors equals attention over the concatenated key matrix."""
    B, Hq, Hkv, D, R = 3, 8, 2, 32, 13
    counts = [13, 7, 0]
    heads = [5, 12, 3]
    hist_k = rand_bf16((B, Hkv, R, D), 100)
    hist_v = rand_bf16((B, Hkv, R, D), 101)
    Kr = np.full((B, Hkv, R, D), NAN, np.uint16)
    Vr = np.full((B, Hkv, R, D), NAN, np.uint16)
    for b in range(B):
        for t in range(counts[b]):  # oldest first: token t sits count - t slots before head
            slot = (heads[b] - counts[b] + t) % R
            Kr[b, :, slot] = hist_k[b, :, t]
            Vr[b, :, slot] = hist_v[b, :, t]
    q = rand_bf16((B, Hq, D), 102)
    kn = rand_bf16((B, Hkv, D), 103)
    vn = rand_bf16((B, Hkv, D), 104)
    g = rand_bf16((B, Hq), 105)
    pos = [40, 41, 0]
    join, _, _ = o.decode_ring(Kr, Vr, heads, counts, q, kn, vn, pos, 32, 1e4, gate=g)
    cat = o.decode_concat(hist_k, hist_v, counts, q, kn, vn, pos, 32, 1e4, gate=g)
    close(join, cat, 1e-12, "join vs concat")


def pin_ring_equals_roll_over_history(o):
    """Ring (write at head, no reordering) and roll (append, drop the oldest,
    concatenate keys) give the same output at every step of a shared history
    longer than the ring."""
    Hq, Hkv, D, R = 4, 2, 16, 7
    r, theta = 16, 1e4
    Kr = np.full((1, Hkv, R, D), NAN, np.uint16)
    Vr = np.full((1, Hkv, R, D), NAN, np.uint16)
    roll_k, roll_v = [], []  # chronological lists of [Hkv, D] entries
    head, count = 0, 0
    for step in range(20):
        q = rand_bf16((1, Hq, D), 200 + step)
        kn = rand_bf16((1, Hkv, D), 300 + step)
        vn = rand_bf16((1, Hkv, D), 400 + step)
        out_ring, ke, ve = o.decode_ring(Kr, Vr, [head], [count], q, kn, vn, [step], r, theta)
        kc = np.full((1, Hkv, R, D), NAN, np.uint16)
        vc = np.full((1, Hkv, R, D), NAN, np.uint16)
        for t, (a, b_) in enumerate(zip(roll_k, roll_v)):
            kc[0, :, t] = a
            vc[0, :, t] = b_
        out_roll = o.decode_concat(kc, vc, [len(roll_k)], q, kn, vn, [step], r, theta)
        close(out_ring, out_roll, 1e-12, f"ring vs roll step {step}")
        # ring: drop the entry into slot `head`; roll: append, slice off the oldest
        Kr[0, :, head] = ke[0]
        Vr[0, :, head] = ve[0]
        head = (head + 1) % R
        count = min(count + 1, R)
        roll_k.append(ke[0])
        roll_v.append(ve[0])
        if len(roll_k) > R:
            roll_k.pop(0)
            roll_v.pop(0)


def pin_slot_order_irrelevant_and_masked_nan(o):
    """Permuting the physical pages of a paged cache, or adding NaN-filled
    unused pages, changes nothing."""
    B, Hq, Hkv, D, P = 2, 4, 2, 16, 4
    lens = [9, 14]
    toks_k = rand_bf16((B, 16, Hkv, D), 500)
    toks_v = rand_bf16((B, 16, Hkv, D), 501)
    q, kn, vn = rand_bf16((B, Hq, D), 502), rand_bf16((B, Hkv, D), 503), rand_bf16((B, Hkv, D), 504)
    outs = []
    for perm_seed in (None, 1, 2):
        n_pages = 12
        phys = np.arange(n_pages) if perm_seed is None else \
            np.random.default_rng(perm_seed).permutation(n_pages)
        Kp = np.full((n_pages, Hkv, P, D), NAN, np.uint16)
        Vp = np.full((n_pages, Hkv, P, D), NAN, np.uint16)
        bt = np.full((B, 4), -1, np.int32)
        nxt = 0
        for b in range(B):
            for pg in range((lens[b] + P - 1) // P):
                bt[b, pg] = phys[nxt]
                nxt += 1
            for t in range(lens[b]):
                Kp[bt[b, t // P], :, t % P] = toks_k[b, t]
                Vp[bt[b, t // P], :, t % P] = toks_v[b, t]
        out, _, _ = o.decode_paged(Kp, Vp, bt, lens, q, kn, vn, lens, 16, 1e6)
        outs.append(out)
    close(outs[1], outs[0], 1e-15, "page permutation 1")
    close(outs[2], outs[0], 1e-15, "page permutation 2")


def pin_batch_equals_alone(o):
    """A stream's result does not depend on the other streams in the call."""
    B, Hq, Hkv, D, R = 4, 4, 2, 16, 9
    Kr = rand_bf16((B, Hkv, R, D), 600)
    Vr = rand_bf16((B, Hkv, R, D), 601)
    q, kn, vn = rand_bf16((B, Hq, D), 602), rand_bf16((B, Hkv, D), 603), rand_bf16((B, Hkv, D), 604)
    g = rand_bf16((B, Hq), 605)
    heads, counts, pos = [0, 3, 8, 5], [9, 4, 2, 0], [11, 4, 2, 0]
    full, ke, ve = o.decode_ring(Kr, Vr, heads, counts, q, kn, vn, pos, 16, 1e4, gate=g)
    for b in range(B):
        one, k1, v1 = o.decode_ring(Kr[b:b + 1], Vr[b:b + 1], heads[b:b + 1], counts[b:b + 1],
                                    q[b:b + 1], kn[b:b + 1], vn[b:b + 1], pos[b:b + 1], 16, 1e4,
                                    gate=g[b:b + 1])
        assert np.array_equal(one[0], full[b]) and np.array_equal(k1[0], ke[b])


# ------------------------------------------------------------------ verify

def _prefix_pool(S, Hkv, D, P, lens, room, seed):
    pages = [(n + room + P - 1) // P for n in lens]
    n_pages = sum(pages) + 1
    phys = np.random.default_rng(seed).permutation(n_pages)
    Kp = np.full((n_pages, Hkv, P, D), NAN, np.uint16)
    Vp = np.full((n_pages, Hkv, P, D), NAN, np.uint16)
    bt = np.full((S, max(pages)), -1, np.int32)
    nxt = 0
    for s in range(S):
        bt[s, :pages[s]] = phys[nxt:nxt + pages[s]]
        nxt += pages[s]
        kk = rand_bf16((lens[s], Hkv, D), seed + 10 + s)
        vv = rand_bf16((lens[s], Hkv, D), seed + 40 + s)
        for t in range(lens[s]):
            Kp[bt[s, t // P], :, t % P] = kk[t]
            Vp[bt[s, t // P], :, t % P] = vv[t]
    return Kp, Vp, bt


def pin_verify_row_equals_decode_of_its_path(o):
    """Each verify row equals a plain decode of that row's token after its
    root-to-parent path has been appended to the prefix at positions
    prefix_len + depth (drafted == serial)."""
    S, T, Hq, Hkv, D, P = 2, 8, 6, 2, 16, 4
    r, theta = 8, 5e6
    lens = [10, 5]
    parent = np.array([[-1, 0, 0, 1, 3, 2, 4, -1], [-1, 0, 1, 2, 3, 4, 5, 6]], np.int32)
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, lens, T + 1, 700)
    q = rand_bf16((S, T, Hq, D), 701)
    k = rand_bf16((S, T, Hkv, D), 702)
    v = rand_bf16((S, T, Hkv, D), 703)
    g = rand_bf16((S, T, Hq), 704)
    out, ke = o.verify(Kp, Vp, bt, lens, q, k, v, parent, r, theta, gate=g)
    for s in range(S):
        for i in range(T):
            path = []
            a = parent[s, i]
            while a >= 0:
                path.append(a)
                a = parent[s, a]
            path.reverse()  # root first; node path[d] has depth d
            Kd, Vd = Kp.copy(), Vp.copy()
            for d, a in enumerate(path):
                t = lens[s] + d
                Kd[bt[s, t // P], :, t % P] = [o.rope_bf16(k[s, a, j], r, theta, t) for j in range(Hkv)]
                Vd[bt[s, t // P], :, t % P] = v[s, a]
            n = lens[s] + len(path)
            dec, kent, _ = o.decode_paged(Kd, Vd, bt[s:s + 1], [n], q[s, i][None], k[s, i][None],
                                          v[s, i][None], [n], r, theta, gate=g[s, i][None])
            close(out[s, i], dec[0], 1e-12, f"verify row {s},{i}")
            assert np.array_equal(ke[s, i], kent[0]), "window entry differs from the decode entry"


def pin_verify_chain_equals_sequential_decodes(o):
    """A chain tree is T serial decode steps, each appending its entry."""
    S, T, Hq, Hkv, D, P = 1, 6, 4, 2, 16, 4
    r, theta = 16, 1e4
    lens = [7]
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, lens, T + 1, 800)
    q = rand_bf16((S, T, Hq, D), 801)
    k = rand_bf16((S, T, Hkv, D), 802)
    v = rand_bf16((S, T, Hkv, D), 803)
    parent = np.arange(-1, T - 1, dtype=np.int32)[None]
    out, _ = o.verify(Kp, Vp, bt, lens, q, k, v, parent, r, theta)
    Kd, Vd = Kp.copy(), Vp.copy()
    n = lens[0]
    for i in range(T):
        dec, ke, ve = o.decode_paged(Kd, Vd, bt, [n], q[0, i][None], k[0, i][None], v[0, i][None],
                                     [n], r, theta)
        close(out[0, i], dec[0], 1e-12, f"chain step {i}")
        Kd[bt[0, n // P], :, n % P] = ke[0]
        Vd[bt[0, n // P], :, n % P] = ve[0]
        n += 1


def pin_append_places_rotated_entries(o):
    """Bulk append writes token t at cache index start + t, rotated at its own
    position; the one-hot layout shows where each token landed."""
    Hkv, D, P = 2, 8, 4
    bt = np.array([[3, 1, 0], [2, 4, -1]], np.int32)
    Kp = np.full((5, Hkv, P, D), NAN, np.uint16)
    Vp = Kp.copy()
    Tm = 5
    k = rand_bf16((2, Tm, Hkv, D), 900)
    v = rand_bf16((2, Tm, Hkv, D), 901)
    start_index, start_pos, count = [2, 1], [100, 7], [5, 4]
    Ko, Vo = o.append_paged(Kp, Vp, bt, start_index, start_pos, count, k, v, 8, 1e4, rotate=True)
    for b in range(2):
        for t in range(count[b]):
            i = start_index[b] + t
            for j in range(Hkv):
                assert np.array_equal(Ko[bt[b, i // P], j, i % P],
                                      o.rope_bf16(k[b, t, j], 8, 1e4, start_pos[b] + t))
                assert np.array_equal(Vo[bt[b, i // P], j, i % P], v[b, t, j])
    written = sum(count) * Hkv * D
    assert np.sum(Ko != NAN) == written and np.sum(Vo != NAN) == written


def _path(parent_row, i):
    """Root-first list of node i's ancestors (without i)."""
    out = []
    a = parent_row[i]
    while a >= 0:
        out.append(int(a))
        a = parent_row[a]
    return out[::-1]


def pin_ring_verify_row_equals_decode_of_its_path(o):
    """Verify over a ring (sliding) layer: each row equals the plain ring
    decode of its token after its root-to-parent path was appended to the ring
    (so the ring drops its oldest entries as it fills), for full and partly
    filled rings, and its window entry equals that decode's entry."""
    S, T, Hq, Hkv, D, R = 3, 7, 4, 2, 16, 9
    r, theta = 16, 1e4
    parent = np.array([[-1, 0, 1, 2, 3, 4, 5], [-1, 0, 0, 1, 3, 4, 2], [-1, 0, 1, 1, 0, 4, 5]], np.int32)
    Kr = rand_bf16((4, Hkv, R, D), 1601)
    Vr = rand_bf16((4, Hkv, R, D), 1602)
    rows = np.array([2, 0, 3], np.int32)
    head = np.array([4, 0, 8], np.int32)
    count = np.array([R, R - 2, 3], np.int32)
    pos = np.array([50, 7, 3], np.int32)
    q = rand_bf16((S, T, Hq, D), 1603)
    k = rand_bf16((S, T, Hkv, D), 1604)
    v = rand_bf16((S, T, Hkv, D), 1605)
    g = rand_bf16((S, T, Hq), 1606)
    out, ke = o.verify_ring(Kr, Vr, head, count, pos, q, k, v, parent, r, theta, gate=g, stream_rows=rows)
    for s in range(S):
        for i in range(T):
            path = _path(parent[s], i)
            d = len(path)
            Ks, Vs = Kr, Vr
            if d:
                kp = k[s, path][None]
                vp = v[s, path][None]
                Ks, Vs = o.append_ring(Kr, Vr, [head[s]], [pos[s]], [d], kp, vp, r, theta,
                                       stream_rows=rows[s:s + 1])
            dec, kent, _ = o.decode_ring(Ks, Vs, [(head[s] + d) % R], [min(count[s] + d, R)], q[s, i][None],
                                         k[s, i][None], v[s, i][None], [pos[s] + d], r, theta,
                                         gate=g[s, i][None], stream_rows=rows[s:s + 1])
            close(out[s, i], dec[0], 1e-12, f"ring verify row {s},{i}")
            assert np.array_equal(ke[s, i], kent[0]), "window entry differs from the decode entry"


def pin_commit_equals_serial_decode_write_backs(o):
    """Committing an accepted path writes the same cache as decoding the
    path's tokens one after another with write-back, on ring and paged
    layers; a list that is not a path from a root leaves its stream alone."""
    S, T, Hq, Hkv, D, R, P = 3, 6, 4, 2, 16, 7, 4
    r, theta = 16, 5e6
    parent = np.array([[-1, 0, 0, 1, 3, 2], [-1, 0, 1, 2, 3, 4], [-1, 0, 0, 2, 2, 4]], np.int32)
    accepted = np.full((S, T), -1, np.int32)
    acc = [[0, 2, 5], [0, 1, 2, 3, 4, 5], [0, 2, 4, 5]]
    for s, a in enumerate(acc):
        accepted[s, :len(a)] = a
    num = np.array([3, 6, 4], np.int32)
    k = rand_bf16((S, T, Hkv, D), 1701)
    v = rand_bf16((S, T, Hkv, D), 1702)
    q = rand_bf16((S, 1, Hq, D), 1703)
    # ring
    Kr = rand_bf16((S, Hkv, R, D), 1704)
    Vr = rand_bf16((S, Hkv, R, D), 1705)
    head = np.array([5, 0, 2], np.int32)
    pos = np.array([30, 0, 12], np.int32)
    Kc, Vc, rc = o.commit_ring(Kr, Vr, head, pos, k, v, parent, accepted, num, r, theta)
    assert rc == 0
    Ks, Vs = Kr.copy(), Vr.copy()
    for s in range(S):
        for d, a in enumerate(acc[s]):
            _, ke, ve = o.decode_ring(Ks, Vs, [(head[s] + d) % R], [R], q[s], k[s, a][None], v[s, a][None],
                                      [pos[s] + d], r, theta, stream_rows=[s])
            Ks[s, :, (head[s] + d) % R] = ke[0]
            Vs[s, :, (head[s] + d) % R] = ve[0]
    assert np.array_equal(Kc, Ks) and np.array_equal(Vc, Vs), "ring commit"
    # paged
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, [5, 0, 9], T + 1, 1706)
    seq = np.array([5, 0, 9], np.int32)
    Kc, Vc, rc = o.commit_paged(Kp, Vp, bt, seq, seq, k, v, parent, accepted, num, r, theta)
    assert rc == 0
    Ks, Vs = Kp.copy(), Vp.copy()
    for s in range(S):
        for d, a in enumerate(acc[s]):
            t = seq[s] + d
            _, ke, ve = o.decode_paged(Ks, Vs, bt[s:s + 1], [t], q[s], k[s, a][None], v[s, a][None], [t],
                                       r, theta)
            Ks[bt[s, t // P], :, t % P] = ke[0]
            Vs[bt[s, t // P], :, t % P] = ve[0]
    assert np.array_equal(Kc, Ks) and np.array_equal(Vc, Vs), "paged commit"
    # a broken path (node 3's parent is 2, not 1) leaves stream 2 alone
    bad = accepted.copy()
    bad[2, :3] = [0, 1, 3]
    Kc, Vc, rc = o.commit_ring(Kr, Vr, head, pos, k, v, parent, bad, np.array([0, 0, 3], np.int32), r, theta)
    assert rc == 3 and np.array_equal(Kc, Kr) and np.array_equal(Vc, Vr), "broken path"


def pin_prefill_one_token_is_decode_with_write_back(o):
    """A prefill of one token is one decode step that writes its entry back."""
    Hq, Hkv, D, R = 4, 2, 16, 6
    Kr = rand_bf16((2, Hkv, R, D), 1801)
    Vr = rand_bf16((2, Hkv, R, D), 1802)
    q = rand_bf16((1, 1, Hq, D), 1803)
    k = rand_bf16((1, 1, Hkv, D), 1804)
    v = rand_bf16((1, 1, Hkv, D), 1805)
    out, Kp, Vp = o.prefill_ring(Kr, Vr, [4], [5], [1], [77], q, k, v, 16, 1e4, stream_rows=[1])
    dec, ke, ve = o.decode_ring(Kr, Vr, [4], [5], q[0], k[0], v[0], [77], 16, 1e4, stream_rows=[1])
    close(out[0, 0], dec[0], 0.0, "one token")
    Kd, Vd = Kr.copy(), Vr.copy()
    Kd[1, :, 4], Vd[1, :, 4] = ke[0], ve[0]
    assert np.array_equal(Kp, Kd) and np.array_equal(Vp, Vd), "its entry written at the head"


def pin_prefill_in_two_parts_equals_one(o):
    """Prefilling tokens [0, a) and then [a, n) - the second call starting
    where the first one left the cache - equals prefilling [0, n): outputs and
    caches, ring (the ring wraps and drops its oldest entries) and paged."""
    S, Hq, Hkv, D, R, P, n = 2, 4, 2, 16, 7, 4, 9
    q = rand_bf16((S, n, Hq, D), 1901)
    k = rand_bf16((S, n, Hkv, D), 1902)
    v = rand_bf16((S, n, Hkv, D), 1903)
    cnt = np.array([n, 6], np.int32)
    Kr = rand_bf16((S, Hkv, R, D), 1904)
    Vr = rand_bf16((S, Hkv, R, D), 1905)
    head, rc_, pos = np.array([3, 0], np.int32), np.array([R, 2], np.int32), np.array([40, 2], np.int32)
    out, Kf, Vf = o.prefill_ring(Kr, Vr, head, rc_, cnt, pos, q, k, v, 16, 1e4)
    a = 4
    c1 = np.minimum(cnt, a).astype(np.int32)
    o1, K1, V1 = o.prefill_ring(Kr, Vr, head, rc_, c1, pos, q[:, :a], k[:, :a], v[:, :a], 16, 1e4)
    o2, K2, V2 = o.prefill_ring(K1, V1, (head + c1) % R, np.minimum(rc_ + c1, R), cnt - c1, pos + c1,
                                q[:, a:], k[:, a:], v[:, a:], 16, 1e4)
    for s in range(S):
        close(out[s, :c1[s]], o1[s, :c1[s]], 0.0, "first part")
        close(out[s, a:cnt[s]], o2[s, :cnt[s] - a], 0.0, "second part")
    assert np.array_equal(Kf, K2) and np.array_equal(Vf, V2), "ring after both parts"
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, [5, 0], n + 1, 1906)
    seq = np.array([5, 0], np.int32)
    out, Kf, Vf = o.prefill_paged(Kp, Vp, bt, seq, cnt, seq, q, k, v, 16, 5e6)
    o1, K1, V1 = o.prefill_paged(Kp, Vp, bt, seq, c1, seq, q[:, :a], k[:, :a], v[:, :a], 16, 5e6)
    o2, K2, V2 = o.prefill_paged(K1, V1, bt, seq + c1, cnt - c1, seq + c1, q[:, a:], k[:, a:], v[:, a:], 16, 5e6)
    for s in range(S):
        close(out[s, :c1[s]], o1[s, :c1[s]], 0.0, "first part (paged)")
        close(out[s, a:cnt[s]], o2[s, :cnt[s] - a], 0.0, "second part (paged)")
    assert np.array_equal(Kf, K2) and np.array_equal(Vf, V2), "pages after both parts"


def pin_prefill_equals_chain_verify_then_commit(o):
    """Prefill (serial decodes) and tree verify over a chain followed by the
    commit of the whole chain give the same outputs and caches, on ring and
    paged layers: two independent routes to the same attention."""
    S, T, Hq, Hkv, D, R, P = 2, 6, 4, 2, 16, 8, 4
    q = rand_bf16((S, T, Hq, D), 2001)
    k = rand_bf16((S, T, Hkv, D), 2002)
    v = rand_bf16((S, T, Hkv, D), 2003)
    g = rand_bf16((S, T, Hq), 2004)
    chain = np.stack([np.arange(-1, T - 1, dtype=np.int32)] * S)
    acc = np.stack([np.arange(T, dtype=np.int32)] * S)
    full = np.array([T, T], np.int32)
    Kr = rand_bf16((S, Hkv, R, D), 2005)
    Vr = rand_bf16((S, Hkv, R, D), 2006)
    head, cnt, pos = np.array([5, 1], np.int32), np.array([R, 3], np.int32), np.array([100, 3], np.int32)
    out, Kf, Vf = o.prefill_ring(Kr, Vr, head, cnt, full, pos, q, k, v, 16, 1e4, gate=g)
    ver, _ = o.verify_ring(Kr, Vr, head, cnt, pos, q, k, v, chain, 16, 1e4, gate=g)
    Kc, Vc, rc = o.commit_ring(Kr, Vr, head, pos, k, v, chain, acc, full, 16, 1e4)
    close(out, ver, 1e-12, "ring: prefill vs chain verify")
    assert rc == 0 and np.array_equal(Kf, Kc) and np.array_equal(Vf, Vc), "ring: prefill vs commit"
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, [7, 2], T + 1, 2007)
    seq = np.array([7, 2], np.int32)
    out, Kf, Vf = o.prefill_paged(Kp, Vp, bt, seq, full, seq, q, k, v, 16, 5e6, gate=g)
    ver, _ = o.verify(Kp, Vp, bt, seq, q, k, v, chain, 16, 5e6, gate=g)
    Kc, Vc, rc = o.commit_paged(Kp, Vp, bt, seq, seq, k, v, chain, acc, full, 16, 5e6)
    close(out, ver, 1e-12, "paged: prefill vs chain verify")
    assert rc == 0 and np.array_equal(Kf, Kc) and np.array_equal(Vf, Vc), "paged: prefill vs commit"


# ------------------------------------------------------------------ fp8 cache
# OCP FP8 E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no
# infinities (0x7f is NaN), subnormals m * 2^-9. Golden values worked out by
# hand from that definition.
E4M3_GOLDEN = [  # (byte, value)
    (0x00, 0.0), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x38, 1.0), (0x39, 1.125),
    (0x3C, 1.5), (0x40, 2.0), (0x7E, 448.0), (0xB8, -1.0), (0xFE, -448.0), (0x30, 0.5), (0x58, 16.0),
]
E4M3_ROUNDING = [  # (x, byte): nearest, ties to even, saturating at 448
    (1.0625, 0x38),          # tie between 1.0 (even) and 1.125
    (1.1875, 0x3A),          # tie between 1.125 and 1.25 (even)
    (1.06, 0x38), (1.07, 0x39),
    (2.0 ** -10, 0x00),      # tie between 0 and 2^-9
    (3 * 2.0 ** -10, 0x02),  # tie between 2^-9 and 2^-8 (even)
    (7.5 * 2.0 ** -9, 0x08), # rounds up into the normals
    (447.0, 0x7E), (460.0, 0x7E), (1e6, 0x7E), (-1e6, 0xFE), (-0.0, 0x80),
    (0.3, 0x2A),             # 0.3 = 1.2 * 2^-2 -> 1.25 * 2^-2 (mantissa 2)
]


def pin_e4m3_golden_values_and_rounding(o):
    """E4M3 decoding and nearest-even saturating rounding against values
    worked out by hand from the format's definition; every byte round-trips."""
    for b, v in E4M3_GOLDEN:
        assert o.e4m3_value(b) == v, (hex(b), o.e4m3_value(b), v)
    for x, b in E4M3_ROUNDING:
        assert o.e4m3_round(x) == b, (x, hex(o.e4m3_round(x)), hex(b))
    for b in range(256):
        if b & 0x7F == 0x7F:
            assert math.isnan(o.e4m3_value(b))
            continue
        v = o.e4m3_value(b)
        assert o.e4m3_round(v) == (0x00 if v == 0 and b == 0 else b) or (v == 0 and b == 0x80), hex(b)


def pin_fp8_decode_equals_bf16_decode_on_exact_values(o):
    """When every cached value and the new token are E4M3 numbers times the
    scales (powers of two, so every step is exact), the fp8 decode equals the
    bf16 decode of the dequantised cache, and stores the token's bytes."""
    rng = np.random.default_rng(2101)
    Hq, Hkv, D, R = 4, 2, 32, 6
    ks, vs = 0.5, 4.0
    bytes_ok = np.array([b for b in range(256) if b & 0x7F != 0x7F and b & 0x78 != 0x78], np.uint8)  # |x| < 256
    K8 = rng.choice(bytes_ok, (2, Hkv, R, D)).astype(np.uint8)
    V8 = rng.choice(bytes_ok, (2, Hkv, R, D)).astype(np.uint8)
    deq = lambda a, s: bf16(np.vectorize(o.e4m3_value)(a) * s)
    q = rand_bf16((1, Hq, D), 2102)
    kn8 = rng.choice(bytes_ok, (1, Hkv, D)).astype(np.uint8)
    vn8 = rng.choice(bytes_ok, (1, Hkv, D)).astype(np.uint8)
    k_new, v_new = deq(kn8, ks), deq(vn8, vs)
    # no rotation (r = 0): the new K entry is k_new itself, exactly E4M3 * ks
    out8, ke, ve = o.decode_fp8(K8, V8, q, k_new, v_new, [13], 0, 0.0, ks, vs, ring=([2], [5], [1]))
    out, _, _ = o.decode_ring(deq(K8, ks), deq(V8, vs), [2], [5], q, k_new, v_new, [13], 0, 0.0, stream_rows=[1])
    close(out8, out, 1e-12, "fp8 vs bf16 on exact values")
    assert np.array_equal(ke, kn8) and np.array_equal(ve, vn8), "stored bytes"


# ------------------------------------------------------------------ QK-norm
# "pega-omni PR #4", talker kernels: RoPE with QK-norm. Reading (the page
# gives no formula): y = bf16(w * x / sqrt(mean(x^2) + eps)), per head.

def pin_qk_norm_closed_forms(o):
    """Vectors whose norm is known in closed form: a constant vector c maps to
    sign(c) * w (eps = 0); ones with eps = 3 map to w / 2; a single nonzero
    entry a maps to sign(a) * sqrt(D) * w there and 0 elsewhere."""
    D = 256
    w = bf16(np.linspace(-1.5, 2.0, D).astype(np.float32).round(2))
    wv = bf16_val(w)
    for c in (1.0, 3.0, -2.0, 0.375):
        y = o.qk_norm(bf16(np.full(D, c)), w, 0.0)
        assert np.array_equal(bf16_val(y), np.sign(c) * wv), f"constant {c}"
    y = o.qk_norm(bf16(np.ones(D)), w, 3.0)
    assert np.array_equal(bf16_val(y), wv / 2), "eps inside the root"
    x = np.zeros(D, np.float32)
    x[5] = -0.75
    y = bf16_val(o.qk_norm(bf16(x), w, 0.0))
    want = np.zeros(D)
    want[5] = -math.sqrt(D) * wv[5]  # sqrt(256) = 16: exact
    assert np.array_equal(y, want), "single entry"


def pin_qk_norm_scale_invariance(o):
    """With eps = 0 the norm does not see a power-of-two scale of its input
    (every step scales exactly), bit for bit."""
    D = 128
    x = rand_bf16(D, 1201)
    w = rand_bf16(D, 1202)
    base = o.qk_norm(x, w, 0.0)
    for k in (-20, -3, 5, 30):
        xs = bf16(bf16_val(x) * 2.0 ** k)
        assert np.array_equal(o.qk_norm(xs, w, 0.0), base), f"scale 2^{k}"


def pin_qk_norm_is_rounded_exact_value(o):
    """Each element is the bf16 nearest (ties to even) to the exact
    w_d x_d / sqrt(mean(x^2) + eps), the root to 50 digits (mpmath) and the
    rounding in rational arithmetic; elements whose exact value lies within
    2^-40 of a rounding boundary (relative) are skipped and must be rare."""
    from fractions import Fraction
    mpmath = __import__("mpmath")
    mpmath.mp.dps = 50
    skipped = checked = 0
    for n, (D, eps, scale) in enumerate(((256, 1e-6, 1.0), (128, 1e-5, 1e-3), (256, 0.5, 4.0), (64, 0.0, 30.0))):
        x = bf16(bf16_val(rand_bf16(D, 1300 + n)) * scale)
        w = rand_bf16(D, 1400 + n)
        y = o.qk_norm(x, w, eps)
        xv, wv = bf16_val(x), bf16_val(w)
        ss = sum(mpmath.mpf(float(v)) ** 2 for v in xv)
        inv = 1 / mpmath.sqrt(ss / D + mpmath.mpf(eps))
        for d in range(D):
            exact = _mpf_fraction(mpmath.mpf(float(wv[d])) * mpmath.mpf(float(xv[d])) * inv)
            if exact != 0 and _bf16_midpoint_distance(exact) < abs(float(exact)) * 2.0 ** -40:
                skipped += 1
                continue
            checked += 1
            assert int(y[d]) == _bf16_of_fraction(exact), f"case {n}, element {d}"
    assert skipped <= 2 and checked > 600, (skipped, checked)


def pin_qk_norm_applies_before_rope_to_q_and_new_keys(o):
    """With QK-norm, decode, verify and append equal the same calls without
    it on inputs normalised beforehand: the norm acts on q and on the new
    keys (not on cached entries or V), before RoPE."""
    Hq, Hkv, D, R, P = 4, 2, 16, 5, 4
    eps = 1e-3
    wq, wk = rand_bf16(D, 1501), rand_bf16(D, 1502)
    nq = lambda a: np.stack([o.qk_norm(r, wq, eps) for r in a.reshape(-1, D)]).reshape(a.shape)
    nk = lambda a: np.stack([o.qk_norm(r, wk, eps) for r in a.reshape(-1, D)]).reshape(a.shape)
    norm = (wq, wk, eps)
    # ring decode
    Kr = rand_bf16((2, Hkv, R, D), 1503)
    Vr = rand_bf16((2, Hkv, R, D), 1504)
    q = rand_bf16((2, Hq, D), 1505)
    kn = rand_bf16((2, Hkv, D), 1506)
    vn = rand_bf16((2, Hkv, D), 1507)
    a = o.decode_ring(Kr, Vr, [2, 4], [3, 5], q, kn, vn, [9, 40], 16, 1e4, qk_norm=norm)
    b = o.decode_ring(Kr, Vr, [2, 4], [3, 5], nq(q), nk(kn), vn, [9, 40], 16, 1e4)
    assert all(np.array_equal(x, y) for x, y in zip(a, b)), "ring decode"
    a = o.decode_ring(Kr, Vr, [2, 4], [3, 5], q, kn, vn, [9, 40], 16, 1e4, qk_norm=(None, wk, eps))
    b = o.decode_ring(Kr, Vr, [2, 4], [3, 5], q, nk(kn), vn, [9, 40], 16, 1e4)
    assert all(np.array_equal(x, y) for x, y in zip(a, b)), "ring decode, keys only"
    # verify
    S, T = 1, 4
    Kp, Vp, bt = _prefix_pool(S, Hkv, D, P, [6], T + 1, 1510)
    qv = rand_bf16((S, T, Hq, D), 1511)
    kv = rand_bf16((S, T, Hkv, D), 1512)
    vv = rand_bf16((S, T, Hkv, D), 1513)
    parent = np.array([[-1, 0, 0, 2]], np.int32)
    a = o.verify(Kp, Vp, bt, [6], qv, kv, vv, parent, 16, 5e6, qk_norm=norm)
    b = o.verify(Kp, Vp, bt, [6], nq(qv), nk(kv), vv, parent, 16, 5e6)
    assert all(np.array_equal(x, y) for x, y in zip(a, b)), "verify"
    # append (rotate on: normalised then turned; rotate off: stored as given)
    Ka, Va = o.append_paged(Kp, Vp, bt, [6], [6], [3], kv[:, :3], vv[:, :3], 16, 5e6, qk_norm=norm)
    Kb, Vb = o.append_paged(Kp, Vp, bt, [6], [6], [3], nk(kv[:, :3]), vv[:, :3], 16, 5e6)
    assert np.array_equal(Ka, Kb) and np.array_equal(Va, Vb), "append"
    Ka, _ = o.append_paged(Kp, Vp, bt, [6], [6], [3], kv[:, :3], vv[:, :3], 16, 5e6, rotate=False,
                           qk_norm=norm)
    Kb, _ = o.append_paged(Kp, Vp, bt, [6], [6], [3], kv[:, :3], vv[:, :3], 16, 5e6, rotate=False)
    assert np.array_equal(Ka, Kb), "append without rotation stores the keys as given"


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
