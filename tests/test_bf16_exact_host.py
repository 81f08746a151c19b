"""The library's K-entry rounding (csrc/bf16_exact.h, built for the host):
the integer routine and the fp32 fast path that falls back on it, each
against the oracle's fp64 double-double definition of the same value: the
bf16 nearest to the exact x*c + y*s. Independent implementations of the
rounding the decode, append and verify kernels store; no GPU needed."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_attention_kv_dattn_gb300", "csrc")

SHIM = r"""
#include "bf16_exact.h"
extern "C" void dot2_batch(const unsigned short* x, const unsigned* c, const unsigned short* y,
                           const unsigned* s, unsigned short* out, long n, int fast) {
  for (long i = 0; i < n; ++i)
    out[i] = fast ? dattn::bf16_dot2(x[i], c[i], y[i], s[i]) : dattn::bf16_dot2_exact(x[i], c[i], y[i], s[i]);
}
"""


@pytest.fixture(scope="module")
def shim():
    d = tempfile.mkdtemp(prefix="dattn_bf16_")
    src, lib = os.path.join(d, "shim.cpp"), os.path.join(d, "shim.so")
    open(src, "w").write(SHIM)
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", "-I", CSRC, src, "-o", lib], check=True)
    L = ctypes.CDLL(lib)
    P = ctypes.c_void_p
    L.dot2_batch.argtypes = [P, P, P, P, P, ctypes.c_long, ctypes.c_int]
    return L


def _run(shim, x, c, y, s, fast):
    out = np.empty(len(x), np.uint16)
    arrs = [np.ascontiguousarray(a) for a in (x, c, y, s)]
    shim.dot2_batch(*[a.ctypes.data_as(ctypes.c_void_p) for a in arrs], out.ctypes.data_as(ctypes.c_void_p), len(x),
                    int(fast))
    return out


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(0, 1 << 16, n, dtype=np.uint64).astype(np.uint16)
    y = rng.integers(0, 1 << 16, n, dtype=np.uint64).astype(np.uint16)
    c = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    s = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    # mostly ordinary keys and angles, some of every scale and sign
    k = n // 2
    xv = rng.standard_normal(k).astype(np.float32)
    yv = rng.standard_normal(k).astype(np.float32)
    ang = rng.uniform(-7, 7, k)
    x[:k] = (xv.view(np.uint32) >> 16).astype(np.uint16)
    y[:k] = (yv.view(np.uint32) >> 16).astype(np.uint16)
    c[:k] = np.cos(ang).astype(np.float32).view(np.uint32)
    s[:k] = np.sin(ang).astype(np.float32).view(np.uint32)
    finite = ((x & 0x7F80) != 0x7F80) & ((y & 0x7F80) != 0x7F80) & \
             ((c & 0x7F800000) != 0x7F800000) & ((s & 0x7F800000) != 0x7F800000)
    return x[finite], c[finite], y[finite], s[finite]


@pytest.mark.parametrize("fast", [False, True], ids=["integer", "fp32_fast_path"])
def test_integer_rounding_matches_oracle(shim, oracle, fast):
    x, c, y, s = _cases(40000, 5)
    got = _run(shim, x, c, y, s, fast)
    cf, sf = c.view(np.float32), s.view(np.float32)
    want = np.array([oracle.bf16_dot2(int(x[i]), float(cf[i]), int(y[i]), float(sf[i])) for i in range(len(x))],
                    np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {len(x)} differ, e.g. case {bad[:3]}: got {got[bad[:3]]}, want {want[bad[:3]]}"


@pytest.mark.parametrize("fast", [False, True], ids=["integer", "fp32_fast_path"])
def test_integer_rounding_ties_and_specials(shim, oracle, fast):
    # x*c exactly on a bf16 tie with a tiny second product on either side; zeros
    xs, cs, ys, ss = [], [], [], []
    for k in range(1, 255, 2):
        cval = np.float32(1.0 + k * 2.0 ** -8)
        for yb, sval in ((67 << 7, 1.0), ((67 << 7) | 0x8000, 1.0), (0, 1.0), (0x3F80, 0.0)):
            xs.append(0x3F80), cs.append(cval), ys.append(yb), ss.append(np.float32(sval))
    for xb, yb in ((0, 0), (0x8000, 0), (0x8000, 0x8000), (0x0001, 0x0001), (0x7F7F, 0x7F7F)):
        for cval, sval in ((1.0, 1.0), (-1.0, 1.0), (1.0, -1.0), (0.5, 0.25)):
            xs.append(xb), cs.append(np.float32(cval)), ys.append(yb), ss.append(np.float32(sval))
    x = np.array(xs, np.uint16)
    y = np.array(ys, np.uint16)
    c = np.array(cs, np.float32).view(np.uint32)
    s = np.array(ss, np.float32).view(np.uint32)
    got = _run(shim, x, c, y, s, fast)
    want = np.array([oracle.bf16_dot2(int(x[i]), float(cs[i]), int(y[i]), float(ss[i])) for i in range(len(x))],
                    np.uint16)
    assert np.array_equal(got, want), [(hex(x[i]), cs[i], hex(y[i]), ss[i], hex(got[i]), hex(want[i]))
                                       for i in np.nonzero(got != want)[0][:5]]


def _near_midpoints(n, seed):
    """x*c within a few fp32 units of a bf16 rounding midpoint, plus a second
    product of every size down to nothing; and near-cancelling pairs."""
    rng = np.random.default_rng(seed)
    xv = rng.standard_normal(n).astype(np.float32)
    x = (xv.view(np.uint32) >> 16).astype(np.uint16)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # a midpoint between two bf16 values near |x| * U(0.5, 1)
    target = np.abs(xf) * rng.uniform(0.5, 1.0, n)
    tb = (target.astype(np.float32).view(np.uint32) & 0xFFFF0000) | 0x8000
    mid = tb.view(np.float32).astype(np.float64)
    c = (mid / xf).astype(np.float32)
    c = (c.view(np.uint32).astype(np.int64) + rng.integers(-3, 4, n)).astype(np.uint32)
    y = (rng.standard_normal(n).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    s = (rng.standard_normal(n) * 2.0 ** rng.integers(-40, -8, n)).astype(np.float32).view(np.uint32)
    s[: n // 8] = 0
    # cancelling: y = -x, s close to c
    k = n // 4
    y[-k:] = x[-k:] ^ 0x8000
    s[-k:] = (c[-k:].astype(np.int64) + rng.integers(-300, 300, k)).astype(np.uint32)
    ok = np.isfinite(xf) & (xf != 0)
    return x[ok], c[ok], y[ok], s[ok]


@pytest.mark.parametrize("fast", [False, True], ids=["integer", "fp32_fast_path"])
def test_rounding_near_midpoints_and_cancellation(shim, oracle, fast):
    x, c, y, s = _near_midpoints(20000, 11)
    got = _run(shim, x, c, y, s, fast)
    cf, sf = c.view(np.float32), s.view(np.float32)
    want = np.array([oracle.bf16_dot2(int(x[i]), float(cf[i]), int(y[i]), float(sf[i])) for i in range(len(x))],
                    np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"{bad.size} of {len(x)} differ, e.g. case {bad[:3]}: got {got[bad[:3]]}, want {want[bad[:3]]}"
