"""The library's fp64 -> bf16 and fp64 -> E4M3 roundings (csrc/round_f64.h,
built for the host) against the oracle's own definitions of the same values:
the QK-normalised q and k entries, and every byte the fp8 cache stores, come
from these two functions. Every E4M3 value and every midpoint between two,
each with its fp64 neighbours; bf16 midpoints across the whole exponent
range, subnormals, overflow, signed zeros and NaN. No GPU needed."""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_attention_kv_dattn_gb300", "csrc")

SHIM = r"""
#include "round_f64.h"
extern "C" void bf16_batch(const double* y, unsigned short* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = dattn::bf16_from_f64(y[i]);
}
extern "C" void e4m3_batch(const double* y, unsigned char* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = dattn::e4m3_from_f64(y[i]);
}
"""


@pytest.fixture(scope="module")
def shim():
    d = tempfile.mkdtemp(prefix="dattn_round_")
    src, lib = os.path.join(d, "shim.cpp"), os.path.join(d, "shim.so")
    open(src, "w").write(SHIM)
    subprocess.run(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-shared", "-fPIC", "-I", CSRC, src, "-o", lib],
                   check=True)
    L = ctypes.CDLL(lib)
    P = ctypes.c_void_p
    L.bf16_batch.argtypes = [P, P, ctypes.c_long]
    L.e4m3_batch.argtypes = [P, P, ctypes.c_long]
    return L


def _call(fn, y, dtype):
    y = np.ascontiguousarray(y, np.float64)
    out = np.empty(len(y), dtype)
    fn(y.ctypes.data_as(ctypes.c_void_p), out.ctypes.data_as(ctypes.c_void_p), len(y))
    return out


def _with_neighbours(v):
    """v and the fp64 values one and two units either side of it."""
    v = np.asarray(v, np.float64)
    out = [v]
    lo, hi = v.copy(), v.copy()
    for _ in range(2):
        lo, hi = np.nextafter(lo, -np.inf), np.nextafter(hi, np.inf)
        out += [lo, hi]
    return np.concatenate(out)


def _e4m3_grid(oracle):
    vals = np.array([oracle.e4m3_value(b) for b in range(256)])
    fin = np.unique(vals[np.isfinite(vals)])
    mids = (fin[:-1] + fin[1:]) / 2  # exact in fp64
    edge = np.array([448.0, 464.0, 480.0, 1e9, 2.0 ** -10, 2.0 ** -11, 1e-300, 0.0, -0.0, np.inf, -np.inf, np.nan])
    return np.concatenate([_with_neighbours(np.concatenate([fin, mids, -mids])), edge])


def test_e4m3_every_value_and_midpoint(shim, oracle):
    y = _e4m3_grid(oracle)
    got = _call(shim.e4m3_batch, y, np.uint8)
    want = np.array([oracle.e4m3_round(t) for t in y], np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(y[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_e4m3_random_scaled_values(shim, oracle):
    rng = np.random.default_rng(3)
    y = rng.standard_normal(30000) * 2.0 ** rng.integers(-14, 10, 30000)
    got = _call(shim.e4m3_batch, y, np.uint8)
    want = np.array([oracle.e4m3_round(t) for t in y], np.uint8)
    assert np.array_equal(got, want)


def _bf16_grid():
    # every bf16 exponent: the value, the midpoint above it, each +- 2 fp64 units
    e = np.arange(-133, 128, dtype=np.float64)
    mant = np.array([1.0, 1.0 + 2.0 ** -7, 1.5, 2.0 - 2.0 ** -7])
    base = (mant[None, :] * 2.0 ** e[:, None]).ravel()
    base = base[np.isfinite(base)]
    half = np.maximum(2.0 ** -134, 2.0 ** (np.floor(np.log2(base)) - 8))
    mids = base + half
    sub = np.arange(0, 260, dtype=np.float64) * 2.0 ** -134  # subnormal grid and its midpoints
    big = np.array([3.3895313892515355e38, 3.3961775292304957e38, 3.402823466e38, 1e39, 1e300])
    ys = _with_neighbours(np.concatenate([base, mids, sub, big]))
    ys = np.concatenate([ys, -ys, [0.0, -0.0, np.inf, -np.inf, np.nan, 5e-324, -5e-324]])
    return ys


def test_bf16_midpoints_every_exponent(shim, oracle):
    y = _bf16_grid()
    got = _call(shim.bf16_batch, y, np.uint16)
    want = np.array([oracle.bf16_round(t) for t in y], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(y[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_bf16_random_values(shim, oracle):
    rng = np.random.default_rng(4)
    y = rng.standard_normal(40000) * 2.0 ** rng.integers(-140, 130, 40000)
    got = _call(shim.bf16_batch, y, np.uint16)
    want = np.array([oracle.bf16_round(t) for t in y], np.uint16)
    assert np.array_equal(got, want)
