"""Host check of the kernels' RoPE angle routine (csrc/rope_angle.h:
rope_cos_sin) against the exact cos and sin of its fixed-point phase.

The routine takes a position and the pair's phase step rint(2^64 theta^(-2i/r)
/ 2 pi) and promises fp32 cos and sin within 1.5e-7 of the exact values for
|pos| <= 2^21. The same header is built here for the host (every step is an
integer or correctly rounded fp32 operation, compiled without contraction), and
the phase (pos * step mod 2^64, an exact integer) is turned into an angle in
Python integers and fp64 (error ~1e-16), so the check is independent of the
routine's own arithmetic. A planted mistake in the series or the quadrant logic
moves some value by far more than the bound. A second test checks that the host
library's per-pair steps (kernels.h: rope_phase_step) are that definition, bit
for bit.
"""
import math
import os
import shutil
import struct
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "decode_attention_kv_dattn_gb300", "csrc")
BOUND = 1.5e-7

SHIM = r'''
#include <cstdio>
#include <cstring>
#include "rope_angle.h"
// stdin: "pos step" per line; stdout: the fp32 bit patterns of cos and sin.
int main() {
  long long pos;
  unsigned long long step;
  while (std::scanf("%lld %llu", &pos, &step) == 2) {
    float c, s;
    dattn::rope_cos_sin(static_cast<int64_t>(pos), static_cast<uint64_t>(step), c, s);
    unsigned cb, sb;
    std::memcpy(&cb, &c, 4);
    std::memcpy(&sb, &s, 4);
    std::printf("%08x %08x\n", cb, sb);
  }
  return 0;
}
'''


def phase_step(theta, r, i):
    """The pair's angle per position in 64-bit fixed-point turns (the host
    library's definition: fp64 frequency and division, rounded to nearest)."""
    inv = math.pow(theta, -float(2 * i) / float(r))
    return int(round(math.ldexp(inv / 6.283185307179586, 64)))


def exact_cos_sin(pos, step):
    phase = (pos % (1 << 64)) * step % (1 << 64)
    if phase >= 1 << 63:
        phase -= 1 << 64  # the same angle, within half a turn of 0
    a = 2.0 * math.pi * (phase / float(1 << 64))
    return math.cos(a), math.sin(a)


def _cases():
    rng = np.random.default_rng(4242)
    edges = [0, 1, -1, 2, 1 << 21, -(1 << 21), (1 << 21) - 1, 12345, -98765]
    out = []
    for r in (32, 64, 128, 256):
        for theta in (1e4, 1e6, 5e6):
            for i in range(r // 2):
                st = phase_step(theta, r, i)
                pos = list(edges) + [int(x) for x in rng.integers(-(1 << 21), (1 << 21) + 1, 60)]
                out.extend((p, st) for p in pos)
    # steps whose phases land next to quadrant boundaries and at the ends of the remainder range
    for k in range(4):
        for d in (-3, -1, 0, 1, 3):
            out.append((1, ((k << 62) + (1 << 61) + (d << 32)) % (1 << 64)))
            out.append((1, ((k << 62) + (d << 32)) % (1 << 64)))
    return out


def _build(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "rope_shim.cpp"
    src.write_text(SHIM)
    exe = tmp_path / "rope_shim"
    r = subprocess.run([gxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC, "-o", str(exe), str(src)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-4000:]
    return exe


def test_rope_cos_sin_within_bound(tmp_path):
    exe = _build(tmp_path)
    cases = _cases()
    text = "".join(f"{p} {s}\n" for p, s in cases)
    r = subprocess.run([str(exe)], input=text, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.split()
    assert len(lines) == 2 * len(cases)
    worst = (0.0, None)
    for k, (p, st) in enumerate(cases):
        c = struct.unpack("<f", bytes.fromhex(lines[2 * k])[::-1])[0]
        s = struct.unpack("<f", bytes.fromhex(lines[2 * k + 1])[::-1])[0]
        ec, es = exact_cos_sin(p, st)
        err = max(abs(c - ec), abs(s - es))
        if err > worst[0]:
            worst = (err, (p, st, c, s, ec, es))
    assert worst[0] <= BOUND, f"max error {worst[0]:.3e} at {worst[1]}"


STEP_SHIM = r'''
#include <cstdio>
#include "kernels.h"
// stdin: "theta r i" per line; stdout: the library's phase step.
int main() {
  double theta;
  int r, i;
  while (std::scanf("%lf %d %d", &theta, &r, &i) == 3)
    std::printf("%llu\n", static_cast<unsigned long long>(dattn::rope_phase_step(theta, r, i)));
  return 0;
}
'''


def test_library_phase_steps_match_the_definition(tmp_path):
    """The host library's per-pair steps (kernels.h: rope_phase_step) are
    rint(2^64 theta^(-2i/r) / 2 pi) as defined above, bit for bit."""
    gxx = shutil.which("g++") or shutil.which("c++")
    cuda_inc = "/usr/local/cuda/include"
    if gxx is None or not os.path.isdir(cuda_inc):
        pytest.skip("no host C++ compiler or CUDA headers")
    src = tmp_path / "step_shim.cpp"
    src.write_text(STEP_SHIM)
    exe = tmp_path / "step_shim"
    r = subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, "-I", cuda_inc, "-o", str(exe), str(src)],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-4000:]
    cases = [(theta, rd, i) for rd in (2, 32, 64, 128, 256) for theta in (1e4, 1e6, 5e6, 1.5e5)
             for i in range(rd // 2)]
    r = subprocess.run([str(exe)], input="".join(f"{t!r} {rd} {i}\n" for t, rd, i in cases),
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = [int(x) for x in r.stdout.split()]
    want = [phase_step(t, rd, i) for t, rd, i in cases]
    bad = [(c, g, w) for c, g, w in zip(cases, got, want) if g != w]
    assert len(got) == len(cases) and not bad, bad[:5]
