"""ctypes front end of the fp64 CPU oracle (test infrastructure only).

Only the test suite, `__graft_entry__.smoke()` and the benchmark's CPU-baseline
leg import this package; the library's product path never does. Every array is
a numpy array: bf16 data as uint16 bit patterns, metadata as int32, results as
float64. See dattn_oracle.cpp for the definitions and the passages they follow.
"""
import ctypes
import numpy as np

from .build import build_oracle

_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double
_L = ctypes.c_int64


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _norm(qk_norm):
    """QK-norm arguments: qk_norm = (q weights, k weights, eps) as bf16 [D]
    arrays (either may be None: no norm on that side) and a float, or None
    for a layer without QK-norm."""
    if qk_norm is None:
        return (None, None, 0.0)
    qw, kw, eps = qk_norm
    global _keep_norm
    _keep_norm = tuple(None if w is None else _u16(w) for w in (qw, kw))
    return (_ptr(_keep_norm[0]), _ptr(_keep_norm[1]), float(eps))


_keep_norm = None


class Oracle:
    """One loaded build of the oracle (mutation 0 is the real one)."""

    def __init__(self, mutation: int = 0):
        self.mutation = mutation
        self.lib = ctypes.CDLL(build_oracle(mutation))
        L = self.lib
        L.oracle_bf16_round.argtypes = [_D]
        L.oracle_bf16_round.restype = ctypes.c_uint16
        L.oracle_bf16_dot2.argtypes = [ctypes.c_uint16, ctypes.c_float, ctypes.c_uint16, ctypes.c_float]
        L.oracle_bf16_dot2.restype = ctypes.c_uint16
        L.oracle_rope_cos_sin.argtypes = [_I, _D, _L, _I, ctypes.POINTER(_D), ctypes.POINTER(_D)]
        L.oracle_rope_cos_sin.restype = None
        L.oracle_rope_f64.argtypes = [_P, _I, _I, _D, _L, _P]
        L.oracle_rope_bf16.argtypes = [_P, _I, _I, _D, _L, _P]
        N3 = [_P, _P, _D]  # QK-norm: q weight, k weight (bf16 [D] or null), eps
        L.oracle_decode_ring.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P,
                                         _P, _P, _P, _P, _P, _P, _P, _P, _I] + N3
        L.oracle_decode_paged.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _I, _P,
                                          _P, _P, _P, _P, _P, _P, _P, _P, _I] + N3
        L.oracle_decode_concat.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _P, _P, _P, _P,
                                           _P, _P, _P, _I] + N3
        L.oracle_verify.argtypes = [_I, _I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _I, _P,
                                    _P, _P, _P, _P, _P, _P, _P, _P, _I] + N3
        L.oracle_verify_ring.argtypes = [_I, _I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P,
                                         _P, _P, _P, _P, _P, _P, _P, _P, _I] + N3
        L.oracle_commit_ring.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P,
                                         _P, _P, _P, _P, _P, _P, _D]
        L.oracle_commit_paged.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _I, _P, _P,
                                          _P, _P, _P, _P, _P, _P, _D]
        L.oracle_append_ring.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P,
                                         _P, _P, _P, _I, _P, _D]
        L.oracle_append_paged.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _I, _P,
                                          _P, _P, _P, _P, _I, _P, _D]
        L.oracle_prefill_ring.argtypes = [_I, _I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P, _P] + N3
        L.oracle_prefill_paged.argtypes = [_I, _I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _I, _P, _P, _P,
                                           _P, _P, _P, _P, _P] + N3
        L.oracle_decode_fp8.argtypes = [_I, _I, _I, _I, _I, _I, _D, _P, _P, _I, _I, _P, _P, _P, _P, _I, _P,
                                        _D, _D, _P, _P, _P, _P, _P, _P, _P, _P] + N3
        L.oracle_decode_fp8.restype = _I
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = _D
        L.oracle_e4m3_round.argtypes = [_D]
        L.oracle_e4m3_round.restype = ctypes.c_uint8
        L.oracle_qk_norm.argtypes = [_P, _P, _I, _D, _P]
        L.oracle_qk_norm.restype = None
        for f in ("oracle_rope_f64", "oracle_rope_bf16", "oracle_decode_ring",
                  "oracle_decode_paged", "oracle_decode_concat", "oracle_verify",
                  "oracle_verify_ring", "oracle_commit_ring", "oracle_commit_paged",
                  "oracle_prefill_ring", "oracle_prefill_paged",
                  "oracle_append_ring", "oracle_append_paged", "oracle_hardware_threads"):
            getattr(L, f).restype = _I

    @staticmethod
    def _check(rc, what):
        if rc != 0:
            raise ValueError(f"oracle {what}: invalid arguments (code {rc})")

    # ---- numbers and RoPE
    def bf16_round(self, t: float) -> int:
        return int(self.lib.oracle_bf16_round(float(t)))

    def bf16_dot2(self, x_bits, c, y_bits, s) -> int:
        """bf16 bits nearest to the exact x*c + y*s (x, y bf16 bits; c, s fp32)."""
        return int(self.lib.oracle_bf16_dot2(int(x_bits), float(c), int(y_bits), float(s)))

    def rope_cos_sin(self, r, theta, pos, i):
        c, s = _D(), _D()
        self.lib.oracle_rope_cos_sin(r, theta, pos, i, ctypes.byref(c), ctypes.byref(s))
        return c.value, s.value

    def rope_f64(self, x, r, theta, pos):
        x = _u16(x)
        out = np.empty(x.shape[-1], np.float64)
        self._check(self.lib.oracle_rope_f64(_ptr(x), x.shape[-1], r, theta, pos, _ptr(out)), "rope")
        return out

    def qk_norm(self, x, w, eps):
        """QK-norm of one bf16 head vector x with bf16 weights w: bf16 bits."""
        x, w = _u16(x), _u16(w)
        out = np.empty(x.shape[-1], np.uint16)
        self.lib.oracle_qk_norm(_ptr(x), _ptr(w), x.shape[-1], float(eps), _ptr(out))
        return out

    def rope_bf16(self, x, r, theta, pos):
        x = _u16(x)
        out = np.empty(x.shape[-1], np.uint16)
        self._check(self.lib.oracle_rope_bf16(_ptr(x), x.shape[-1], r, theta, pos, _ptr(out)), "rope")
        return out

    # ---- decode
    def decode_ring(self, k_ring, v_ring, ring_head, ring_count, q, k_new, v_new, pos,
                    r, theta, gate=None, stream_rows=None, n_threads=0, qk_norm=None):
        """k_ring/v_ring [rows, Hkv, R, D]; q [B, Hq, D]; k_new/v_new [B, Hkv, D].
        Returns (out [B,Hq,D] f64, k_entry [B,Hkv,D] u16, v_entry [B,Hkv,D] u16)."""
        k_ring, v_ring, q, k_new, v_new = map(_u16, (k_ring, v_ring, q, k_new, v_new))
        gate = None if gate is None else _u16(gate)
        n_rows, Hkv, R, D = k_ring.shape
        B, Hq, _ = q.shape
        out = np.empty((B, Hq, D), np.float64)
        ke = np.empty((B, Hkv, D), np.uint16)
        ve = np.empty((B, Hkv, D), np.uint16)
        sr, hd, ct, ps = _i32(stream_rows), _i32(ring_head), _i32(ring_count), _i32(pos)
        rc = self.lib.oracle_decode_ring(B, Hq, Hkv, D, r, theta, _ptr(k_ring), _ptr(v_ring),
                                         n_rows, R, _ptr(sr), _ptr(hd), _ptr(ct), _ptr(q),
                                         _ptr(k_new), _ptr(v_new), _ptr(gate), _ptr(ps),
                                         _ptr(out), _ptr(ke), _ptr(ve), n_threads, *_norm(qk_norm))
        self._check(rc, "decode_ring")
        return out, ke, ve

    def decode_paged(self, k_pages, v_pages, block_table, seq_len, q, k_new, v_new, pos,
                     r, theta, gate=None, n_threads=0, qk_norm=None):
        """k_pages/v_pages [num_pages, Hkv, P, D]; block_table [B, max_pages]."""
        k_pages, v_pages, q, k_new, v_new = map(_u16, (k_pages, v_pages, q, k_new, v_new))
        gate = None if gate is None else _u16(gate)
        num_pages, Hkv, P, D = k_pages.shape
        B, Hq, _ = q.shape
        bt = _i32(block_table)
        out = np.empty((B, Hq, D), np.float64)
        ke = np.empty((B, Hkv, D), np.uint16)
        ve = np.empty((B, Hkv, D), np.uint16)
        sl, ps = _i32(seq_len), _i32(pos)
        rc = self.lib.oracle_decode_paged(B, Hq, Hkv, D, r, theta, _ptr(k_pages), _ptr(v_pages),
                                          num_pages, P, _ptr(bt), bt.shape[1], _ptr(sl),
                                          _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(gate),
                                          _ptr(ps), _ptr(out), _ptr(ke), _ptr(ve), n_threads,
                                          *_norm(qk_norm))
        self._check(rc, "decode_paged")
        return out, ke, ve

    def decode_concat(self, k_chrono, v_chrono, count, q, k_new, v_new, pos, r, theta,
                      gate=None, n_threads=0, qk_norm=None):
        """Key-space twin: k_chrono/v_chrono [B, Hkv, cap, D] oldest first."""
        k_chrono, v_chrono, q, k_new, v_new = map(_u16, (k_chrono, v_chrono, q, k_new, v_new))
        gate = None if gate is None else _u16(gate)
        B, Hkv, cap, D = k_chrono.shape
        Hq = q.shape[1]
        out = np.empty((B, Hq, D), np.float64)
        ct, ps = _i32(count), _i32(pos)
        rc = self.lib.oracle_decode_concat(B, Hq, Hkv, D, r, theta, _ptr(k_chrono),
                                           _ptr(v_chrono), cap, _ptr(ct), _ptr(q), _ptr(k_new),
                                           _ptr(v_new), _ptr(gate), _ptr(ps), _ptr(out),
                                           n_threads, *_norm(qk_norm))
        self._check(rc, "decode_concat")
        return out

    # ---- verify
    def verify(self, k_pages, v_pages, block_table, prefix_len, q, k, v, parent, r, theta,
               gate=None, n_threads=0, qk_norm=None, pos=None):
        """q [S,T,Hq,D]; k/v [S,T,Hkv,D]; parent [S,T]; pos [S] root positions
        (default prefix_len). Returns (out f64, k_entry u16)."""
        k_pages, v_pages, q, k, v = map(_u16, (k_pages, v_pages, q, k, v))
        gate = None if gate is None else _u16(gate)
        num_pages, Hkv, P, D = k_pages.shape
        S, T, Hq, _ = q.shape
        bt = _i32(block_table)
        out = np.empty((S, T, Hq, D), np.float64)
        ke = np.empty((S, T, Hkv, D), np.uint16)
        pl, pa = _i32(prefix_len), _i32(parent)
        ps = _i32(pos)
        rc = self.lib.oracle_verify(S, T, Hq, Hkv, D, r, theta, _ptr(k_pages), _ptr(v_pages),
                                    num_pages, P, _ptr(bt), bt.shape[1], _ptr(pl), _ptr(ps), _ptr(q),
                                    _ptr(k), _ptr(v), _ptr(pa), _ptr(gate), _ptr(out), _ptr(ke),
                                    n_threads, *_norm(qk_norm))
        self._check(rc, "verify")
        return out, ke

    def verify_ring(self, k_ring, v_ring, ring_head, ring_count, pos, q, k, v, parent, r, theta,
                    gate=None, stream_rows=None, n_threads=0, qk_norm=None):
        """Tree verify over ring (sliding) layers: k_ring/v_ring [rows, Hkv, R, D];
        pos [S] root positions. Returns (out f64, k_entry u16)."""
        k_ring, v_ring, q, k, v = map(_u16, (k_ring, v_ring, q, k, v))
        gate = None if gate is None else _u16(gate)
        n_rows, Hkv, R, D = k_ring.shape
        S, T, Hq, _ = q.shape
        out = np.empty((S, T, Hq, D), np.float64)
        ke = np.empty((S, T, Hkv, D), np.uint16)
        sr, hd, ct, ps, pa = map(_i32, (stream_rows, ring_head, ring_count, pos, parent))
        rc = self.lib.oracle_verify_ring(S, T, Hq, Hkv, D, r, theta, _ptr(k_ring), _ptr(v_ring), n_rows, R,
                                         _ptr(sr), _ptr(hd), _ptr(ct), _ptr(ps), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(pa), _ptr(gate), _ptr(out), _ptr(ke), n_threads,
                                         *_norm(qk_norm))
        self._check(rc, "verify_ring")
        return out, ke

    # ---- commit of accepted paths (returns updated copies and the status:
    # 0, or 3 when some stream's list was not a path and was skipped)
    def commit_ring(self, k_ring, v_ring, ring_head, pos, k, v, parent, accepted, num_accepted,
                    r, theta, stream_rows=None, qk_norm=None):
        kr, vr = _u16(k_ring).copy(), _u16(v_ring).copy()
        k, v = _u16(k), _u16(v)
        n_rows, Hkv, R, D = kr.shape
        S, T = k.shape[:2]
        rc = self.lib.oracle_commit_ring(S, T, Hkv, D, r, theta, _ptr(kr), _ptr(vr), n_rows, R,
                                         _ptr(_i32(stream_rows)), _ptr(_i32(ring_head)), _ptr(_i32(pos)),
                                         _ptr(k), _ptr(v), _ptr(_i32(parent)), _ptr(_i32(accepted)),
                                         _ptr(_i32(num_accepted)), *_norm(qk_norm)[1:])
        if rc not in (0, 3):
            self._check(rc, "commit_ring")
        return kr, vr, rc

    def commit_paged(self, k_pages, v_pages, block_table, seq_len, pos, k, v, parent, accepted,
                     num_accepted, r, theta, qk_norm=None):
        kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
        k, v = _u16(k), _u16(v)
        num_pages, Hkv, P, D = kp.shape
        S, T = k.shape[:2]
        bt = _i32(block_table)
        rc = self.lib.oracle_commit_paged(S, T, Hkv, D, r, theta, _ptr(kp), _ptr(vp), num_pages, P, _ptr(bt),
                                          bt.shape[1], _ptr(_i32(seq_len)), _ptr(_i32(pos)), _ptr(k), _ptr(v),
                                          _ptr(_i32(parent)), _ptr(_i32(accepted)),
                                          _ptr(_i32(num_accepted)), *_norm(qk_norm)[1:])
        if rc not in (0, 3):
            self._check(rc, "commit_paged")
        return kp, vp, rc

    # ---- fp8 (E4M3) caches
    def e4m3_value(self, b) -> float:
        return float(self.lib.oracle_e4m3_value(int(b)))

    def e4m3_round(self, x) -> int:
        return int(self.lib.oracle_e4m3_round(float(x)))

    def decode_fp8(self, k_cache, v_cache, q, k_new, v_new, pos, r, theta, k_scale, v_scale, gate=None,
                   ring=None, paged=None, qk_norm=None):
        """Decode over E4M3 caches (uint8): ring=(head, count, stream_rows or None) with
        k/v [rows, Hkv, R, D], or paged=(block_table, seq_len) with k/v [pages, Hkv, P, D].
        Returns (out f64, k_entry u8, v_entry u8)."""
        k_cache = np.ascontiguousarray(k_cache, np.uint8)
        v_cache = np.ascontiguousarray(v_cache, np.uint8)
        q, k_new, v_new = map(_u16, (q, k_new, v_new))
        gate = None if gate is None else _u16(gate)
        n_rows, Hkv, RP, D = k_cache.shape
        B, Hq, _ = q.shape
        out = np.empty((B, Hq, D), np.float64)
        ke = np.empty((B, Hkv, D), np.uint8)
        ve = np.empty((B, Hkv, D), np.uint8)
        if ring is not None:
            head, count, rows = map(_i32, ring)
            bt, sl, bts = None, None, 0
        else:
            bt, sl = map(_i32, paged)
            head = count = rows = None
            bts = bt.shape[1]
        rc = self.lib.oracle_decode_fp8(0 if ring is not None else 1, B, Hq, Hkv, D, r, theta, _ptr(k_cache),
                                        _ptr(v_cache), n_rows, RP, _ptr(rows), _ptr(head), _ptr(count), _ptr(bt),
                                        bts, _ptr(sl), float(k_scale), float(v_scale), _ptr(q), _ptr(k_new),
                                        _ptr(v_new), _ptr(gate), _ptr(_i32(pos)), _ptr(out), _ptr(ke), _ptr(ve),
                                        *_norm(qk_norm))
        self._check(rc, "decode_fp8")
        return out, ke, ve

    # ---- ragged prefill (returns out and updated copies of the pools)
    def prefill_ring(self, k_ring, v_ring, ring_head, ring_count, count, start_pos, q, k, v, r, theta,
                     gate=None, stream_rows=None, qk_norm=None):
        kr, vr = _u16(k_ring).copy(), _u16(v_ring).copy()
        q, k, v = _u16(q), _u16(k), _u16(v)
        gate = None if gate is None else _u16(gate)
        n_rows, Hkv, R, D = kr.shape
        S, Tmax, Hq, _ = q.shape
        out = np.full((S, Tmax, Hq, D), np.nan)
        rc = self.lib.oracle_prefill_ring(S, Tmax, Hq, Hkv, D, r, theta, _ptr(kr), _ptr(vr), n_rows, R,
                                          _ptr(_i32(stream_rows)), _ptr(_i32(ring_head)), _ptr(_i32(ring_count)),
                                          _ptr(_i32(count)), _ptr(_i32(start_pos)), _ptr(q), _ptr(k), _ptr(v),
                                          _ptr(gate), _ptr(out), *_norm(qk_norm))
        self._check(rc, "prefill_ring")
        return out, kr, vr

    def prefill_paged(self, k_pages, v_pages, block_table, seq_len, count, start_pos, q, k, v, r, theta,
                      gate=None, qk_norm=None):
        kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
        q, k, v = _u16(q), _u16(k), _u16(v)
        gate = None if gate is None else _u16(gate)
        num_pages, Hkv, P, D = kp.shape
        S, Tmax, Hq, _ = q.shape
        bt = _i32(block_table)
        out = np.full((S, Tmax, Hq, D), np.nan)
        rc = self.lib.oracle_prefill_paged(S, Tmax, Hq, Hkv, D, r, theta, _ptr(kp), _ptr(vp), num_pages, P,
                                           _ptr(bt), bt.shape[1], _ptr(_i32(seq_len)), _ptr(_i32(count)),
                                           _ptr(_i32(start_pos)), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                           _ptr(out), *_norm(qk_norm))
        self._check(rc, "prefill_paged")
        return out, kp, vp

    # ---- append (returns updated copies)
    def append_ring(self, k_ring, v_ring, start_index, start_pos, count, k, v, r, theta,
                    rotate=True, stream_rows=None, qk_norm=None):
        kr, vr = _u16(k_ring).copy(), _u16(v_ring).copy()
        k, v = _u16(k), _u16(v)
        n_rows, Hkv, R, D = kr.shape
        B, Tmax = k.shape[:2]
        rc = self.lib.oracle_append_ring(B, Tmax, Hkv, D, r, theta, _ptr(kr), _ptr(vr), n_rows, R,
                                         _ptr(_i32(stream_rows)), _ptr(_i32(start_index)),
                                         _ptr(_i32(start_pos)), _ptr(_i32(count)), _ptr(k),
                                         _ptr(v), int(rotate), *_norm(qk_norm)[1:])
        self._check(rc, "append_ring")
        return kr, vr

    def append_paged(self, k_pages, v_pages, block_table, start_index, start_pos, count, k, v,
                     r, theta, rotate=True, qk_norm=None):
        kp, vp = _u16(k_pages).copy(), _u16(v_pages).copy()
        k, v = _u16(k), _u16(v)
        num_pages, Hkv, P, D = kp.shape
        B, Tmax = k.shape[:2]
        bt = _i32(block_table)
        rc = self.lib.oracle_append_paged(B, Tmax, Hkv, D, r, theta, _ptr(kp), _ptr(vp),
                                          num_pages, P, _ptr(bt), bt.shape[1],
                                          _ptr(_i32(start_index)), _ptr(_i32(start_pos)),
                                          _ptr(_i32(count)), _ptr(k), _ptr(v), int(rotate),
                                          *_norm(qk_norm)[1:])
        self._check(rc, "append_paged")
        return kp, vp

    def hardware_threads(self) -> int:
        return int(self.lib.oracle_hardware_threads())


_default = None


def get() -> Oracle:
    """The real (unmutated) oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
