"""Python binding of the dattn C ABI (include/dattn.h).

Argument marshalling only: tensors are passed to the library as raw device
pointers (torch is used for device memory and streams), and every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback:
importing this package fails if libdattn.so has not been built (run
`python -c "import __graft_entry__ as g; g.build()"` or
`python decode_attention_kv_dattn_gb300/build.py`).
"""
import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"dattn CUDA library not built: {LIB_PATH} is missing "
                      "(build it with decode_attention_kv_dattn_gb300/build.py)")

lib = ctypes.CDLL(LIB_PATH)

# ---------------------------------------------------------------- C types

OK, EINVAL, EXCEEDS, ECUDA, EINDEX, ETIMEOUT, EUNSUPPORTED, ELENGTH, ERANGE = range(9)
CACHE_RING, CACHE_PAGED = 0, 1
KV_BF16, KV_E4M3 = 0, 1

_vp = ctypes.c_void_p
_int = ctypes.c_int


class LayerConfig(ctypes.Structure):
    _fields_ = [("cache_kind", _int), ("ring_slots", _int), ("page_size", _int),
                ("rotary_dim", _int), ("rope_theta", ctypes.c_double),
                ("q_norm_weight", _vp), ("k_norm_weight", _vp), ("norm_eps", ctypes.c_double),
                ("kv_format", _int), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


def _host_bf16(w, D, what):
    """QK-norm weights as a contiguous host array of D bf16 bit patterns
    (numpy uint16, or a CPU bfloat16 tensor), or None."""
    if w is None:
        return None
    if isinstance(w, torch.Tensor):
        if w.is_cuda or w.dtype != torch.bfloat16:
            raise TypeError(f"{what}: a CPU bfloat16 tensor or a uint16 numpy array")
        w = w.contiguous().view(torch.int16).numpy().view(np.uint16)
    w = np.ascontiguousarray(w, dtype=np.uint16)
    if w.shape != (D,):
        raise ValueError(f"{what}: shape {w.shape}, expected ({D},)")
    return w


class Config(ctypes.Structure):
    _fields_ = [("num_q_heads", _int), ("num_kv_heads", _int), ("head_dim", _int),
                ("max_streams", _int), ("max_context", _int), ("max_verify_rows", _int),
                ("num_layers", _int), ("layers", ctypes.POINTER(LayerConfig))]


class Cache(ctypes.Structure):
    _fields_ = [("k", _vp), ("v", _vp), ("n_rows", _int), ("ring_head", _vp),
                ("ring_count", _vp), ("stream_rows", _vp), ("block_table", _vp),
                ("bt_stride", _int), ("seq_len", _vp)]


class DecodeArgs(ctypes.Structure):
    _fields_ = [("num_streams", _int), ("q", _vp), ("k_new", _vp), ("v_new", _vp), ("gate", _vp),
                ("pos", _vp), ("out", _vp), ("max_seq_len", _int), ("write_back", _int)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("num_streams", _int), ("rows", _int), ("q", _vp), ("k", _vp), ("v", _vp),
                ("parent", _vp), ("gate", _vp), ("out", _vp), ("max_prefix_len", _int),
                ("write_back", _int), ("pos", _vp)]


lib.dattn_create.argtypes = [ctypes.POINTER(Config), _int, ctypes.POINTER(_vp)]
lib.dattn_create.restype = _int
lib.dattn_append_kv.argtypes = [_vp, _int, ctypes.POINTER(Cache), _int, _int, _vp, _vp, _vp,
                                _vp, _vp, _int, _vp]
lib.dattn_append_kv.restype = _int
lib.dattn_decode.argtypes = [_vp, _int, ctypes.POINTER(Cache), ctypes.POINTER(DecodeArgs), _vp]
lib.dattn_decode.restype = _int
lib.dattn_verify.argtypes = [_vp, _int, ctypes.POINTER(Cache), ctypes.POINTER(VerifyArgs), _vp]
lib.dattn_verify.restype = _int
lib.dattn_commit.argtypes = [_vp, _int, ctypes.POINTER(Cache), _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
lib.dattn_commit.restype = _int
lib.dattn_prefill.argtypes = [_vp, _int, ctypes.POINTER(Cache), _int, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
lib.dattn_prefill.restype = _int
lib.dattn_get_error.argtypes = [_vp, _vp]
lib.dattn_get_error.restype = _int
lib.dattn_error_string.argtypes = [_int]
lib.dattn_error_string.restype = ctypes.c_char_p
lib.dattn_destroy.argtypes = [_vp]
lib.dattn_destroy.restype = None
lib.dattn_decode_noalloc.argtypes = [ctypes.POINTER(Config), _int, ctypes.POINTER(Cache),
                                     ctypes.POINTER(DecodeArgs), _vp]
lib.dattn_decode_noalloc.restype = _int
lib.dattn_debug_config.argtypes = [_vp, _int, ctypes.c_uint]
lib.dattn_debug_config.restype = _int
DEBUG_WITHHOLD_Q = 1

EXPORTS = ("dattn_create", "dattn_append_kv", "dattn_decode", "dattn_verify", "dattn_commit", "dattn_prefill",
           "dattn_get_error", "dattn_error_string", "dattn_destroy", "dattn_decode_noalloc",
           "dattn_debug_config")


class DattnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} (status {code})")


def error_string(code: int) -> str:
    return lib.dattn_error_string(code).decode()


def _check(code, what):
    if code != OK:
        raise DattnError(code, what)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("dattn takes device tensors")
    if not t.is_contiguous():
        raise ValueError("dattn takes contiguous tensors")
    return t.data_ptr()


def _stream_ptr(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


# ---------------------------------------------------------------- cache descriptors

def ring_cache(k, v, ring_head, ring_count, stream_rows=None) -> Cache:
    """k, v: [rows, Hkv, R, D] bf16; ring_head, ring_count (, stream_rows): [B] int32.
    The descriptor holds the tensors it points to, so they live as long as it does."""
    c = Cache(_ptr(k), _ptr(v), k.shape[0], _ptr(ring_head), _ptr(ring_count),
              _ptr(stream_rows), None, 0, None)
    c._tensors = (k, v, ring_head, ring_count, stream_rows)
    return c


def paged_cache(k, v, block_table, seq_len) -> Cache:
    """k, v: [pages, Hkv, P, D] bf16; block_table [B, max_pages] int32; seq_len [B] int32.
    The descriptor holds the tensors it points to, so they live as long as it does."""
    c = Cache(_ptr(k), _ptr(v), k.shape[0], None, None, None, _ptr(block_table),
              block_table.shape[1], _ptr(seq_len))
    c._tensors = (k, v, block_table, seq_len)
    return c


# ---------------------------------------------------------------- handle

class Handle:
    """A dattn handle: per-layer RoPE tables and the split-K workspace."""

    def __init__(self, num_q_heads, num_kv_heads, head_dim, layers, max_streams,
                 max_context=0, max_verify_rows=0, device=None):
        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        # QK-norm weights (layer keys "q_norm", "k_norm", "norm_eps"): host
        # arrays the config points at, kept alive with it (dattn_create copies
        # them; decode_noalloc reads them on every call)
        self._norm_keep = []
        cfgs = []
        for l in layers:
            qn = _host_bf16(l.get("q_norm"), head_dim, "q_norm")
            kn = _host_bf16(l.get("k_norm"), head_dim, "k_norm")
            self._norm_keep += [qn, kn]
            cfgs.append(LayerConfig(l["kind"], l.get("ring_slots", 0), l.get("page_size", 0),
                                    l.get("rotary_dim", 0), float(l.get("rope_theta", 0.0)),
                                    None if qn is None else qn.ctypes.data,
                                    None if kn is None else kn.ctypes.data,
                                    float(l.get("norm_eps", 0.0)), int(l.get("kv_format", KV_BF16)),
                                    float(l.get("k_scale", 1.0)), float(l.get("v_scale", 1.0))))
        self._layers = (LayerConfig * len(layers))(*cfgs)
        self.config = Config(num_q_heads, num_kv_heads, head_dim, max_streams, max_context,
                             max_verify_rows, len(layers), self._layers)
        h = _vp()
        _check(lib.dattn_create(ctypes.byref(self.config), device, ctypes.byref(h)), "dattn_create")
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib.dattn_destroy(self._h)
            self._h = _vp()

    __del__ = close

    def append_kv(self, layer, cache: Cache, k, v, start_index, count, start_pos=None,
                  rotate=True, stream=None):
        """k, v: [B, T, Hkv, D] bf16; start_index, count (, start_pos): [B] int32."""
        B, T = k.shape[0], k.shape[1]
        _check(lib.dattn_append_kv(self._h, layer, ctypes.byref(cache), B, T, _ptr(start_index),
                                   _ptr(start_pos), _ptr(count), _ptr(k), _ptr(v), int(rotate),
                                   _stream_ptr(stream)), "dattn_append_kv")

    def decode(self, layer, cache: Cache, q, k_new, v_new, pos, out, gate=None, max_seq_len=0,
               write_back=True, stream=None):
        """q [B, Hq, D], k_new/v_new [B, Hkv, D] bf16; pos [B] int32; out [B, Hq, D] fp32;
        gate [B, Hq] bf16 or None."""
        args = DecodeArgs(q.shape[0], _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(gate), _ptr(pos),
                          _ptr(out), int(max_seq_len), int(write_back))
        _check(lib.dattn_decode(self._h, layer, ctypes.byref(cache), ctypes.byref(args),
                                _stream_ptr(stream)), "dattn_decode")

    def verify(self, layer, cache: Cache, q, k, v, parent, out, gate=None, max_prefix_len=0,
               write_back=True, pos=None, stream=None):
        """q [S, T, Hq, D], k/v [S, T, Hkv, D] bf16; parent [S, T] int32; out [S, T, Hq, D]
        fp32; gate [S, T, Hq] bf16 or None; pos [S] int32 root positions (default: the
        cache's seq_len; ring layers need it and take write_back=False)."""
        args = VerifyArgs(q.shape[0], q.shape[1], _ptr(q), _ptr(k), _ptr(v), _ptr(parent),
                          _ptr(gate), _ptr(out), int(max_prefix_len), int(write_back), _ptr(pos))
        _check(lib.dattn_verify(self._h, layer, ctypes.byref(cache), ctypes.byref(args),
                                _stream_ptr(stream)), "dattn_verify")

    def commit(self, layer, cache: Cache, k, v, parent, accepted, num_accepted, pos, stream=None):
        """Write each stream's accepted path (accepted [S, T] int32 node indices root
        first, num_accepted [S]) at the cache's next indices, rotated at pos + d;
        k, v, parent as given to the verify call."""
        _check(lib.dattn_commit(self._h, layer, ctypes.byref(cache), k.shape[0], k.shape[1], _ptr(k),
                                _ptr(v), _ptr(parent), _ptr(accepted), _ptr(num_accepted), _ptr(pos),
                                _stream_ptr(stream)), "dattn_commit")

    def prefill(self, layer, cache: Cache, q, k, v, count, start_pos, out, gate=None, stream=None):
        """Ragged prefill: q [S, T, Hq, D], k/v [S, T, Hkv, D] bf16, count/start_pos [S] int32,
        out [S, T, Hq, D] fp32 (rows t < count written), gate [S, T, Hq] bf16 or None."""
        _check(lib.dattn_prefill(self._h, layer, ctypes.byref(cache), q.shape[0], q.shape[1], _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(gate), _ptr(count), _ptr(start_pos), _ptr(out),
                                 _stream_ptr(stream)), "dattn_prefill")

    def debug_config(self, flags=0, wait_limit_us=0):
        """Testing aid: the limit of the device's bounded waits and fault
        injection on the host's side of the wait (see dattn_debug_config)."""
        _check(lib.dattn_debug_config(self._h, int(flags), int(wait_limit_us)), "dattn_debug_config")

    def get_error(self, stream=None) -> int:
        """Synchronize the stream; return and clear the sticky device status."""
        return lib.dattn_get_error(self._h, _stream_ptr(stream))


def decode_noalloc(config: Config, layer, cache: Cache, q, k_new, v_new, pos, out, gate=None,
                   max_seq_len=0, write_back=True, stream=None):
    """Decode without a handle, for callers that cannot allocate device memory:
    the library's fixed scratch array stands in for a handle's workspace.
    `config` is a Config structure (for instance Handle.config)."""
    args = DecodeArgs(q.shape[0], _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(gate), _ptr(pos),
                      _ptr(out), int(max_seq_len), int(write_back))
    _check(lib.dattn_decode_noalloc(ctypes.byref(config), layer, ctypes.byref(cache),
                                    ctypes.byref(args), _stream_ptr(stream)), "dattn_decode_noalloc")
