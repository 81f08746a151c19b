"""Helpers of the GPU parity tests: move synthetic cases to the device, run the
library through its C ABI, and compare with the oracle.

Tolerance (fp32 outputs from bf16 inputs, fp32 accumulation), per element:
|gpu - oracle| <= 2e-3 and |gpu - oracle| / max(|oracle|, 0.2) <= 1e-2. The
floor 0.2 = 2e-3 / 1e-2 makes the two bounds meet. Index work and the K/V
entries written back are compared bit for bit.
"""
import numpy as np
import torch

import synth

ABS_TOL = 2e-3
REL_TOL = 1e-2
REL_FLOOR = 0.2


def dev(a):
    """numpy -> CUDA tensor; uint16 arrays become bf16 tensors (same bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def host_u16(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    d = np.abs(gpu - ref)
    worst = np.unravel_index(np.argmax(d), d.shape) if d.size else ()
    assert d.max(initial=0.0) <= ABS_TOL, \
        f"{what}: max abs error {d.max():.3e} at {worst} (gpu {gpu[worst]:.6f}, ref {ref[worst]:.6f})"
    rel = d / np.maximum(np.abs(ref), REL_FLOOR)
    assert rel.max(initial=0.0) <= REL_TOL, f"{what}: max rel error {rel.max():.3e}"
    return float(d.max(initial=0.0))


def layer_dict(case, qk_norm=None):
    """The case's layer for dattn.Handle; qk_norm = (q weights, k weights, eps)
    (bf16 bits [D] each, either may be None) adds a QK-norm."""
    if case.kind == "ring":
        d = {"kind": 0, "ring_slots": case.cache.R, "rotary_dim": case.rope.rotary_dim,
             "rope_theta": case.rope.theta}
    else:
        d = {"kind": 1, "page_size": case.cache.P, "rotary_dim": case.rope.rotary_dim,
             "rope_theta": case.rope.theta}
    if qk_norm is not None:
        d.update(q_norm=qk_norm[0], k_norm=qk_norm[1], norm_eps=qk_norm[2])
    return d


class DeviceCase:
    """A synth DecodeCase resident on the GPU."""

    def __init__(self, case):
        self.case = case
        c, x = case.cache, case.inputs
        self.k = dev(c.k)
        self.v = dev(c.v)
        if case.kind == "ring":
            self.head = dev(c.head)
            self.count = dev(c.count)
            self.rows = dev(c.stream_rows)
        else:
            self.bt = dev(c.block_table)
            self.seq = dev(c.seq_len)
        self.q = dev(x.q)
        self.k_new = dev(x.k_new)
        self.v_new = dev(x.v_new)
        self.gate = None if x.gate is None else dev(x.gate)
        self.pos = dev(x.pos)
        B = x.q.shape[0]
        self.out = torch.full((B, case.Hq, case.D), float("nan"), device="cuda")

    def cache_desc(self, dattn):
        if self.case.kind == "ring":
            return dattn.ring_cache(self.k, self.v, self.head, self.count, self.rows)
        return dattn.paged_cache(self.k, self.v, self.bt, self.seq)


def make_handle(dattn, case, max_streams=None, max_context=None, max_verify_rows=0, qk_norm=None):
    B = case.inputs.q.shape[0] if hasattr(case, "inputs") else case.q.shape[0]
    if max_context is None:
        max_context = int(case.cache.seq_len.max()) if case.kind == "paged" else 0
    return dattn.Handle(case.Hq, case.Hkv, case.D, [layer_dict(case, qk_norm)],
                        max_streams or B, max_context=max_context,
                        max_verify_rows=max_verify_rows)


def oracle_decode(oracle, case, streams=None, qk_norm=None):
    """Oracle output and entries for the case (optionally a subset of streams)."""
    c, x = case.cache, case.inputs
    sel = slice(None) if streams is None else np.asarray(streams)
    gate = None if x.gate is None else x.gate[sel]
    r, th = case.rope.rotary_dim, case.rope.theta
    if case.kind == "ring":
        return oracle.decode_ring(c.k, c.v, c.head[sel], c.count[sel], x.q[sel], x.k_new[sel],
                                  x.v_new[sel], x.pos[sel], r, th, gate=gate,
                                  stream_rows=c.stream_rows[sel], qk_norm=qk_norm)
    return oracle.decode_paged(c.k, c.v, c.block_table[sel], c.seq_len[sel], x.q[sel],
                               x.k_new[sel], x.v_new[sel], x.pos[sel], r, th, gate=gate,
                               qk_norm=qk_norm)


def entry_slots(case):
    """(array index tuples) of the slot each stream's new entry is written to,
    per KV head: ring -> (row, head, slot); paged -> (page, head, offset)."""
    c = case.cache
    B = case.inputs.q.shape[0]
    out = []
    for b in range(B):
        if case.kind == "ring":
            out.append((int(c.stream_rows[b]), int(c.head[b])))
        else:
            n = int(c.seq_len[b])
            out.append((int(c.block_table[b, n // c.P]), n % c.P))
    return out


def check_write_back(case, k_after, v_after, ke, ve):
    """Only the new entries' slots changed, and they hold the oracle's bits."""
    c = case.cache
    kexp, vexp = c.k.copy(), c.v.copy()
    for b, (a0, a1) in enumerate(entry_slots(case)):
        if case.kind == "ring":
            kexp[a0, :, a1] = ke[b]
            vexp[a0, :, a1] = ve[b]
        else:
            kexp[a0, :, a1] = ke[b]
            vexp[a0, :, a1] = ve[b]
    kd = np.flatnonzero(k_after.reshape(-1) != kexp.reshape(-1))
    vd = np.flatnonzero(v_after.reshape(-1) != vexp.reshape(-1))
    assert kd.size == 0, f"K pool differs from the expected write-back at {kd.size} elements"
    assert vd.size == 0, f"V pool differs from the expected write-back at {vd.size} elements"
