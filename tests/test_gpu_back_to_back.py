"""Decode calls launched back to back on one stream, with no host sync and no
other kernel between them, against the oracle applied step by step.

A decode call may start streaming its cache while the launch before it on the
stream is still finishing, unless that launch writes into the same cache. These
tests make every call read the entry that an earlier call wrote back: the same
ring layer stepped repeatedly (each call must wait for its predecessor's
write-back), and a ring layer interleaved with a paged layer (each call
overlaps a launch that writes the other cache, and reads the entry its own
layer wrote two launches earlier). The metadata of every step (ring head and
count, paged lengths) is prepared on the device before the first launch.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev, host_u16

pytestmark = pytest.mark.gpu

HQ, HKV, D = 8, 2, 256
SLIDING, FULL = synth.SLIDING_ROPE, synth.FULL_ROPE


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


class RingLayer:
    """A ring layer with per-step inputs and metadata; a numpy twin of the
    cache that the oracle steps forward."""

    def __init__(self, gen, B, R, counts, steps):
        self.B, self.R, self.steps = B, R, steps
        self.cache = synth.ring_cache(gen, B, HKV, D, R, counts)
        self.k_np, self.v_np = self.cache.k.copy(), self.cache.v.copy()
        heads = [np.asarray(self.cache.head, np.int32)]
        cnts = [np.asarray(self.cache.count, np.int32)]
        for _ in range(steps - 1):
            heads.append(((heads[-1] + 1) % R).astype(np.int32))
            cnts.append(np.minimum(cnts[-1] + 1, R).astype(np.int32))
        self.heads, self.cnts = heads, cnts
        self.inputs = [synth.decode_inputs(gen, B, HQ, HKV, D, cnts[s] + 100, True) for s in range(steps)]
        self.k, self.v = dev(self.cache.k), dev(self.cache.v)
        self.rows = dev(self.cache.stream_rows)
        self.dev_meta = [(dev(heads[s]), dev(cnts[s])) for s in range(steps)]
        self.dev_in = [(dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.gate), dev(x.pos)) for x in self.inputs]
        self.outs = [torch.full((B, HQ, D), float("nan"), device="cuda") for _ in range(steps)]

    def layer(self, dattn):
        return {"kind": dattn.CACHE_RING, "ring_slots": self.R, "rotary_dim": SLIDING.rotary_dim,
                "rope_theta": SLIDING.theta}

    def launch(self, dattn, h, layer, s):
        head, cnt = self.dev_meta[s]
        q, kn, vn, g, pos = self.dev_in[s]
        h.decode(layer, dattn.ring_cache(self.k, self.v, head, cnt, self.rows), q, kn, vn, pos, self.outs[s],
                 gate=g, write_back=True)

    def oracle_step(self, oracle, s):
        x = self.inputs[s]
        out, ke, ve = oracle.decode_ring(self.k_np, self.v_np, self.heads[s], self.cnts[s], x.q, x.k_new, x.v_new,
                                         x.pos, SLIDING.rotary_dim, SLIDING.theta, gate=x.gate,
                                         stream_rows=self.cache.stream_rows)
        for b in range(self.B):
            row, hd = int(self.cache.stream_rows[b]), int(self.heads[s][b])
            self.k_np[row, :, hd] = ke[b]
            self.v_np[row, :, hd] = ve[b]
        return out


class PagedLayer:
    def __init__(self, gen, B, P, lens, steps):
        self.B, self.P, self.steps = B, P, steps
        self.cache = synth.paged_cache(gen, B, HKV, D, P, lens, room=steps)
        self.k_np, self.v_np = self.cache.k.copy(), self.cache.v.copy()
        self.lens = [np.asarray(lens, np.int32) + s for s in range(steps)]
        self.inputs = [synth.decode_inputs(gen, B, HQ, HKV, D, self.lens[s], True) for s in range(steps)]
        self.k, self.v = dev(self.cache.k), dev(self.cache.v)
        self.bt = dev(self.cache.block_table)
        self.dev_len = [dev(n) for n in self.lens]
        self.dev_in = [(dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.gate), dev(x.pos)) for x in self.inputs]
        self.outs = [torch.full((B, HQ, D), float("nan"), device="cuda") for _ in range(steps)]
        self.max_len = int(self.lens[-1].max()) + 1

    def layer(self, dattn):
        return {"kind": dattn.CACHE_PAGED, "page_size": self.P, "rotary_dim": FULL.rotary_dim,
                "rope_theta": FULL.theta}

    def launch(self, dattn, h, layer, s):
        q, kn, vn, g, pos = self.dev_in[s]
        h.decode(layer, dattn.paged_cache(self.k, self.v, self.bt, self.dev_len[s]), q, kn, vn, pos, self.outs[s],
                 gate=g, max_seq_len=self.max_len, write_back=True)

    def oracle_step(self, oracle, s):
        x = self.inputs[s]
        out, ke, ve = oracle.decode_paged(self.k_np, self.v_np, self.cache.block_table, self.lens[s], x.q,
                                          x.k_new, x.v_new, x.pos, FULL.rotary_dim, FULL.theta, gate=x.gate)
        for b in range(self.B):
            n = int(self.lens[s][b])
            pg = int(self.cache.block_table[b, n // self.P])
            self.k_np[pg, :, n % self.P] = ke[b]
            self.v_np[pg, :, n % self.P] = ve[b]
        return out


def test_same_ring_layer_back_to_back(dattn, oracle):
    """Six steps of one ring layer (full, nearly full, short and empty rings of
    33 slots): every call reads the slot its predecessor just wrote."""
    gen = synth.generator(900)
    L = RingLayer(gen, 4, 33, [33, 32, 10, 0], 6)
    h = dattn.Handle(HQ, HKV, D, [L.layer(dattn)], L.B)
    for s in range(L.steps):
        L.launch(dattn, h, 0, s)
    assert h.get_error() == dattn.OK
    for s in range(L.steps):
        assert_close(L.outs[s].cpu().numpy(), L.oracle_step(oracle, s), f"step {s}")
    assert np.array_equal(host_u16(L.k), L.k_np) and np.array_equal(host_u16(L.v), L.v_np)
    h.close()


def test_ring_and_paged_layers_interleaved(dattn, oracle):
    """Ring and paged layers alternating for five steps each: every call may
    overlap the other layer's launch, and reads the entry its own layer wrote
    two launches earlier."""
    gen = synth.generator(901)
    ring = RingLayer(gen, 3, 511, [511, 300, 5], 5)
    paged = PagedLayer(gen, 3, 16, [20, 31, 47], 5)
    h = dattn.Handle(HQ, HKV, D, [ring.layer(dattn), paged.layer(dattn)], 3, max_context=paged.max_len)
    for s in range(5):
        ring.launch(dattn, h, 0, s)
        paged.launch(dattn, h, 1, s)
    assert h.get_error() == dattn.OK
    for s in range(5):
        assert_close(ring.outs[s].cpu().numpy(), ring.oracle_step(oracle, s), f"ring step {s}")
        assert_close(paged.outs[s].cpu().numpy(), paged.oracle_step(oracle, s), f"paged step {s}")
    assert np.array_equal(host_u16(ring.k), ring.k_np) and np.array_equal(host_u16(ring.v), ring.v_np)
    assert np.array_equal(host_u16(paged.k), paged.k_np) and np.array_equal(host_u16(paged.v), paged.v_np)
    h.close()


def test_back_to_back_in_a_graph(dattn, oracle):
    """The interleaved sequence captured in one CUDA graph and replayed once
    (from fresh caches) gives the same outputs and caches as the oracle."""
    gen = synth.generator(902)
    ring = RingLayer(gen, 2, 64, [64, 20], 4)
    paged = PagedLayer(gen, 2, 16, [15, 16], 4)
    h = dattn.Handle(HQ, HKV, D, [ring.layer(dattn), paged.layer(dattn)], 2, max_context=paged.max_len)
    k0 = [t.clone() for t in (ring.k, ring.v, paged.k, paged.v)]
    for s in range(4):  # eager first: kernel attributes are set outside the capture
        ring.launch(dattn, h, 0, s)
        paged.launch(dattn, h, 1, s)
    assert h.get_error() == dattn.OK
    for t, t0 in zip((ring.k, ring.v, paged.k, paged.v), k0):
        t.copy_(t0)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for s in range(4):
                ring.launch(dattn, h, 0, s)
                paged.launch(dattn, h, 1, s)
    torch.cuda.synchronize()
    for t, t0 in zip((ring.k, ring.v, paged.k, paged.v), k0):
        t.copy_(t0)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert h.get_error() == dattn.OK
    for s in range(4):
        assert_close(ring.outs[s].cpu().numpy(), ring.oracle_step(oracle, s), f"ring step {s}")
        assert_close(paged.outs[s].cpu().numpy(), paged.oracle_step(oracle, s), f"paged step {s}")
    assert np.array_equal(host_u16(ring.k), ring.k_np) and np.array_equal(host_u16(paged.k), paged.k_np)
    h.close()
