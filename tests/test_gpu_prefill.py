"""Ragged prefill on the GPU vs the fp64 oracle, through the C ABI.

Stream s brings count[s] new tokens; token t attends to the cache and to new
tokens 0..t, and every entry is written back - the oracle decodes the tokens
one after another. The library runs the tokens through the verify pass in
chunks (chain trees) and commits each chunk before the next. Inputs past a
stream's count are NaN (they must not be read), and output rows past it keep
a sentinel (they must not be written). Rings wrap (more new tokens than
slots); paged prefixes are ragged, empty and page-aligned. Caches are
compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev, host_u16

pytestmark = pytest.mark.gpu
SENTINEL = 12345.0


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def new_tokens(gen, S, Tmax, Hq, Hkv, D, count, gate):
    q = synth.randn_bf16((S, Tmax, Hq, D), gen)
    k = synth.randn_bf16((S, Tmax, Hkv, D), gen)
    v = synth.randn_bf16((S, Tmax, Hkv, D), gen)
    g = synth.randn_bf16((S, Tmax, Hq), gen) if gate else None
    for s in range(S):  # rows past the stream's tokens must not be read
        for a in (q, k, v) + ((g,) if gate else ()):
            a[s, count[s]:] = synth.NAN_BF16
    return q, k, v, g


def check_out(out, ref, count, what):
    o = out.cpu().numpy()
    for s in range(len(count)):
        assert_close(o[s, :count[s]], ref[s, :count[s]], f"{what}, stream {s}")
        assert np.all(o[s, count[s]:] == SENTINEL), f"{what}: rows past count[{s}] were written"


def run_paged(dattn, oracle, seed, S, Hq, Hkv, D, P, lens, count, rope, gate=False, qk_norm=None):
    gen = synth.generator(seed)
    Tmax = max(max(count), 1)
    cache = synth.paged_cache(gen, S, Hkv, D, P, lens, room=Tmax)
    count = np.asarray(count, np.int32)
    q, k, v, g = new_tokens(gen, S, Tmax, Hq, Hkv, D, count, gate)
    start = (np.asarray(lens, np.int32) + synth.randint(0, 3, S, gen)).astype(np.int32)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": P, "rotary_dim": rope[0], "rope_theta": rope[1]}
    if qk_norm is not None:
        layer.update(q_norm=qk_norm[0], k_norm=qk_norm[1], norm_eps=qk_norm[2])
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_context=int(max(l + Tmax for l in lens)), max_verify_rows=16)
    kd, vd = dev(cache.k), dev(cache.v)
    desc = dattn.paged_cache(kd, vd, dev(cache.block_table), dev(cache.seq_len))
    out = torch.full((S, Tmax, Hq, D), SENTINEL, device="cuda")
    h.prefill(0, desc, dev(q), dev(k), dev(v), dev(count), dev(start), out, gate=None if g is None else dev(g))
    assert h.get_error() == dattn.OK
    ref, Ko, Vo = oracle.prefill_paged(cache.k, cache.v, cache.block_table, cache.seq_len, count, start, q, k, v,
                                       rope[0], rope[1], gate=g, qk_norm=qk_norm)
    check_out(out, ref, count, "paged prefill")
    assert np.array_equal(host_u16(kd), Ko), f"K pool: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo), "V pool"
    h.close()


def test_paged_full_layer(dattn, oracle):
    """Full layers: 8 q / 2 KV heads, head_dim 256, first 64 dims rotated
    (theta 5e6); ragged counts over ragged prefixes, gate on; 7 chunks."""
    run_paged(dattn, oracle, 4000, 4, 8, 2, 256, 16, [0, 300, 17, 1000], [37, 0, 16, 100], (64, 5e6), gate=True)


def test_paged_head_dim_128_with_qk_norm(dattn, oracle):
    gen = torch.Generator().manual_seed(4101)
    w = lambda: (1.0 + 0.25 * torch.randn(128, generator=gen)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    run_paged(dattn, oracle, 4100, 3, 16, 2, 128, 64, [64, 0, 129], [33, 16, 5], (128, 1e6),
              qk_norm=(w(), w(), 1e-6))


def test_ring_sliding_layer(dattn, oracle):
    """Sliding layers: all 256 dims rotated (theta 1e4), rings of 511 slots:
    full, partly filled and empty, one stream prefilling more tokens than the
    ring holds (the ring wraps and keeps its newest 511)."""
    S, Hq, Hkv, D, R = 4, 8, 2, 256, 511
    gen = synth.generator(4200)
    counts_ring = [R, 200, 0, R - 3]
    cache = synth.ring_cache(gen, S, Hkv, D, R, counts_ring, n_rows=S + 1,
                             stream_rows=synth.randperm(S + 1, gen)[:S])
    count = np.array([600, 5, 0, 40], np.int32)
    Tmax = int(count.max())
    q, k, v, g = new_tokens(gen, S, Tmax, Hq, Hkv, D, count, True)
    start = synth.randint(0, 50000, S, gen)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 256, "rope_theta": 1e4}
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_verify_rows=16)
    kd, vd = dev(cache.k), dev(cache.v)
    desc = dattn.ring_cache(kd, vd, dev(cache.head), dev(cache.count), dev(cache.stream_rows))
    out = torch.full((S, Tmax, Hq, D), SENTINEL, device="cuda")
    h.prefill(0, desc, dev(q), dev(k), dev(v), dev(count), dev(start), out, gate=dev(g))
    assert h.get_error() == dattn.OK
    ref, Ko, Vo = oracle.prefill_ring(cache.k, cache.v, cache.head, cache.count, count, start, q, k, v, 256, 1e4,
                                      gate=g, stream_rows=cache.stream_rows)
    check_out(out, ref, count, "ring prefill")
    assert np.array_equal(host_u16(kd), Ko), f"K ring: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo), "V ring"
    h.close()


def test_small_ring_shorter_than_a_chunk(dattn, oracle):
    """A ring of 7 slots: chunks shrink to the ring, tokens keep wrapping."""
    S, Hq, Hkv, D, R = 2, 4, 1, 128, 7
    gen = synth.generator(4300)
    cache = synth.ring_cache(gen, S, Hkv, D, R, [3, R])
    count = np.array([23, 9], np.int32)
    q, k, v, _ = new_tokens(gen, S, 23, Hq, Hkv, D, count, False)
    start = np.array([3, 1000], np.int32)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 128, "rope_theta": 1e4}
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_verify_rows=16)
    kd, vd = dev(cache.k), dev(cache.v)
    desc = dattn.ring_cache(kd, vd, dev(cache.head), dev(cache.count), dev(cache.stream_rows))
    out = torch.full((S, 23, Hq, D), SENTINEL, device="cuda")
    h.prefill(0, desc, dev(q), dev(k), dev(v), dev(count), dev(start), out)
    assert h.get_error() == dattn.OK
    ref, Ko, Vo = oracle.prefill_ring(cache.k, cache.v, cache.head, cache.count, count, start, q, k, v, 128, 1e4,
                                      stream_rows=cache.stream_rows)
    check_out(out, ref, count, "small ring prefill")
    assert np.array_equal(host_u16(kd), Ko) and np.array_equal(host_u16(vd), Vo)
    h.close()


def test_prefill_then_decode(dattn, oracle):
    """Prefill, advance the metadata, decode the next token."""
    S, Hq, Hkv, D, P = 2, 8, 2, 256, 16
    gen = synth.generator(4400)
    lens = [100, 0]
    cache = synth.paged_cache(gen, S, Hkv, D, P, lens, room=40)
    count = np.array([30, 17], np.int32)
    q, k, v, _ = new_tokens(gen, S, 30, Hq, Hkv, D, count, False)
    start = np.array(lens, np.int32)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": P, "rotary_dim": 64, "rope_theta": 5e6}
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_context=200, max_verify_rows=16)
    kd, vd, bt = dev(cache.k), dev(cache.v), dev(cache.block_table)
    desc = dattn.paged_cache(kd, vd, bt, dev(cache.seq_len))
    out = torch.full((S, 30, Hq, D), SENTINEL, device="cuda")
    h.prefill(0, desc, dev(q), dev(k), dev(v), dev(count), dev(start), out)
    seq2 = (cache.seq_len + count).astype(np.int32)
    seq2_d = dev(seq2)
    desc2 = dattn.paged_cache(kd, vd, bt, seq2_d)
    x = synth.decode_inputs(gen, S, Hq, Hkv, D, seq2, gate=True)
    o2 = torch.full((S, Hq, D), float("nan"), device="cuda")
    h.decode(0, desc2, dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.pos), o2, gate=dev(x.gate), write_back=False)
    assert h.get_error() == dattn.OK
    _, Ko, Vo = oracle.prefill_paged(cache.k, cache.v, cache.block_table, cache.seq_len, count, start, q, k, v,
                                     64, 5e6)
    ref, _, _ = oracle.decode_paged(Ko, Vo, cache.block_table, seq2, x.q, x.k_new, x.v_new, x.pos, 64, 5e6,
                                    gate=x.gate)
    assert_close(o2.cpu().numpy(), ref, "decode after prefill")
    h.close()


def test_prefill_reports_a_bad_count(dattn):
    """count[s] beyond max_tokens: the stream gets no tokens, DATTN_EINDEX."""
    D, R = 128, 31
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 0, "rope_theta": 0.0}
    h = dattn.Handle(2, 1, D, [layer], 2, max_verify_rows=16)
    K = torch.zeros((2, 1, R, D), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    z = torch.zeros(2, dtype=torch.int32, device="cuda")
    desc = dattn.ring_cache(K, V, z, z)
    x = torch.ones((2, 4, 2, D), dtype=torch.bfloat16, device="cuda")
    kv = torch.ones((2, 4, 1, D), dtype=torch.bfloat16, device="cuda")
    count = torch.tensor([2, 5], dtype=torch.int32, device="cuda")
    out = torch.full((2, 4, 2, D), SENTINEL, device="cuda")
    h.prefill(0, desc, x, kv, kv, count, z, out)
    assert h.get_error() == dattn.EINDEX
    assert torch.count_nonzero(K[1]) == 0 and torch.count_nonzero(K[0]) == 2 * D
    assert torch.all(out[1] == SENTINEL)
    h.close()
