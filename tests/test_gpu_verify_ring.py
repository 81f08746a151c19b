"""Tree verify over ring (sliding-window) layers and the commit of accepted
paths, on the GPU vs the fp64 oracle, through the C ABI ("TensorFold PR #608":
verify windows under tree masks, a round commits only each stream's accepted
path; "vllm-omni commits", Spark model commit: three of every four layers are
sliding).

A row at depth d sees the newest min(count, R - d) entries of its ring, its
ancestors and itself; rings are full, nearly full (the oldest entries are
masked per row), partly filled and empty, with unwritten slots NaN and decoy
ring rows. Commit writes the accepted path at the next cache indices; the
pools are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def ring_verify_case(seed, S, T, Hq, Hkv, D, R, counts, trees="random", gate=True):
    gen = synth.generator(seed)
    n_rows = S + 2
    rows = synth.randperm(n_rows, gen)[:S]
    cache = synth.ring_cache(gen, S, Hkv, D, R, counts, n_rows=n_rows, stream_rows=rows)
    if trees == "random":
        parent = np.stack([synth.tree_parents(gen, T) for _ in range(S)])
    else:
        parent = np.stack([synth.chain_parents(T)] * S)
    pos = (np.asarray(counts, np.int32) + synth.randint(0, 5000, S, gen)).astype(np.int32)
    q = synth.randn_bf16((S, T, Hq, D), gen)
    k = synth.randn_bf16((S, T, Hkv, D), gen)
    v = synth.randn_bf16((S, T, Hkv, D), gen)
    g = synth.randn_bf16((S, T, Hq), gen) if gate else None
    return cache, parent, pos, q, k, v, g


def run_ring_verify(dattn, oracle, Hq, Hkv, D, R, rope, case):
    cache, parent, pos, q, k, v, g = case
    S, T = q.shape[:2]
    kd, vd = dev(cache.k), dev(cache.v)
    head, count, rows = dev(cache.head), dev(cache.count), dev(cache.stream_rows)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": rope[0], "rope_theta": rope[1]}
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_verify_rows=T)
    out = torch.full((S, T, Hq, D), float("nan"), device="cuda")
    pos_d, par_d = dev(pos), dev(parent)
    h.verify(0, dattn.ring_cache(kd, vd, head, count, rows), dev(q), dev(k), dev(v), par_d, out,
             gate=None if g is None else dev(g), write_back=False, pos=pos_d)
    assert h.get_error() == dattn.OK
    ref, _ = oracle.verify_ring(cache.k, cache.v, cache.head, cache.count, pos, q, k, v, parent, rope[0],
                                rope[1], gate=g, stream_rows=cache.stream_rows)
    assert_close(out.cpu().numpy(), ref, "ring verify")
    # verify writes nothing into a ring
    assert np.array_equal(host_u16(kd), cache.k) and np.array_equal(host_u16(vd), cache.v)
    h.close()


def test_sliding_layer_verify(dattn, oracle):
    """The sliding layers' shape: 8 q / 2 KV heads, head_dim 256, window 512,
    RoPE on all 256 dims (theta 1e4); 16 rows of random trees per stream."""
    R = 511
    counts = [0, 1, 300, R, R - 3, R - 15, R, 100]
    case = ring_verify_case(3000, 8, 16, 8, 2, 256, R, counts)
    run_ring_verify(dattn, oracle, 8, 2, 256, R, (256, 1e4), case)


def test_chain_trees_on_full_rings(dattn, oracle):
    """Chains reach depth 15: the deepest rows drop 15 of the oldest entries."""
    R = 511
    case = ring_verify_case(3100, 4, 16, 8, 2, 256, R, [R, R, R - 7, 200], trees="chain")
    run_ring_verify(dattn, oracle, 8, 2, 256, R, (256, 1e4), case)


def test_small_ring_head_dim_128(dattn, oracle):
    """A ring shorter than one tile, head_dim 128, 8 query heads per KV head."""
    R = 40
    case = ring_verify_case(3200, 3, 8, 16, 2, 128, R, [R, 33, 12], gate=False)
    run_ring_verify(dattn, oracle, 16, 2, 128, R, (128, 1e6), case)


def accepted_paths(parent, gen, T):
    """A random accepted path per stream (root first), as [S, T] and counts."""
    S = parent.shape[0]
    acc = np.full((S, T), -1, np.int32)
    num = np.zeros(S, np.int32)
    for s in range(S):
        node = int(synth.randint(0, T - 1, 1, gen)[0])
        path = []
        while node >= 0:
            path.append(node)
            node = int(parent[s, node])
        path = path[::-1][: int(synth.randint(0, len(path), 1, gen)[0])]
        acc[s, :len(path)] = path
        num[s] = len(path)
    return acc, num


def test_commit_ring(dattn, oracle):
    R, S, T, Hkv, D = 511, 6, 16, 2, 256
    case = ring_verify_case(3300, S, T, 8, Hkv, D, R, [R, 0, 300, R - 1, 17, R])
    cache, parent, pos, q, k, v, g = case
    acc, num = accepted_paths(parent, synth.generator(3301), T)
    num[1] = 0  # a stream with nothing accepted
    kd, vd = dev(cache.k), dev(cache.v)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 256, "rope_theta": 1e4}
    h = dattn.Handle(8, Hkv, D, [layer], S, max_verify_rows=T)
    desc = dattn.ring_cache(kd, vd, dev(cache.head), dev(cache.count), dev(cache.stream_rows))
    h.commit(0, desc, dev(k), dev(v), dev(parent), dev(acc), dev(num), dev(pos))
    assert h.get_error() == dattn.OK
    Ko, Vo, rc = oracle.commit_ring(cache.k, cache.v, cache.head, pos, k, v, parent, acc, num, 256, 1e4,
                                    stream_rows=cache.stream_rows)
    assert rc == 0
    assert np.array_equal(host_u16(kd), Ko), f"K ring: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo)
    h.close()


def test_commit_paged_after_verify(dattn, oracle):
    """A paged verify with write-back puts every window entry at seq_len + i;
    commit then rewrites seq_len + d with the accepted path's entries."""
    from test_gpu_verify import small_case
    case = small_case(3400, 4, 16, 24, 4, 256, [700, 0, 129, 2000])
    c = case.cache
    S, T = case.q.shape[:2]
    acc, num = accepted_paths(case.parent, synth.generator(3401), T)
    kd, vd = dev(c.k), dev(c.v)
    bt, seq = dev(c.block_table), dev(c.seq_len)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": c.P, "rotary_dim": 64, "rope_theta": 5e6}
    h = dattn.Handle(24, 4, 256, [layer], S, max_context=int(c.seq_len.max()), max_verify_rows=T)
    desc = dattn.paged_cache(kd, vd, bt, seq)
    out = torch.empty((S, T, 24, 256), device="cuda")
    kq, kk, kv, kp = dev(case.q), dev(case.k), dev(case.v), dev(case.parent)
    h.verify(0, desc, kq, kk, kv, kp, out, write_back=True)
    h.commit(0, desc, kk, kv, kp, dev(acc), dev(num), seq)
    assert h.get_error() == dattn.OK
    # expected: the verify's node-order write-back, then the committed path
    _, ke = oracle.verify(c.k, c.v, c.block_table, c.seq_len, case.q, case.k, case.v, case.parent, 64, 5e6)
    Kw, Vw = c.k.copy(), c.v.copy()
    for s in range(S):
        for i in range(T):
            t = int(c.seq_len[s]) + i
            Kw[c.block_table[s, t // c.P], :, t % c.P] = ke[s, i]
            Vw[c.block_table[s, t // c.P], :, t % c.P] = case.v[s, i]
    Ko, Vo, rc = oracle.commit_paged(Kw, Vw, c.block_table, c.seq_len, c.seq_len, case.k, case.v, case.parent,
                                     acc, num, 64, 5e6)
    assert rc == 0
    assert np.array_equal(host_u16(kd), Ko), f"K pool: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo)
    h.close()


def test_verify_commit_then_decode(dattn, oracle):
    """One speculative round on a sliding layer end to end: verify, commit the
    accepted path, advance the ring, decode the next token - against the
    oracle doing the same."""
    R, S, T, Hq, Hkv, D = 511, 4, 8, 8, 2, 256
    case = ring_verify_case(3500, S, T, Hq, Hkv, D, R, [R, 250, R - 2, 0], gate=False)
    cache, parent, pos, q, k, v, _ = case
    acc, num = accepted_paths(parent, synth.generator(3501), T)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 256, "rope_theta": 1e4}
    h = dattn.Handle(Hq, Hkv, D, [layer], S, max_verify_rows=T)
    kd, vd = dev(cache.k), dev(cache.v)
    head_d, count_d, rows_d = dev(cache.head), dev(cache.count), dev(cache.stream_rows)
    desc = dattn.ring_cache(kd, vd, head_d, count_d, rows_d)
    out = torch.empty((S, T, Hq, D), device="cuda")
    kk, kv, kp, pos_d = dev(k), dev(v), dev(parent), dev(pos)
    h.verify(0, desc, dev(q), kk, kv, kp, out, write_back=False, pos=pos_d)
    h.commit(0, desc, kk, kv, kp, dev(acc), dev(num), pos_d)
    head2 = ((cache.head + num) % R).astype(np.int32)
    count2 = np.minimum(cache.count + num, R).astype(np.int32)
    pos2 = (pos + num).astype(np.int32)
    gen = synth.generator(3502)
    x = synth.decode_inputs(gen, S, Hq, Hkv, D, pos2, gate=True)
    head2_d, count2_d = dev(head2), dev(count2)
    desc2 = dattn.ring_cache(kd, vd, head2_d, count2_d, rows_d)
    o2 = torch.full((S, Hq, D), float("nan"), device="cuda")
    h.decode(0, desc2, dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.pos), o2, gate=dev(x.gate), write_back=False)
    assert h.get_error() == dattn.OK
    Kc, Vc, rc = oracle.commit_ring(cache.k, cache.v, cache.head, pos, k, v, parent, acc, num, 256, 1e4,
                                    stream_rows=cache.stream_rows)
    ref, _, _ = oracle.decode_ring(Kc, Vc, head2, count2, x.q, x.k_new, x.v_new, x.pos, 256, 1e4, gate=x.gate,
                                   stream_rows=cache.stream_rows)
    assert_close(o2.cpu().numpy(), ref, "decode after verify + commit")
    h.close()


def test_commit_rejects_a_broken_path(dattn):
    """A list that is not a path from a root writes nothing for its stream and
    is reported as DATTN_EINDEX; the other streams are committed."""
    R, Hkv, D, T = 31, 1, 128, 4
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 0, "rope_theta": 0.0}
    h = dattn.Handle(2, Hkv, D, [layer], 2, max_verify_rows=T)
    K = torch.zeros((2, Hkv, R, D), dtype=torch.bfloat16, device="cuda")
    V = torch.zeros_like(K)
    head = torch.tensor([3, 3], dtype=torch.int32, device="cuda")
    count = torch.zeros(2, dtype=torch.int32, device="cuda")
    desc = dattn.ring_cache(K, V, head, count)
    k = torch.ones((2, T, Hkv, D), dtype=torch.bfloat16, device="cuda")
    parent = torch.tensor([[-1, 0, 1, 1], [-1, 0, 1, 1]], dtype=torch.int32, device="cuda")
    acc = torch.tensor([[0, 1, 3, -1], [0, 2, 3, -1]], dtype=torch.int32, device="cuda")  # stream 1: 2's parent is 1
    num = torch.tensor([3, 3], dtype=torch.int32, device="cuda")
    pos = torch.zeros(2, dtype=torch.int32, device="cuda")
    h.commit(0, desc, k, k, parent, acc, num, pos)
    assert h.get_error() == dattn.EINDEX
    assert torch.count_nonzero(K[1]) == 0, "the broken stream wrote nothing"
    assert torch.count_nonzero(K[0]) == 3 * D * Hkv, "the other stream was committed"
    h.close()


def test_ring_verify_argument_checks(dattn):
    R, D = 31, 128
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 0, "rope_theta": 0.0}
    h = dattn.Handle(2, 1, D, [layer], 1, max_verify_rows=2)
    K = torch.zeros((1, 1, R, D), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = dattn.ring_cache(K, K, z, z)
    q = torch.zeros((1, 2, 2, D), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 2, 1, D), dtype=torch.bfloat16, device="cuda")
    par = torch.tensor([[-1, 0]], dtype=torch.int32, device="cuda")
    out = torch.empty((1, 2, 2, D), device="cuda")
    for kw in ({"write_back": False}, {"write_back": True, "pos": z}):  # no pos; write-back on a ring
        with pytest.raises(dattn.DattnError) as e:
            h.verify(0, desc, q, kv, kv, par, out, **kw)
        assert e.value.code == dattn.EINVAL
    h.close()
