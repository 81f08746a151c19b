"""GPU tree verify vs the fp64 oracle, through the C ABI.

Covers the tree-verify workload (16 streams x 16 rows, random best-first trees,
paged prefixes U[512, 8192], 24 q / 4 KV heads, head_dim 256), chain and star
trees, empty and short prefixes, the gate, head_dim 128, and the window entries
written back (bit for bit).
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


def run_verify(dattn, oracle, case: synth.VerifyCase, write_back=True, qk_norm=None):
    c = case.cache
    S, T = case.q.shape[:2]
    k_pool, v_pool = dev(c.k), dev(c.v)
    bt, seq = dev(c.block_table), dev(c.seq_len)
    q, k, v, par = dev(case.q), dev(case.k), dev(case.v), dev(case.parent)
    gate = None if case.gate is None else dev(case.gate)
    out = torch.full((S, T, case.Hq, case.D), float("nan"), device="cuda")
    layer = {"kind": dattn.CACHE_PAGED, "page_size": c.P, "rotary_dim": case.rope.rotary_dim,
             "rope_theta": case.rope.theta}
    if qk_norm is not None:
        layer.update(q_norm=qk_norm[0], k_norm=qk_norm[1], norm_eps=qk_norm[2])
    h = dattn.Handle(case.Hq, case.Hkv, case.D, [layer], S, max_context=int(c.seq_len.max()) or 1,
                     max_verify_rows=T)
    h.verify(0, dattn.paged_cache(k_pool, v_pool, bt, seq), q, k, v, par, out, gate=gate,
             write_back=write_back)
    assert h.get_error() == dattn.OK
    ref, ke = oracle.verify(c.k, c.v, c.block_table, c.seq_len, case.q, case.k, case.v,
                            case.parent, case.rope.rotary_dim, case.rope.theta, gate=case.gate,
                            qk_norm=qk_norm)
    err = assert_close(out.cpu().numpy(), ref, "verify")
    if write_back:
        kexp, vexp = c.k.copy(), c.v.copy()
        for s in range(S):
            for i in range(T):
                idx = int(c.seq_len[s]) + i
                pg, off = int(c.block_table[s, idx // c.P]), idx % c.P
                kexp[pg, :, off] = ke[s, i]
                vexp[pg, :, off] = case.v[s, i]
        assert np.array_equal(host_u16(k_pool), kexp), "K pool after write-back"
        assert np.array_equal(host_u16(v_pool), vexp), "V pool after write-back"
    h.close()
    return err


def small_case(seed, S, T, Hq, Hkv, D, lens, trees="random", gate=False, rope=(64, 5e6), P=16):
    gen = synth.generator(seed)
    cache = synth.paged_cache(gen, S, Hkv, D, P, lens, room=T)
    if trees == "random":
        parent = np.stack([synth.tree_parents(gen, T) for _ in range(S)])
    elif trees == "chain":
        parent = np.stack([synth.chain_parents(T)] * S)
    else:
        parent = np.stack([synth.star_parents(T)] * S)
    q = synth.randn_bf16((S, T, Hq, D), gen)
    k = synth.randn_bf16((S, T, Hkv, D), gen)
    v = synth.randn_bf16((S, T, Hkv, D), gen)
    g = synth.randn_bf16((S, T, Hq), gen) if gate else None
    return synth.VerifyCase(Hq, Hkv, D, synth.RopeSpec(*rope), cache, q, k, v, parent, g)


def test_tree_verify_workload(dattn, oracle):
    run_verify(dattn, oracle, synth.tree_verify(3))


@pytest.mark.parametrize("trees", ["chain", "star"])
def test_chain_and_star_trees(dattn, oracle, trees):
    run_verify(dattn, oracle, synth.tree_verify(5, S=4, trees=trees, lo=512, hi=2000))


@pytest.mark.parametrize("lens", [[0, 1, 5, 63], [64, 65, 130, 700]])
def test_short_and_empty_prefixes(dattn, oracle, lens):
    run_verify(dattn, oracle, small_case(11, 4, 16, 24, 4, 256, lens, gate=True))


@pytest.mark.parametrize("T", [1, 3, 16])
def test_row_counts(dattn, oracle, T):
    run_verify(dattn, oracle, small_case(12 + T, 3, T, 24, 4, 256, [300, 1000, 77]))


def test_head_dim_128(dattn, oracle):
    run_verify(dattn, oracle, small_case(20, 5, 16, 16, 8, 128, [900, 40, 2048, 0, 333],
                                         rope=(128, 1e6), gate=True))


def test_page_size_64(dattn, oracle):
    run_verify(dattn, oracle, small_case(21, 3, 8, 8, 2, 256, [1500, 64, 65], P=64))


def test_verify_run_to_run_bit_identity(dattn):
    case = small_case(30, 4, 16, 24, 4, 256, [2000, 600, 1300, 900])
    c = case.cache
    k_pool, v_pool = dev(c.k), dev(c.v)
    bt, seq = dev(c.block_table), dev(c.seq_len)
    q, k, v, par = dev(case.q), dev(case.k), dev(case.v), dev(case.parent)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": 16, "rotary_dim": 64, "rope_theta": 5e6}
    h = dattn.Handle(24, 4, 256, [layer], 4, max_context=2000, max_verify_rows=16)
    outs = []
    for _ in range(2):
        out = torch.empty((4, 16, 24, 256), device="cuda")
        h.verify(0, dattn.paged_cache(k_pool, v_pool, bt, seq), q, k, v, par, out, write_back=False)
        outs.append(out)
    assert torch.equal(outs[0], outs[1])


def test_bad_parent_is_reported(dattn):
    case = small_case(31, 2, 4, 24, 4, 256, [100, 100])
    case.parent[1, 2] = 3  # not an earlier node
    c = case.cache
    layer = {"kind": dattn.CACHE_PAGED, "page_size": 16, "rotary_dim": 64, "rope_theta": 5e6}
    h = dattn.Handle(24, 4, 256, [layer], 2, max_context=128, max_verify_rows=4)
    out = torch.empty((2, 4, 24, 256), device="cuda")
    h.verify(0, dattn.paged_cache(dev(c.k), dev(c.v), dev(c.block_table), dev(c.seq_len)),
             dev(case.q), dev(case.k), dev(case.v), dev(case.parent), out, write_back=False)
    assert h.get_error() == dattn.EINDEX
