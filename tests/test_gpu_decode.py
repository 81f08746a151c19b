"""GPU decode vs the fp64 oracle, through the C ABI.

Covers the single sliding layer, the 28-layer hybrid step, paged batched decode
and long-context decode workloads, plus edge cases of the ring (empty, one
entry, full ring whose write-back takes the oldest slot, wrap-around, decoy
rows) and of the page table (lengths 0, 1, P-1, P, P+1, permuted pages).
Outputs are compared element by element within the stated tolerance; the K/V
entries written back and the rest of the pools are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (DeviceCase, assert_close, check_write_back, dev, host_u16, make_handle,
                      oracle_decode, layer_dict)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def run_and_check(dattn, oracle, case, streams=None, check_pool=True):
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate)
    assert h.get_error() == dattn.OK
    out = dc.out.cpu().numpy()
    ref, ke, ve = oracle_decode(oracle, case, streams)
    sel = slice(None) if streams is None else np.asarray(streams)
    err = assert_close(out[sel], ref, "decode")
    if check_pool:
        assert streams is None
        check_write_back(case, host_u16(dc.k), host_u16(dc.v), ke, ve)
    h.close()
    return err


def ring_case(seed, B, Hq, Hkv, D, R, counts, heads=None, gate=True, rope=(None, 1e4),
              n_rows=None, stream_rows=None, pos=None):
    gen = synth.generator(seed)
    cache = synth.ring_cache(gen, B, Hkv, D, R, counts, heads=heads, n_rows=n_rows,
                             stream_rows=stream_rows)
    r = D if rope[0] is None else rope[0]
    pos = counts if pos is None else pos
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, pos, gate)
    return synth.DecodeCase(Hq, Hkv, D, synth.RopeSpec(r, rope[1]), cache, x)


def paged_case(seed, B, Hq, Hkv, D, P, lens, gate=False, rope=(64, 5e6)):
    gen = synth.generator(seed)
    cache = synth.paged_cache(gen, B, Hkv, D, P, lens)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, lens, gate)
    return synth.DecodeCase(Hq, Hkv, D, synth.RopeSpec(*rope), cache, x)


# ------------------------------------------------------------------ workloads

def test_single_sliding_layer(dattn, oracle):
    run_and_check(dattn, oracle, synth.single_sliding_layer(0))


def test_paged_batched_64_streams(dattn, oracle):
    run_and_check(dattn, oracle, synth.paged_batched(2))


@pytest.mark.parametrize("B,context", [(1, 1024), (8, 1024), (8, 4096)])
def test_hybrid_step_all_layers(dattn, oracle, B, context):
    """All 28 layers of the hybrid step through one handle, each checked."""
    cases = [synth.hybrid_layer(1, l, B, context) for l in range(28)]
    h = dattn.Handle(8, 2, 256, [layer_dict(c) for c in cases], B, max_context=context)
    for l, case in enumerate(cases):
        dc = DeviceCase(case)
        h.decode(l, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate)
        ref, ke, ve = oracle_decode(oracle, case)
        assert_close(dc.out.cpu().numpy(), ref, f"layer {l}")
        check_write_back(case, host_u16(dc.k), host_u16(dc.v), ke, ve)
    assert h.get_error() == dattn.OK


def test_hybrid_step_64_streams_sampled(dattn, oracle):
    """The benchmark's configuration (64 streams, context 4096): one sliding and
    one full layer, 8 sampled streams each compared with the oracle."""
    for l in (0, 3):
        case = synth.hybrid_layer(1, l, 64, 4096)
        run_and_check(dattn, oracle, case, streams=[0, 7, 19, 31, 40, 52, 61, 63], check_pool=False)


@pytest.mark.parametrize("B,context,streams", [(1, 1 << 20, [0]), (8, 1 << 18, [0, 5])])
def test_long_context(dattn, oracle, B, context, streams):
    case = synth.long_context(4, B, context)
    run_and_check(dattn, oracle, case, streams=streams, check_pool=False)


# ------------------------------------------------------------------ ring edge cases

@pytest.mark.parametrize("D,Hq,Hkv", [(256, 8, 2), (128, 16, 8), (256, 8, 1), (256, 24, 4),
                                      (128, 4, 4), (128, 16, 2)])
def test_ring_group_sizes(dattn, oracle, D, Hq, Hkv):
    case = ring_case(10 + Hq, 3, Hq, Hkv, D, 61, [61, 17, 40], heads=[5, 60, 0])
    run_and_check(dattn, oracle, case)


@pytest.mark.parametrize("counts,heads", [([0], [7]), ([1], [0]), ([511], [0]), ([511], [300]),
                                          ([300], [100]), ([7], [3]), ([510], [509])])
def test_ring_fill_states(dattn, oracle, counts, heads):
    case = ring_case(20, 1, 8, 2, 256, 511, counts, heads=heads, pos=[counts[0] + 1000])
    run_and_check(dattn, oracle, case)


def test_ring_stream_rows_with_decoys(dattn, oracle):
    """Call rows map to permuted ring rows; the unused rows are NaN decoys."""
    case = ring_case(30, 4, 8, 2, 256, 100, [100, 3, 55, 0], heads=[0, 99, 20, 5],
                     n_rows=7, stream_rows=[5, 0, 3, 6])
    run_and_check(dattn, oracle, case)


def test_ring_no_gate_no_rope(dattn, oracle):
    case = ring_case(31, 2, 8, 2, 256, 33, [33, 10], gate=False, rope=(0, 1e4))
    run_and_check(dattn, oracle, case)


# ------------------------------------------------------------------ paged edge cases

@pytest.mark.parametrize("P", [16, 64])
def test_paged_ragged_lengths(dattn, oracle, P):
    lens = [0, 1, P - 1, P, P + 1, 3 * P + 5, 1000, 2 * P]
    case = paged_case(40 + P, len(lens), 8, 2, 256, P, lens, gate=True)
    run_and_check(dattn, oracle, case)


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 16, 8), (256, 8, 2), (256, 24, 4), (128, 8, 8)])
def test_paged_group_sizes(dattn, oracle, D, Hq, Hkv):
    lens = [700, 33, 1500]
    case = paged_case(50 + Hq, len(lens), Hq, Hkv, D, 16, lens, rope=(D, 1e6))
    run_and_check(dattn, oracle, case)


def test_many_short_units_per_cta(dattn, oracle):
    """512 (stream, KV head) units, most of them a few keys long (some empty)
    and a few long ones: the weighted split gives some CTAs dozens of unit
    segments, each prepared and ended by the helper warp while the streaming
    warps go on."""
    rng = np.random.default_rng(7)
    lens = [int(x) for x in rng.integers(0, 40, 256)]
    for b in (3, 100, 200):
        lens[b] = 3000
    for b in (5, 6, 50):
        lens[b] = 0
    case = paged_case(61, len(lens), 4, 2, 128, 16, lens, gate=True, rope=(128, 1e6))
    run_and_check(dattn, oracle, case)


def test_many_short_ring_units(dattn, oracle):
    """The same on ring caches: 256 streams x 2 KV heads, short and empty rings."""
    rng = np.random.default_rng(8)
    counts = [int(x) for x in rng.integers(0, 30, 256)]
    counts[10] = 63
    case = ring_case(62, 256, 8, 2, 256, 63, counts)
    run_and_check(dattn, oracle, case)


def test_lengths_far_below_the_planned_bound(dattn, oracle):
    """The split grid is sized from the call's bound; when the streams are much
    shorter, many split CTAs get no keys and the combine must skip them."""
    case = paged_case(45, 3, 8, 2, 256, 16, [17, 0, 5], gate=True)
    dc = DeviceCase(case)
    h = make_handle(dattn, case, max_context=65536)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate,
             max_seq_len=65536)
    assert h.get_error() == dattn.OK
    ref, ke, ve = oracle_decode(oracle, case)
    assert_close(dc.out.cpu().numpy(), ref)


# ------------------------------------------------------------------ properties

def test_run_to_run_bit_identity(dattn):
    """No atomics in the reductions: two identical calls give identical bits."""
    case = synth.paged_batched(2, B=16)
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    outs = []
    for _ in range(2):
        h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out,
                 write_back=False)
        outs.append(dc.out.clone())
    assert torch.equal(outs[0], outs[1])


def test_graph_replay_matches_eager(dattn):
    """Three layers captured in a CUDA graph replay to the same bits."""
    cases = [synth.hybrid_layer(2, l, 4, 1024) for l in (0, 1, 3)]
    h = dattn.Handle(8, 2, 256, [layer_dict(c) for c in cases], 4, max_context=1024)
    dcs = [DeviceCase(c) for c in cases]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l, dc in enumerate(dcs):
            h.decode(l, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out,
                     gate=dc.gate, write_back=False)
    torch.cuda.current_stream().wait_stream(s)
    eager = [dc.out.clone() for dc in dcs]
    for dc in dcs:
        dc.out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for l, dc in enumerate(dcs):
            h.decode(l, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out,
                     gate=dc.gate, write_back=False)
    g.replay()
    torch.cuda.synchronize()
    for e, dc in zip(eager, dcs):
        assert torch.equal(e, dc.out)


def test_batch_equals_alone(dattn):
    """A stream's output does not depend on the other streams of the call."""
    case = paged_case(60, 5, 8, 2, 256, 16, [300, 17, 0, 999, 64], gate=True)
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate,
             write_back=False)
    full = dc.out.clone()
    for b in range(5):
        out1 = torch.empty_like(dc.out[b:b + 1])
        desc = dattn.paged_cache(dc.k, dc.v, dc.bt[b:b + 1].contiguous(), dc.seq[b:b + 1].contiguous())
        h.decode(0, desc, dc.q[b:b + 1].contiguous(), dc.k_new[b:b + 1].contiguous(),
                 dc.v_new[b:b + 1].contiguous(), dc.pos[b:b + 1].contiguous(), out1,
                 gate=dc.gate[b:b + 1].contiguous(), write_back=False)
        # the split plan depends on B, so agreement is to rounding, not bits
        assert torch.allclose(out1, full[b:b + 1], atol=1e-5, rtol=1e-5)


# ------------------------------------------------------------------ failures stay on the host

def test_bad_page_id_is_reported_not_faulted(dattn):
    case = paged_case(70, 2, 8, 2, 256, 16, [100, 40])
    case.cache.block_table[1, 1] = 10 ** 6  # outside the pool
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out)
    assert h.get_error() == dattn.EINDEX
    assert h.get_error() == dattn.OK  # the status is cleared once read


def test_length_above_bound_is_reported(dattn):
    case = paged_case(71, 2, 8, 2, 256, 16, [100, 40])
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, max_seq_len=64)
    assert h.get_error() == dattn.ELENGTH


def test_bad_ring_metadata_is_reported(dattn):
    case = ring_case(72, 2, 8, 2, 256, 31, [5, 31])
    case.cache.head[0] = 31  # outside [0, R)
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out)
    assert h.get_error() == dattn.EINDEX


def test_host_validation(dattn):
    case = paged_case(73, 2, 8, 2, 256, 16, [100, 40])
    dc = DeviceCase(case)
    h = make_handle(dattn, case, max_context=128)
    desc = dc.cache_desc(dattn)
    with pytest.raises(dattn.DattnError) as e:
        h.decode(0, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, max_seq_len=4096)
    assert e.value.code == dattn.EXCEEDS
    with pytest.raises(dattn.DattnError) as e:
        h.decode(5, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out)
    assert e.value.code == dattn.EINVAL
    big = torch.zeros((3, 8, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dattn.DattnError) as e:
        h.decode(0, desc, big, dc.k_new, dc.v_new, dc.pos, dc.out)
    assert e.value.code == dattn.EXCEEDS
    buf = torch.zeros(dc.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    misaligned = buf[1:1 + dc.q.numel()].view(dc.q.shape)  # 2 bytes off a 16-byte boundary
    with pytest.raises(dattn.DattnError) as e:
        h.decode(0, desc, misaligned, dc.k_new, dc.v_new, dc.pos, dc.out)
    assert e.value.code == dattn.EINVAL
    assert h.get_error() == dattn.OK
