"""Decode over fp8 (E4M3) KV caches on the GPU vs the fp64 oracle, through
the C ABI ("TensorFold PR #608" names the fp8 cache and leaves it out).

A cached K value is e4m3 * k_scale and a V value e4m3 * v_scale. Decode
scores the cache as stored and stores the new token as the E4M3 bytes nearest
entry / k_scale and v_new / v_scale, joined in score space as stored. Pools
hold random E4M3 codes in written slots and NaN bytes (0x7f) elsewhere; the
written-back bytes are compared bit for bit, outputs within the tolerance.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import assert_close, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def u8(t):
    return t.detach().cpu().numpy()


def f32(x):
    """The ABI carries the scales as fp32: the oracle gets the same values
    (E4M3's 3-bit grid turns a scale's last bit into 12.5% steps)."""
    return float(np.float32(x))


def run(dattn, oracle, gen, kind, Hq, Hkv, D, lens, rope, ks, vs, P=16, R=511, gate=True, q_mul=1.0,
        qk_norm=None):
    B = len(lens)
    ks, vs = f32(ks), f32(vs)
    if kind == "ring":
        c = synth.ring_cache(gen, B, Hkv, D, R, lens, n_rows=B + 1, stream_rows=synth.randperm(B + 1, gen)[:B])
    else:
        c = synth.paged_cache(gen, B, Hkv, D, P, lens)
    K8, V8 = synth.e4m3_pool_like(c.k, gen), synth.e4m3_pool_like(c.v, gen)
    pos = [n + 5 for n in lens] if kind == "ring" else list(lens)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, pos, gate=gate)
    if q_mul != 1.0:
        x.q = (torch.from_numpy(x.q.view(np.int16)).view(torch.bfloat16).float() * q_mul).to(
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    layer = {"kind": dattn.CACHE_RING if kind == "ring" else dattn.CACHE_PAGED, "ring_slots": R, "page_size": P,
             "rotary_dim": rope[0], "rope_theta": rope[1], "kv_format": dattn.KV_E4M3, "k_scale": ks,
             "v_scale": vs}
    if qk_norm is not None:
        layer.update(q_norm=qk_norm[0], k_norm=qk_norm[1], norm_eps=qk_norm[2])
    h = dattn.Handle(Hq, Hkv, D, [layer], B, max_context=max(max(lens), 1) if kind != "ring" else 0)
    kd, vd = dev(K8), dev(V8)
    if kind == "ring":
        keep = (dev(c.head), dev(c.count), dev(c.stream_rows))
        desc = dattn.ring_cache(kd, vd, *keep)
        ring, paged = (c.head, c.count, c.stream_rows), None
    else:
        keep = (dev(c.block_table), dev(c.seq_len))
        desc = dattn.paged_cache(kd, vd, *keep)
        ring, paged = None, (c.block_table, c.seq_len)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    h.decode(0, desc, dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.pos), out,
             gate=None if x.gate is None else dev(x.gate), write_back=True)
    assert h.get_error() == dattn.OK
    ref, ke, ve = oracle.decode_fp8(K8, V8, x.q, x.k_new, x.v_new, x.pos, rope[0], rope[1], ks, vs, gate=x.gate,
                                    ring=ring, paged=paged, qk_norm=qk_norm)
    assert_close(out.cpu().numpy(), ref, f"fp8 {kind} decode")
    # the written-back bytes, and nothing else changed
    Ke, Ve = K8.copy(), V8.copy()
    for b in range(B):
        if kind == "ring":
            Ke[c.stream_rows[b], :, c.head[b]] = ke[b]
            Ve[c.stream_rows[b], :, c.head[b]] = ve[b]
        else:
            n = int(c.seq_len[b])
            Ke[c.block_table[b, n // P], :, n % P] = ke[b]
            Ve[c.block_table[b, n // P], :, n % P] = ve[b]
    assert np.array_equal(u8(kd), Ke), f"K pool: {np.sum(u8(kd) != Ke)} bytes differ"
    assert np.array_equal(u8(vd), Ve), f"V pool: {np.sum(u8(vd) != Ve)} bytes differ"
    h.close()


def test_ring_sliding_layer(dattn, oracle):
    """The sliding layers' shape (8 q / 2 KV heads, head_dim 256, 511 slots,
    RoPE on all dims): empty, one, partial, full and nearly full rings."""
    run(dattn, oracle, synth.generator(5000), "ring", 8, 2, 256, [0, 1, 300, 511, 77, 510], (256, 1e4), 0.05, 0.07)


@pytest.mark.parametrize("Hq", [4, 16])
def test_paged_full_layer(dattn, oracle, Hq):
    """Full layers (first 64 dims rotated), G = 2 and 8, ragged lengths with
    page boundaries and an empty stream."""
    run(dattn, oracle, synth.generator(5100 + Hq), "paged", Hq, 2, 256, [0, 15, 16, 17, 1000, 3000], (64, 5e6),
        0.3, 0.02)


def test_paged_head_dim_128(dattn, oracle):
    """The paged batch's heads (16 q / 8 KV, head_dim 128, RoPE on all dims),
    64-token pages."""
    run(dattn, oracle, synth.generator(5200), "paged", 16, 8, 128, [64, 200, 1, 4096], (128, 1e6), 1.0, 1.0,
        P=64, gate=False)


def test_long_context_split(dattn, oracle):
    """One long stream split over every SM, merged across CTAs."""
    run(dattn, oracle, synth.generator(5300), "paged", 8, 2, 256, [30000], (64, 5e6), 0.125, 0.5, P=64)


def test_peaked_queries(dattn, oracle):
    """q scaled x8: the score precision of the fp16 hi/lo query terms."""
    run(dattn, oracle, synth.generator(5400), "paged", 8, 2, 256, [700, 2000], (64, 5e6), 0.25, 0.25, q_mul=8.0)


def test_with_qk_norm(dattn, oracle):
    gen = synth.generator(5500)
    w = lambda: (1.0 + 0.25 * torch.randn(256, generator=gen)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    run(dattn, oracle, gen, "ring", 8, 2, 256, [200, 511], (256, 1e4), 0.05, 0.05, qk_norm=(w(), w(), 1e-6))


@pytest.mark.parametrize("rotate", [True, False])
def test_append(dattn, oracle, rotate):
    """Appending to an E4M3 pool stores the E4M3 bytes nearest entry / k_scale
    (the bf16 entry of a rotating append, or the key as given) and
    v / v_scale."""
    gen = synth.generator(5600)
    D, Hkv, P, B, Tm = 256, 2, 16, 2, 20
    ks, vs = f32(0.04), f32(0.3)
    bt = np.array([[4, 1], [0, 3]], np.int32)
    starts, count, spos = np.array([3, 10], np.int32), np.array([20, 9], np.int32), np.array([100, 7], np.int32)
    k = synth.randn_bf16((B, Tm, Hkv, D), gen)
    v = synth.randn_bf16((B, Tm, Hkv, D), gen)
    K8 = np.full((5, Hkv, P, D), synth.NAN_E4M3, np.uint8)
    V8 = K8.copy()
    layer = {"kind": dattn.CACHE_PAGED, "page_size": P, "rotary_dim": 64, "rope_theta": 5e6,
             "kv_format": dattn.KV_E4M3, "k_scale": ks, "v_scale": vs}
    h = dattn.Handle(8, Hkv, D, [layer], B, max_context=32)
    kd, vd = dev(K8), dev(V8)
    bt_d, seq = dev(bt), torch.zeros(B, dtype=torch.int32, device="cuda")
    h.append_kv(0, dattn.paged_cache(kd, vd, bt_d, seq), dev(k), dev(v), dev(starts), dev(count),
                start_pos=dev(spos), rotate=rotate)
    assert h.get_error() == dattn.OK
    # expected: the oracle's bf16 entries, each rounded to E4M3 by the oracle
    Kb = np.full((5, Hkv, P, D), synth.NAN_BF16, np.uint16)
    Ko, Vo = oracle.append_paged(Kb, Kb.copy(), bt, starts, spos, count, k, v, 64, 5e6, rotate=rotate)
    written = Ko != synth.NAN_BF16
    val = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Ke, Ve = K8.copy(), V8.copy()
    Ke[written] = [oracle.e4m3_round(x / ks) for x in val(Ko[written])]
    Ve[written] = [oracle.e4m3_round(x / vs) for x in val(Vo[written])]
    assert np.array_equal(u8(kd), Ke), f"K pool: {np.sum(u8(kd) != Ke)} bytes differ"
    assert np.array_equal(u8(vd), Ve), f"V pool: {np.sum(u8(vd) != Ve)} bytes differ"
    h.close()


def test_fp8_layers_refuse_what_they_do_not_support(dattn):
    D, R = 128, 31
    base = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 0, "rope_theta": 0.0, "kv_format": dattn.KV_E4M3}
    for bad in ({"k_scale": 0.0, "v_scale": 1.0}, {"k_scale": 1.0, "v_scale": float("inf")}):
        with pytest.raises(dattn.DattnError) as e:
            dattn.Handle(2, 1, D, [dict(base, **bad)], 1)
        assert e.value.code == dattn.EINVAL
    h = dattn.Handle(2, 1, D, [dict(base, k_scale=1.0, v_scale=1.0)], 1, max_verify_rows=2)
    K = torch.zeros((1, 1, R, D), dtype=torch.uint8, device="cuda")
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = dattn.ring_cache(K, K, z, z)
    q = torch.zeros((1, 2, 2, D), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 2, 1, D), dtype=torch.bfloat16, device="cuda")
    par = torch.tensor([[-1, 0]], dtype=torch.int32, device="cuda")
    with pytest.raises(dattn.DattnError) as e:
        h.verify(0, desc, q, kv, kv, par, torch.empty((1, 2, 2, D), device="cuda"), write_back=False, pos=z)
    assert e.value.code == dattn.EUNSUPPORTED
    h.close()
