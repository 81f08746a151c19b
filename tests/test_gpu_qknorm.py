"""QK-norm before RoPE on the GPU vs the fp64 oracle, through the C ABI
("pega-omni PR #4", talker kernels: RoPE with QK-norm).

Per head, y = bf16(w * x / sqrt(mean(x^2) + eps)), then RoPE turns y: for the
queries and the new key of decode (ring and paged), for every row and window
key of verify, and for the keys of a rotating append. Outputs within the
tolerance of gpu_util; the K entries written back - normalised, then rotated -
bit for bit. Weights ~ 1 + N(0, 0.25) (a trained norm's spread), inputs of
several scales (the norm removes them).
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import (DeviceCase, assert_close, check_write_back, dev, host_u16, make_handle,
                      oracle_decode)
from test_gpu_verify import run_verify, small_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def norm_weights(gen, D, sides="qk", eps=1e-6):
    def w():
        x = 1.0 + 0.25 * torch.randn(D, generator=gen)
        return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return (w() if "q" in sides else None, w() if "k" in sides else None, eps)


def scaled(a, s):
    """bf16 bits of s * a (rounded to bf16)."""
    v = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float() * s
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def run_decode(dattn, oracle, case, norm):
    dc = DeviceCase(case)
    h = make_handle(dattn, case, qk_norm=norm)
    desc = dc.cache_desc(dattn)
    h.decode(0, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate, write_back=True)
    assert h.get_error() == dattn.OK
    ref, ke, ve = oracle_decode(oracle, case, qk_norm=norm)
    assert_close(dc.out.cpu().numpy(), ref, "decode with QK-norm")
    check_write_back(case, host_u16(dc.k), host_u16(dc.v), ke, ve)
    h.close()
    return ke


@pytest.mark.parametrize("sides", ["qk", "q", "k"])
def test_ring_decode(dattn, oracle, sides):
    gen = synth.generator(2000 + len(sides))
    B, Hq, Hkv, D, R = 6, 8, 2, 256, 511
    counts = [0, 1, 300, 511, 77, 510]
    cache = synth.ring_cache(gen, B, Hkv, D, R, counts)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, [c + 3 for c in counts], gate=True)
    x.q = scaled(x.q, 7.0)      # the norm removes the scale of q
    x.k_new = scaled(x.k_new, 0.01)
    case = synth.DecodeCase(Hq, Hkv, D, synth.SLIDING_ROPE, cache, x)
    run_decode(dattn, oracle, case, norm_weights(gen, D, sides))


@pytest.mark.parametrize("G", [2, 8])
def test_paged_decode(dattn, oracle, G):
    gen = synth.generator(2100 + G)
    B, Hkv, D, P = 5, 2, 256, 16
    lens = [0, 15, 16, 1000, 4097]
    cache = synth.paged_cache(gen, B, Hkv, D, P, lens)
    x = synth.decode_inputs(gen, B, G * Hkv, Hkv, D, lens, gate=True)
    case = synth.DecodeCase(G * Hkv, Hkv, D, synth.FULL_ROPE, cache, x)
    run_decode(dattn, oracle, case, norm_weights(gen, D, eps=1e-5))


def test_paged_decode_head_dim_128(dattn, oracle):
    gen = synth.generator(2200)
    B, Hq, Hkv, D, P = 4, 16, 8, 128, 16
    lens = [64, 100, 1, 2048]
    cache = synth.paged_cache(gen, B, Hkv, D, P, lens)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, lens, gate=False)
    case = synth.DecodeCase(Hq, Hkv, D, synth.RopeSpec(128, 1e6), cache, x)
    run_decode(dattn, oracle, case, norm_weights(gen, D, eps=1e-6))


def test_verify(dattn, oracle):
    gen = synth.generator(2300)
    case = small_case(2301, 4, 16, 24, 4, 256, [700, 0, 129, 2000], gate=True)
    run_verify(dattn, oracle, case, qk_norm=norm_weights(gen, 256))


def test_verify_head_dim_128_q_only(dattn, oracle):
    gen = synth.generator(2400)
    case = small_case(2401, 3, 8, 8, 2, 128, [300, 17, 1024], rope=(128, 1e6))
    run_verify(dattn, oracle, case, qk_norm=norm_weights(gen, 128, sides="q"))


@pytest.mark.parametrize("rotate", [True, False])
def test_append(dattn, oracle, rotate):
    """Rotating appends store normalised, rotated keys; rotate=False stores
    the keys as given (they are already entries)."""
    gen = synth.generator(2500)
    D, Hkv, P = 256, 2, 16
    B, Tmax = 3, 40
    starts = np.array([0, 15, 33], np.int32)
    count = np.array([40, 17, 0], np.int32)
    start_pos = np.array([0, 900, 5], np.int32)
    pages = [(int(s) + int(c) + P - 1) // P + 1 for s, c in zip(starts, count)]
    total = sum(pages) + 2
    perm = synth.randperm(total, gen)
    bt = np.full((B, max(pages)), -1, np.int32)
    nxt = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[nxt:nxt + pages[b]]
        nxt += pages[b]
    k = scaled(synth.randn_bf16((B, Tmax, Hkv, D), gen), 3.0)
    v = synth.randn_bf16((B, Tmax, Hkv, D), gen)
    Kp = np.full((total, Hkv, P, D), synth.NAN_BF16, np.uint16)
    Vp = Kp.copy()
    norm = norm_weights(gen, D)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": P, "rotary_dim": 64, "rope_theta": 5e6,
             "q_norm": norm[0], "k_norm": norm[1], "norm_eps": norm[2]}
    h = dattn.Handle(Hkv * 4, Hkv, D, [layer], B, max_context=int(bt.shape[1] * P))
    kd, vd = dev(Kp), dev(Vp)
    bt_d, seq = dev(bt), torch.zeros(B, dtype=torch.int32, device="cuda")
    desc = dattn.paged_cache(kd, vd, bt_d, seq)
    h.append_kv(0, desc, dev(k), dev(v), dev(starts), dev(count), start_pos=dev(start_pos), rotate=rotate)
    assert h.get_error() == dattn.OK
    Ko, Vo = oracle.append_paged(Kp, Vp, bt, starts, start_pos, count, k, v, 64, 5e6, rotate=rotate,
                                 qk_norm=norm)
    assert np.array_equal(host_u16(kd), Ko), f"K pool: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo)
    h.close()


def test_handle_rejects_negative_eps(dattn):
    D = 128
    w = np.full(D, 0x3F80, np.uint16)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": 7, "rotary_dim": 0, "rope_theta": 0.0,
             "q_norm": w, "norm_eps": -1.0}
    with pytest.raises(dattn.DattnError) as e:
        dattn.Handle(2, 1, D, [layer], 1)
    assert e.value.code == dattn.EINVAL
