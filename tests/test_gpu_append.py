"""GPU bulk append (dattn_append_kv) vs the fp64 oracle, through the C ABI.

The append writes prefill tokens (or a cache set-up) into ring slots or page
slots, optionally turning each key at its own position into the same bf16
entry decode writes back ("vllm-omni commits", score-space join commit: the
layer hands back the new K/V entry and the runtime drops it into its slot).
The whole pool after the call is compared bit for bit with the oracle's:
written slots hold the oracle's entries, every other slot keeps its NaN.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import dev, host_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def _nan_pool(shape):
    return np.full(shape, synth.NAN_BF16, np.uint16)


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("D,Hkv,r,theta", [(256, 2, 256, 1e4), (128, 8, 128, 1e6), (256, 4, 64, 5e6)])
def test_append_ring(dattn, oracle, rotate, D, Hkv, r, theta):
    """Three call rows mapped to permuted ring rows (two decoy rows stay NaN);
    start indices that wrap past the ring's end; one row filling the whole
    ring; one row with no tokens."""
    R, n_rows = 61, 5
    gen = synth.generator(100 + D + Hkv)
    B, Tmax = 4, R
    k = synth.randn_bf16((B, Tmax, Hkv, D), gen)
    v = synth.randn_bf16((B, Tmax, Hkv, D), gen)
    stream_rows = np.array([3, 0, 4, 1], np.int32)
    start_index = np.array([50, 0, 7, 122], np.int32)   # 50 + 20 wraps; 122 = 2 R
    count = np.array([20, R, 0, 33], np.int32)
    start_pos = np.array([1000, 0, 5, 70000], np.int32)
    Kr, Vr = _nan_pool((n_rows, Hkv, R, D)), _nan_pool((n_rows, Hkv, R, D))
    kd, vd = dev(Kr), dev(Vr)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": r, "rope_theta": theta}
    h = dattn.Handle(Hkv * 2, Hkv, D, [layer], B)
    zeros = torch.zeros(B, dtype=torch.int32, device="cuda")
    rows_d = dev(stream_rows)  # the descriptor holds raw pointers: keep the tensors alive
    desc = dattn.ring_cache(kd, vd, zeros, zeros, rows_d)
    h.append_kv(0, desc, dev(k), dev(v), dev(start_index), dev(count), start_pos=dev(start_pos),
                rotate=rotate)
    assert h.get_error() == dattn.OK
    Ko, Vo = oracle.append_ring(Kr, Vr, start_index, start_pos, count, k, v, r, theta, rotate=rotate,
                                stream_rows=stream_rows)
    assert np.array_equal(host_u16(kd), Ko), f"K pool: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo), f"V pool: {np.sum(host_u16(vd) != Vo)} elements differ"
    h.close()


@pytest.mark.parametrize("rotate", [True, False])
@pytest.mark.parametrize("D,Hkv,P,r,theta", [(256, 2, 16, 64, 5e6), (128, 8, 16, 128, 1e6),
                                             (256, 2, 64, 64, 5e6)])
def test_append_paged(dattn, oracle, rotate, D, Hkv, P, r, theta):
    """Start indices inside a page, at a page boundary and one past it; runs
    that cross several page boundaries; a row with no tokens; a permuted pool
    with NaN spare pages."""
    gen = synth.generator(200 + D + P)
    B, Tmax = 5, 3 * P + 5
    starts = np.array([0, P - 1, P, P + 1, 5], np.int32)
    count = np.array([Tmax, 2 * P + 3, 1, 0, P], np.int32)
    start_pos = np.array([0, P - 1, 4096, 17, 300000], np.int32)
    pages = [(int(s) + int(c) + P - 1) // P + 1 for s, c in zip(starts, count)]
    total = sum(pages) + 4
    perm = synth.randperm(total, gen)
    bt = np.full((B, max(pages)), -1, np.int32)
    nxt = 0
    for b in range(B):
        bt[b, :pages[b]] = perm[nxt:nxt + pages[b]]
        nxt += pages[b]
    k = synth.randn_bf16((B, Tmax, Hkv, D), gen)
    v = synth.randn_bf16((B, Tmax, Hkv, D), gen)
    Kp, Vp = _nan_pool((total, Hkv, P, D)), _nan_pool((total, Hkv, P, D))
    kd, vd = dev(Kp), dev(Vp)
    layer = {"kind": dattn.CACHE_PAGED, "page_size": P, "rotary_dim": r, "rope_theta": theta}
    h = dattn.Handle(Hkv * 2, Hkv, D, [layer], B, max_context=int(bt.shape[1] * P))
    seq = torch.zeros(B, dtype=torch.int32, device="cuda")
    bt_d = dev(bt)
    desc = dattn.paged_cache(kd, vd, bt_d, seq)
    h.append_kv(0, desc, dev(k), dev(v), dev(starts), dev(count), start_pos=dev(start_pos), rotate=rotate)
    assert h.get_error() == dattn.OK
    Ko, Vo = oracle.append_paged(Kp, Vp, bt, starts, start_pos, count, k, v, r, theta, rotate=rotate)
    assert np.array_equal(host_u16(kd), Ko), f"K pool: {np.sum(host_u16(kd) != Ko)} elements differ"
    assert np.array_equal(host_u16(vd), Vo), f"V pool: {np.sum(host_u16(vd) != Vo)} elements differ"
    h.close()


def test_append_then_decode_equals_oracle(dattn, oracle):
    """A ring filled by the append kernel (rotated entries) and then decoded
    gives the oracle's decode of the oracle-appended ring."""
    D, Hkv, Hq, R = 256, 2, 8, 511
    gen = synth.generator(300)
    B, n = 2, 300
    k = synth.randn_bf16((B, n, Hkv, D), gen)
    v = synth.randn_bf16((B, n, Hkv, D), gen)
    Kr, Vr = _nan_pool((B, Hkv, R, D)), _nan_pool((B, Hkv, R, D))
    start = np.array([400, 3], np.int32)
    count = np.array([n, n], np.int32)
    pos0 = np.zeros(B, np.int32)
    kd, vd = dev(Kr), dev(Vr)
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 256, "rope_theta": 1e4}
    h = dattn.Handle(Hq, Hkv, D, [layer], B)
    head = ((start + n) % R).astype(np.int32)
    head_d, count_d = dev(head), dev(count)
    desc = dattn.ring_cache(kd, vd, head_d, count_d)
    h.append_kv(0, desc, dev(k), dev(v), dev(start), dev(count), start_pos=dev(pos0))
    Ko, Vo = oracle.append_ring(Kr, Vr, start, pos0, count, k, v, 256, 1e4)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, [n, n], gate=True)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    h.decode(0, desc, dev(x.q), dev(x.k_new), dev(x.v_new), dev(x.pos), out, gate=dev(x.gate),
             write_back=False)
    assert h.get_error() == dattn.OK
    ref, _, _ = oracle.decode_ring(Ko, Vo, head, count, x.q, x.k_new, x.v_new, x.pos, 256, 1e4,
                                   gate=x.gate)
    from gpu_util import assert_close
    assert_close(out.cpu().numpy(), ref, "decode after append")
    h.close()


def test_append_more_than_a_ring_is_reported(dattn):
    """More tokens than ring slots in one call would write a slot twice: the
    row is refused on the device and reported as DATTN_EINDEX."""
    D, Hkv, R = 128, 2, 31
    layer = {"kind": dattn.CACHE_RING, "ring_slots": R, "rotary_dim": 0, "rope_theta": 0.0}
    h = dattn.Handle(2, Hkv, D, [layer], 1)
    Kr = torch.zeros((1, Hkv, R, D), dtype=torch.bfloat16, device="cuda")
    Vr = torch.zeros_like(Kr)
    zeros = torch.zeros(1, dtype=torch.int32, device="cuda")
    desc = dattn.ring_cache(Kr, Vr, zeros, zeros)
    k = torch.ones((1, R + 1, Hkv, D), dtype=torch.bfloat16, device="cuda")
    h.append_kv(0, desc, k, k, zeros, torch.tensor([R + 1], dtype=torch.int32, device="cuda"),
                rotate=False)
    assert h.get_error() == dattn.EINDEX
    assert torch.count_nonzero(Kr) == 0, "nothing is written for a refused row"
    h.close()
