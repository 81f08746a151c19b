"""GPU decode and verify on sharply peaked softmax, vs the fp64 oracle.

Synthetic N(0, 1) queries and keys at head_dim 256 give scores of standard
deviation about 1: a nearly flat softmax. These cases make it peaked, where
the kernels' precision choices matter - decode's hi/lo bf16 split of q and of
the probabilities and its rescale only when a running maximum moves; verify's
hi/lo bf16 q, fp16 P and its lazy rescale (threshold 2^8 in base-2 units):
  * q scaled by 8 and by 32 (exact in bf16);
  * one cached key equal to a multiple of a head's rotated query, placed early,
    mid-stream and as the last key, so that the running maximum jumps by far
    more than 2^8 after many tiles;
  * keys whose scores rise step by step along the stream (many rescales);
  * a new key (decode) or a window key (verify) equal to a multiple of the
    query: the joined token dominates.
Inputs are built from seeded synthetic data; a rotated query is taken from
the oracle's fp64 RoPE and rounded to bf16 by torch. Outputs are compared per
element within the stated tolerance.
"""
import numpy as np
import pytest
import torch

import synth
from gpu_util import DeviceCase, assert_close, dev, make_handle, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dattn():
    import decode_attention_kv_dattn_gb300 as d
    return d


def to_bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_val(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def run_decode(dattn, oracle, case):
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    h.decode(0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate,
             write_back=False)
    assert h.get_error() == dattn.OK
    ref, _, _ = oracle_decode(oracle, case)
    err = assert_close(dc.out.cpu().numpy(), ref, "peaked decode")
    h.close()
    return err


def paged_decode_case(seed, B, n, Hq=8, Hkv=2, D=256, P=16, rope=(64, 5e6)):
    gen = synth.generator(seed)
    cache = synth.paged_cache(gen, B, Hkv, D, P, [n] * B)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, [n] * B, gate=True)
    return synth.DecodeCase(Hq, Hkv, D, synth.RopeSpec(*rope), cache, x)


def ring_decode_case(seed, B, count, Hq=8, Hkv=2, D=256, R=511):
    gen = synth.generator(seed)
    cache = synth.ring_cache(gen, B, Hkv, D, R, [count] * B)
    x = synth.decode_inputs(gen, B, Hq, Hkv, D, [count] * B, gate=True)
    return synth.DecodeCase(Hq, Hkv, D, synth.RopeSpec(256, 1e4), cache, x)


def set_paged_key(case, b, t, j, value_bits):
    c = case.cache
    c.k[c.block_table[b, t // c.P], j, t % c.P] = value_bits


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("scale", [8.0, 32.0])
@pytest.mark.parametrize("kind", ["ring", "paged"])
def test_decode_scaled_queries(dattn, oracle, scale, kind):
    case = ring_decode_case(500, 4, 511) if kind == "ring" else paged_decode_case(501, 16, 2048)
    case.inputs.q = to_bf16(bf16_val(case.inputs.q) * scale)
    run_decode(dattn, oracle, case)


def test_decode_scaled_queries_head_dim_128(dattn, oracle):
    """The paged batch's shape (16 q / 8 KV heads, head_dim 128) with q x 32."""
    case = paged_decode_case(502, 16, 1500, Hq=16, Hkv=8, D=128, rope=(128, 1e6))
    case.inputs.q = to_bf16(bf16_val(case.inputs.q) * 32.0)
    run_decode(dattn, oracle, case)


@pytest.mark.parametrize("c", [1.0, 4.0])
def test_decode_one_dominant_cached_key(dattn, oracle, c):
    """16 streams x 4096 tokens (each CTA streams many tiles per warp): stream b
    holds c times head (b % 8)'s rotated query as its key at a position that
    moves from the first token to the last across the streams."""
    B, n = 16, 4096
    case = paged_decode_case(503, B, n)
    r, th = case.rope.rotary_dim, case.rope.theta
    G = case.Hq // case.Hkv
    for b in range(B):
        h = b % case.Hq
        qr = oracle.rope_f64(case.inputs.q[b, h], r, th, int(case.inputs.pos[b]))
        t = [0, 1, 17, 255, 256, 1000, 2047, 2048, 3000, 4000, 4079, 4080, 4090, 4094, 4095, 4095][b]
        set_paged_key(case, b, t, h // G, to_bf16(c * qr))
    run_decode(dattn, oracle, case)


def test_decode_rising_scores(dattn, oracle):
    """Every 64th key of each stream is a growing multiple of one head's rotated
    query, so that head's running maximum moves again and again."""
    B, n = 8, 4096
    case = paged_decode_case(504, B, n)
    r, th = case.rope.rotary_dim, case.rope.theta
    for b in range(B):
        qr = oracle.rope_f64(case.inputs.q[b, 2 * b % 8], r, th, int(case.inputs.pos[b]))
        for t in range(0, n, 64):
            set_paged_key(case, b, t, (2 * b % 8) // 4, to_bf16(qr * (0.05 * (t // 64))))
    run_decode(dattn, oracle, case)


@pytest.mark.parametrize("kind", ["ring", "paged"])
def test_decode_dominant_new_token(dattn, oracle, kind):
    """k_new = 2 q of one head (both turned at the same position, so the score
    is 2 |q|^2 / 16): the joined token takes almost all the weight."""
    case = ring_decode_case(505, 4, 300) if kind == "ring" else paged_decode_case(506, 4, 1000)
    G = case.Hq // case.Hkv
    for b in range(4):
        h = (3 * b) % case.Hq
        case.inputs.k_new[b, h // G] = to_bf16(2.0 * bf16_val(case.inputs.q[b, h]))
    run_decode(dattn, oracle, case)


def test_decode_ring_dominant_key_in_last_block(dattn, oracle):
    """A full ring whose dominant key sits in the physical block streamed last."""
    case = ring_decode_case(507, 2, 511)
    r, th = case.rope.rotary_dim, case.rope.theta
    c = case.cache
    for b in range(2):
        qr = oracle.rope_f64(case.inputs.q[b, 1], r, th, int(case.inputs.pos[b]))
        last = (int(c.head[b]) - 1) % c.R  # the newest entry
        c.k[c.stream_rows[b], 0, last] = to_bf16(3.0 * qr)
    run_decode(dattn, oracle, case)


# ------------------------------------------------------------------ verify

def verify_case(seed, S, T, lens, Hq=24, Hkv=4, D=256, rope=(64, 5e6)):
    gen = synth.generator(seed)
    cache = synth.paged_cache(gen, S, Hkv, D, 16, lens, room=T)
    parent = np.stack([synth.tree_parents(gen, T) for _ in range(S)])
    q = synth.randn_bf16((S, T, Hq, D), gen)
    k = synth.randn_bf16((S, T, Hkv, D), gen)
    v = synth.randn_bf16((S, T, Hkv, D), gen)
    return synth.VerifyCase(Hq, Hkv, D, synth.RopeSpec(*rope), cache, q, k, v, parent, None)


def depths(parent):
    d = np.zeros(len(parent), np.int32)
    for i, p in enumerate(parent):
        d[i] = 0 if p < 0 else d[p] + 1
    return d


def run_verify(dattn, oracle, case, expect=None):
    c = case.cache
    S, T = case.q.shape[:2]
    out = torch.full((S, T, case.Hq, case.D), float("nan"), device="cuda")
    layer = {"kind": dattn.CACHE_PAGED, "page_size": c.P, "rotary_dim": case.rope.rotary_dim,
             "rope_theta": case.rope.theta}
    h = dattn.Handle(case.Hq, case.Hkv, case.D, [layer], S, max_context=int(c.seq_len.max()) or 1,
                     max_verify_rows=T)
    keep = [dev(c.k), dev(c.v), dev(c.block_table), dev(c.seq_len)]  # the descriptor holds raw pointers
    h.verify(0, dattn.paged_cache(*keep), dev(case.q), dev(case.k), dev(case.v), dev(case.parent), out,
             write_back=False)
    status = h.get_error()
    h.close()
    if expect is not None:
        assert status == expect, f"status {status}, want {expect}"
        return None
    assert status == dattn.OK
    ref, _ = oracle.verify(c.k, c.v, c.block_table, c.seq_len, case.q, case.k, case.v, case.parent,
                           case.rope.rotary_dim, case.rope.theta)
    return assert_close(out.cpu().numpy(), ref, "peaked verify")


@pytest.mark.parametrize("scale", [8.0, 32.0])
def test_verify_scaled_queries(dattn, oracle, scale):
    case = verify_case(600, 4, 16, [3000, 700, 64, 1500])
    case.q = to_bf16(bf16_val(case.q) * scale)
    run_verify(dattn, oracle, case)


def test_verify_dominant_prefix_keys(dattn, oracle):
    """For each stream a few rows get a prefix key equal to twice their rotated
    query (head 0 of the row's group for KV head 0), early, mid-prefix and as
    the prefix's last key: those rows' maxima jump by far more than 2^8."""
    case = verify_case(601, 4, 16, [4000, 2500, 900, 33])
    c = case.cache
    r, th = case.rope.rotary_dim, case.rope.theta
    for s in range(4):
        n = int(c.seq_len[s])
        dep = depths(case.parent[s])
        for i, t in ((0, n - 1), (5, n // 2), (11, 0), (15, n - 2)):
            qr = oracle.rope_f64(case.q[s, i, 0], r, th, n + int(dep[i]))
            c.k[c.block_table[s, t // c.P], 0, t % c.P] = to_bf16(2.0 * qr)
    run_verify(dattn, oracle, case)


def test_verify_dominant_window_key(dattn, oracle):
    """Row i's own window key is 2 q of one of its heads (same position): the
    tree part outweighs the whole prefix for that head."""
    case = verify_case(602, 3, 16, [2000, 100, 0])
    G = case.Hq // case.Hkv
    for s in range(3):
        for i in range(0, 16, 3):
            h = (i + s) % case.Hq
            case.k[s, i, h // G] = to_bf16(2.0 * bf16_val(case.q[s, i, h]))
    run_verify(dattn, oracle, case)


def test_verify_tiny_values_stay_within_tolerance(dattn, oracle):
    """Keys and values scaled by 2^-17 lie in fp16's subnormal range in the
    tensor-core pass; the outputs still match."""
    case = verify_case(603, 2, 16, [1200, 300])
    c = case.cache
    finite = c.k != synth.NAN_BF16
    c.k[finite] = to_bf16(bf16_val(c.k[finite]) * 2.0 ** -17)
    c.v[finite] = to_bf16(bf16_val(c.v[finite]) * 2.0 ** -17)
    run_verify(dattn, oracle, case)


def test_verify_value_beyond_fp16_is_reported(dattn):
    """A cached V value of 65536 (a bf16 number beyond fp16's range, in which
    the tensor-core pass forms P V) is reported as DATTN_ERANGE; nothing
    faults."""
    import decode_attention_kv_dattn_gb300 as d
    case = verify_case(604, 2, 8, [500, 40])
    c = case.cache
    c.v[c.block_table[0, 17 // c.P], 1, 17 % c.P, 5] = 0x4780  # 65536
    run_verify(dattn, None, case, expect=d.ERANGE)


def test_verify_large_cached_keys(dattn, oracle):
    """Keys enter the tensor cores as stored (bf16): a cached key element of
    65536 (beyond fp16's range) is scored exactly and the rows it dominates
    match the oracle."""
    case = verify_case(605, 2, 8, [500, 40])
    c = case.cache
    c.k[c.block_table[0, 17 // c.P], 1, 17 % c.P, 5] = 0x4780  # 65536
    c.k[c.block_table[1, 3 // c.P], 0, 3 % c.P, 9] = 0xC780   # -65536
    run_verify(dattn, oracle, case)
