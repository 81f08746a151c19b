"""The allocation-free decode entry point against the handle-based one.

dattn_decode_noalloc serves callers that cannot allocate device memory (their
memory belongs to a pool someone else owns, or they must not allocate inside a
latency-critical loop): its scratch is a fixed array inside the library. This
file runs last so that a failure here leaves every other test already run.
Two calls in a row (on different workloads, so the second one starts from the
first one's leftover scratch) must each match dattn_decode on the same inputs.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import DeviceCase, assert_close, make_handle

pytestmark = pytest.mark.gpu


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    import decode_attention_kv_dattn_gb300 as dattn
    cases = [synth.paged_batched(2, B=16), synth.single_sliding_layer(0)]
    prepared = []
    for case in cases:
        dc = DeviceCase(case)
        h = make_handle(dattn, case)
        desc = dc.cache_desc(dattn)
        h.decode(0, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate, write_back=False)
        assert h.get_error() == dattn.OK
        prepared.append((dc, h, desc, dc.out.clone()))
    for dc, h, desc, ref in prepared:
        out = torch.full_like(ref, float("nan"))
        args = dattn.DecodeArgs(dc.q.shape[0], dc.q.data_ptr(), dc.k_new.data_ptr(), dc.v_new.data_ptr(),
                                None if dc.gate is None else dc.gate.data_ptr(), dc.pos.data_ptr(),
                                out.data_ptr(), 0, 0)
        rc = dattn.lib.dattn_decode_noalloc(ctypes.byref(h.config), 0, ctypes.byref(desc),
                                            ctypes.byref(args), torch.cuda.current_stream().cuda_stream)
        assert rc == dattn.OK, dattn.error_string(rc)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), ref.cpu().numpy(), "noalloc vs decode")


def test_noalloc_write_back_matches_the_oracle(oracle):
    """With write-back on, the noalloc call stores the oracle's K/V entries bit
    for bit (only the new tokens' slots change) and its outputs match the
    oracle, on a ring layer and a paged layer, two calls in a row."""
    import decode_attention_kv_dattn_gb300 as dattn
    from gpu_util import check_write_back, host_u16, oracle_decode
    for case in (synth.single_sliding_layer(0), synth.paged_batched(2, B=8)):
        dc = DeviceCase(case)
        h = make_handle(dattn, case)  # only its config is used: no workspace is touched
        dattn.decode_noalloc(h.config, 0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out,
                             gate=dc.gate, write_back=True)
        torch.cuda.synchronize()
        ref, ke, ve = oracle_decode(oracle, case)
        assert_close(dc.out.cpu().numpy(), ref, "noalloc vs oracle")
        check_write_back(case, host_u16(dc.k), host_u16(dc.v), ke, ve)
        h.close()


def test_noalloc_with_qk_norm_matches_the_oracle(oracle):
    """A layer with QK-norm: the set-up kernel copies the weights from its
    parameters into the scratch array; outputs and written-back entries match
    the oracle's."""
    import decode_attention_kv_dattn_gb300 as dattn
    from gpu_util import check_write_back, host_u16, oracle_decode
    gen = torch.Generator().manual_seed(31)
    for case in (synth.single_sliding_layer(1), synth.paged_batched(3, B=8)):
        D = case.D
        w = lambda: (1.0 + 0.25 * torch.randn(D, generator=gen)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        norm = (w(), w(), 1e-6)
        dc = DeviceCase(case)
        h = make_handle(dattn, case, qk_norm=norm)
        dattn.decode_noalloc(h.config, 0, dc.cache_desc(dattn), dc.q, dc.k_new, dc.v_new, dc.pos, dc.out,
                             gate=dc.gate, write_back=True)
        torch.cuda.synchronize()
        ref, ke, ve = oracle_decode(oracle, case, qk_norm=norm)
        assert_close(dc.out.cpu().numpy(), ref, "noalloc with QK-norm vs oracle")
        check_write_back(case, host_u16(dc.k), host_u16(dc.v), ke, ve)
        h.close()


def test_noalloc_rejects_what_does_not_fit():
    """256 streams x 4 KV heads are 1024 (stream, KV head) units, more than one
    decode call takes (512): the call is refused with DATTN_EXCEEDS before
    anything is launched. Within that limit the largest call's scratch - split
    partials for 152 CTAs + 512 units of 8 heads x (256 + 2) floats, 5.4 MB -
    fits the 8 MiB array."""
    import decode_attention_kv_dattn_gb300 as dattn
    B, Hq, Hkv, D, P = 256, 32, 4, 256, 16
    layers = (dattn.LayerConfig * 1)(dattn.LayerConfig(dattn.CACHE_PAGED, 0, P, 64, 5e6))
    cfg = dattn.Config(Hq, Hkv, D, B, 64, 0, 1, layers)
    k_pool = torch.zeros((B, Hkv, P, D), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    bt = torch.arange(B, dtype=torch.int32, device="cuda").reshape(B, 1)
    seq = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    desc = dattn.paged_cache(k_pool, v_pool, bt, seq)
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    kn = torch.zeros((B, Hkv, D), dtype=torch.bfloat16, device="cuda")
    pos = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
    with pytest.raises(dattn.DattnError) as e:
        dattn.decode_noalloc(cfg, 0, desc, q, kn, kn, pos, out, max_seq_len=8)
    assert e.value.code == dattn.EXCEEDS
