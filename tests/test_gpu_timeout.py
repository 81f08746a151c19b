"""A bounded device wait that runs out ends the call with DATTN_ETIMEOUT.

Every mbarrier wait in the decode kernel has a time limit. With the testing
aid dattn_debug_config(DATTN_DEBUG_WITHHOLD_Q, 200 us), the kernel's helper
warp withholds the first rotated query of its CTA, so the streaming warps'
waits for it run out after 200 microseconds: they record the timeout, let the
copies they issued land, and the kernel returns. Nothing faults, traps or
hangs. The handle then works normally again (the next call matches the oracle).
One stream with one KV head and 40 cached keys is planned as a single CTA.
"""
import time

import pytest
import torch

import synth
from gpu_util import DeviceCase, assert_close, make_handle, oracle_decode

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports_timeout(oracle):
    import decode_attention_kv_dattn_gb300 as dattn
    gen = synth.generator(900)
    cache = synth.ring_cache(gen, 1, 1, 256, 61, [40])
    x = synth.decode_inputs(gen, 1, 4, 1, 256, [40], gate=True)
    case = synth.DecodeCase(4, 1, 256, synth.RopeSpec(256, 1e4), cache, x)
    dc = DeviceCase(case)
    h = make_handle(dattn, case)
    desc = dc.cache_desc(dattn)
    h.debug_config(dattn.DEBUG_WITHHOLD_Q, wait_limit_us=200)
    t0 = time.perf_counter()
    h.decode(0, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate, write_back=False)
    assert h.get_error() == dattn.ETIMEOUT
    assert time.perf_counter() - t0 < 1.5, "the wait limit was not applied"
    assert h.get_error() == dattn.OK  # the status is cleared once read
    # back to normal: the same call now matches the oracle
    h.debug_config(0, 0)
    dc.out.fill_(float("nan"))
    h.decode(0, desc, dc.q, dc.k_new, dc.v_new, dc.pos, dc.out, gate=dc.gate, write_back=False)
    assert h.get_error() == dattn.OK
    ref, _, _ = oracle_decode(oracle, case)
    assert_close(dc.out.cpu().numpy(), ref, "decode after a timed-out call")
    h.close()


def test_debug_config_rejects_unknown_flags():
    import decode_attention_kv_dattn_gb300 as dattn
    assert dattn.lib.dattn_debug_config(None, 0, 0) == dattn.EINVAL
    layer = {"kind": dattn.CACHE_RING, "ring_slots": 7, "rotary_dim": 0, "rope_theta": 0.0}
    h = dattn.Handle(2, 1, 128, [layer], 1)
    assert dattn.lib.dattn_debug_config(h.ptr, 1 << 5, 0) == dattn.EINVAL
    assert dattn.lib.dattn_debug_config(h.ptr, 0, 0) == dattn.OK
    h.close()
    torch.cuda.synchronize()
