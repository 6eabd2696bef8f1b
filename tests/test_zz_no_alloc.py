"""gqa_decode_noalloc: the decode step for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace (a plugin that only gets its
tensors from a host framework owning all device memory, a runtime that may not
allocate after start-up, a loop that cannot pay for cudaMalloc's device
synchronisation).  For them the library carries its own scratch array.  These
tests call that entry point through the C ABI and check it against the float64
oracle and against gqa_decode with a caller workspace, twice in a row, within
the decode tolerance, and check that a call after one whose pipeline wait ran
out (the test-hooks build withholds a copy) is exact without any reset by the
caller.

This file is collected last on purpose: a run that stops at the first failure
has then already run every other test.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_close, to_device
from kv_cache_decode_06_b300 import gqa
from kv_cache_decode_06_b300.inputs import CONFIGS, DecodeConfig, make_decode_inputs

FAKE = 0x10000   # never dereferenced: the shape is rejected first


def test_noalloc_rejects_shapes_beyond_its_scratch(gqa_lib):
    """T5-XXL shape with one K/V head needs ~18 MB of scratch: refused before any GPU work."""
    c = CONFIGS["t5xxl_sweep"].with_G(1)
    assert gqa.workspace_size(c.B, c.H, c.G, c.d, c.Lmax) > gqa.NOALLOC_WORKSPACE_BYTES
    st = gqa_lib.gqa_decode_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, c.B, c.H, c.G, c.d, c.Lmax, 0.125, None)
    assert st == 3   # GQA_ERR_WORKSPACE
    assert gqa_lib.gqa_decode_noalloc(None, FAKE, FAKE, FAKE, FAKE, 1, 8, 2, 64, 128, 0.125, None) == 1


def _call_noalloc(lib, q, k, v, sl, out, cfg, scale):
    return lib.gqa_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(), out.data_ptr(),
                                  cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax, float(scale),
                                  torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("cfg", [
    CONFIGS["mistral7b"].with_(B=6),
    DecodeConfig("noalloc_ragged", 61, B=3, H=16, G=2, d=64, Lmax=700),
], ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg, gqa_lib):
    assert torch.cuda.is_available()
    inp = make_decode_inputs(cfg) if cfg.seq_hi else make_decode_inputs(cfg, seq_lens=[700, 1, 333])
    q, k, v, sl = to_device(inp)
    ref = gqa.decode(q, k, v, sl, scale=float(inp.scale)).clone()
    torch.cuda.synchronize()
    exact = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale)
    for call in range(2):   # two calls in a row share (and must reset) the scratch
        out = torch.full((cfg.B, cfg.H, cfg.d), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(gqa_lib, q, k, v, sl, out, cfg, inp.scale) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        check_close(got, ref.cpu().numpy(), what=f"noalloc call {call} vs gqa_decode")
        check_close(got, exact, what=f"noalloc call {call} vs the oracle")


@pytest.mark.gpu
def test_noalloc_recovers_after_a_timed_out_call():
    """A call whose pipeline wait runs out (the test-hooks build withholds one K copy, so a
    bounded wait gives up after about a second) leaves the scratch's counters where its
    blocks stopped; the next call clears them itself and is exact, with no reset by the
    caller (who cannot reach the scratch)."""
    from kv_cache_decode_06_b300 import build_lib
    build_lib.build(test_hooks=True)
    lib = gqa.load_test_hooks()
    cfg = CONFIGS["mistral7b"].with_(B=4)
    inp = make_decode_inputs(cfg)
    q, k, v, sl = to_device(inp)
    out = torch.zeros((cfg.B, cfg.H, cfg.d), dtype=torch.float32, device="cuda")
    with gqa.using_library(lib):
        gqa.debug_withhold_copy(1)
        t0 = time.time()
        assert _call_noalloc(lib, q, k, v, sl, out, cfg, inp.scale) == 0
        torch.cuda.synchronize()
        assert 0.5 < time.time() - t0 < 30.0
        out.fill_(float("nan"))
        assert _call_noalloc(lib, q, k, v, sl, out, cfg, inp.scale) == 0
        torch.cuda.synchronize()
    exact = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale)
    check_close(out.cpu().numpy(), exact, what="noalloc after a timed-out call")
