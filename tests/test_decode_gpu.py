"""GPU parity of gqa_decode (through the C ABI) against the float64 CPU oracle.

Inputs are the seeded workloads of kv_cache_decode_06_b300.inputs; positions
past each sequence's length hold bf16 NaN, so any read of them shows up as a
non-finite output.  The tolerance is in gpu_helpers (1e-2 absolute and 2e-3
row-relative).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_close, to_device
from kv_cache_decode_06_b300 import gqa
from kv_cache_decode_06_b300.inputs import (
    CONFIGS, T5XXL_SWEEP_GS, DecodeConfig, make_decode_inputs,
)

pytestmark = pytest.mark.gpu

PATHS = {"simt": gqa.PATH_SIMT, "tcgen05": gqa.PATH_TCGEN05}


@pytest.fixture(scope="module", autouse=True)
def _lib(gqa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gqa_lib


def supports(path, cfg):
    n = cfg.n
    if path == gqa.PATH_SIMT:
        return n <= 8
    return gqa.load() and n <= 64 and _tc_available()


def _tc_available():
    try:
        c = DecodeConfig("probe", 99, B=1, H=8, G=1, d=64, Lmax=128, seq_lo=1, seq_hi=1)
        inp = make_decode_inputs(c)
        q, k, v, sl = to_device(inp)
        gqa.decode(q, k, v, sl, path=gqa.PATH_TCGEN05)
        return True
    except gqa.GQAError as e:
        if e.status == 2:
            return False
        raise


def run(inp, path=gqa.PATH_AUTO, num_ctas=0, ws=None, out=None):
    q, k, v, sl = to_device(inp)
    o = gqa.decode(q, k, v, sl, out=out, workspace=ws, scale=float(inp.scale), path=path, num_ctas=num_ctas)
    torch.cuda.synchronize()
    return o.cpu().numpy()


def oracle_out(inp, rows=None):
    return oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, rows=rows)


# ----------------------------------------------------------- small shapes

SMALL = [
    # (B, H, G, d, Lmax, seq_lens)
    (1, 8, 2, 64, 128, [128]),
    (3, 8, 2, 64, 300, [1, 129, 300]),
    (2, 4, 4, 128, 257, [256, 257]),
    (4, 32, 8, 128, 1000, [1000, 1, 127, 513]),
    (5, 16, 2, 64, 640, [0, 640, 3, 0, 385]),
    (2, 8, 1, 128, 384, [384, 200]),
    (3, 6, 2, 128, 131, [130, 131, 2]),
    (2, 64, 8, 128, 1024, [1024, 777]),
    (2, 8, 2, 64, 257, [257, 100]),        # d = 64, odd Lmax: unpaired layout
    (3, 32, 4, 64, 1030, [1030, 513, 2]),  # d = 64, even Lmax: paired layout, odd lengths
    (2, 64, 1, 64, 515, [515, 130]),       # 64 heads per group at d = 64: heads on M
    (3, 128, 2, 64, 300, [300, 1, 64]),
    (2, 40, 1, 64, 200, [200, 77]),        # 40 heads: padded to 64
    (2, 64, 1, 128, 300, [300, 129]),      # 64 heads at d = 128
    # the largest batch (32 sequences per lane of the prefix warp), and a batch too large for
    # T_b to sit beside the tile prefix in shared memory (B > 512)
    (1024, 8, 2, 64, 130, [(37 * i) % 131 for i in range(1024)]),
    (600, 16, 4, 128, 200, [(53 * i + 7) % 201 for i in range(600)]),
]


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "B{}H{}G{}d{}L{}".format(*s[:5]))
def test_small_shapes(shape, path):
    B, H, G, d, L, seq = shape
    cfg = DecodeConfig("small", 50, B=B, H=H, G=G, d=d, Lmax=L)
    if not supports(PATHS[path], cfg):
        pytest.skip(f"{path} does not take H/G={cfg.n}")
    inp = make_decode_inputs(cfg, seq_lens=seq)
    got = run(inp, path=PATHS[path])
    check_close(got, oracle_out(inp), what=f"{path} {shape}")


@pytest.mark.parametrize("path", sorted(PATHS))
def test_split_invariance(path):
    """The answer does not depend on how the tiles are split across CTAs."""
    cfg = DecodeConfig("split", 51, B=3, H=16, G=4, d=128, Lmax=2048)
    if not supports(PATHS[path], cfg):
        pytest.skip(path)
    inp = make_decode_inputs(cfg, seq_lens=[2048, 700, 1290])
    ref = oracle_out(inp)
    outs = []
    for ctas in (1, 2, 3, 7, 37, 148, 1024):
        got = run(inp, path=PATHS[path], num_ctas=ctas)
        check_close(got, ref, what=f"{path} ctas={ctas}")
        outs.append(got)
    spread = max(np.abs(o - outs[0]).max() for o in outs)
    assert spread <= 1e-5


@pytest.mark.parametrize("shape", [
    (2, 64, 1, 64, 1030, [1030, 600]),        # 64 heads per group at d = 64: heads on M
    (3, 32, 4, 64, 1030, [1030, 515, 77]),    # d = 64, even Lmax: paired layout
    (4, 64, 8, 128, 2000, [2000, 1, 999, 1500]),
    (3, 128, 2, 128, 700, [700, 129, 640]),   # 64 heads at d = 128: chunked softmax
], ids=lambda s: "B{}H{}G{}d{}L{}".format(*s[:5]))
def test_split_invariance_layouts(shape):
    """Every layout (heads on M, paired d = 64, d = 128, chunked softmax), from a few CTAs
    to one tile per CTA, gives the oracle's answer, call after call on one workspace, and
    leaves the workspace's counters at zero."""
    B, H, G, d, L, seq = shape
    cfg = DecodeConfig("splitl", 59, B=B, H=H, G=G, d=d, Lmax=L)
    inp = make_decode_inputs(cfg, seq_lens=seq)
    ref = oracle_out(inp)
    ws = gqa.alloc_workspace(B, H, G, d, L)
    for ctas in (2, 5, 13, 64, 300, 1024):
        for rep in range(2):
            got = run(inp, path=gqa.PATH_TCGEN05, num_ctas=ctas, ws=ws)
            check_close(got, ref, what=f"{shape} ctas={ctas} rep={rep}")
    assert gqa.read_flags(ws) == 0
    hdr = ws[:gqa.WORKSPACE_HEADER_BYTES].cpu()
    assert int(hdr[4:].count_nonzero()) == 0, "counters left non-zero"


@pytest.mark.parametrize("d", [128, 64])
def test_dynamic_pool_with_empty_and_short_sequences(d):
    """Small grids (>= 64 tiles per CTA) put a quarter of the tiles in the claimed pool:
    chunks that cut short, empty-neighboured and whole segments must still merge to the
    oracle's answer.  An odd Lmax keeps d=64 off the paired form, which splits statically."""
    Lmax = 9000 if d == 128 else 9001
    cfg = DecodeConfig("pool", 57, B=8, H=8, G=2, d=d, Lmax=Lmax)
    inp = make_decode_inputs(cfg, seq_lens=[0, Lmax, 5, 0, 8192, 129, 3000, 0])
    ref = oracle_out(inp)
    outs = []
    # 1..5 CTAs: >= 64 tiles each, a pool of 4-tile chunks; 8..40: static ranges only
    for ctas in (1, 2, 3, 5, 8, 16, 30, 40):
        got = run(inp, path=gqa.PATH_TCGEN05, num_ctas=ctas)
        check_close(got, ref, what=f"pool d={d} ctas={ctas}")
        outs.append(got)
    assert max(np.abs(o - outs[0]).max() for o in outs) <= 1e-5


def test_repeated_calls_reuse_workspace():
    """A reused workspace gives bit-identical results, call after call, and no flags."""
    cfg = CONFIGS["mistral7b"].with_(B=4)
    inp = make_decode_inputs(cfg)
    q, k, v, sl = to_device(inp)
    ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    a = gqa.decode(q, k, v, sl, workspace=ws).clone()
    for _ in range(5):
        b = gqa.decode(q, k, v, sl, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert gqa.read_flags(ws) == 0


def test_default_scale_sentinel_matches_explicit_scale():
    """scale = GQA_SCALE_DEFAULT (0) makes the library use 1/sqrt(d): bit-identical to passing
    the fp32 value of 1/sqrt(d) itself, for both head dims."""
    for d in (64, 128):
        cfg = DecodeConfig("scale", 58, B=2, H=8, G=2, d=d, Lmax=300)
        inp = make_decode_inputs(cfg, seq_lens=[300, 77])
        q, k, v, sl = to_device(inp)
        a = gqa.decode(q, k, v, sl, scale=float(np.float32(1.0 / np.sqrt(d)))).clone()
        b = gqa.decode(q, k, v, sl, scale=gqa.SCALE_DEFAULT).clone()
        c = gqa.decode(q, k, v, sl).clone()   # the binding passes the sentinel
        torch.cuda.synchronize()
        assert torch.equal(a, b) and torch.equal(a, c), d
        check_close(a.cpu().numpy(), oracle_out(inp), what=f"default scale d={d}")


def test_back_to_back_calls_on_other_shapes_and_streams():
    """Decode + split-combine pairs launched back to back (programmatic serialisation, each
    kernel starting beside the previous one) never read each other's partials: alternating
    shapes on one workspace and one stream stay exact."""
    cfgs = [DecodeConfig("bb1", 55, B=3, H=16, G=4, d=128, Lmax=2048),
            DecodeConfig("bb2", 56, B=5, H=8, G=2, d=128, Lmax=700)]
    inps = [make_decode_inputs(c) for c in cfgs]
    dev = [to_device(i) for i in inps]
    refs = [oracle_out(i) for i in inps]
    ws = gqa.alloc_workspace(5, 16, 4, 128, 2048)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for rep in range(6):
            j = rep % 2
            q, k, v, sl = dev[j]
            outs.append((j, gqa.decode(q, k, v, sl, workspace=ws[:gqa.workspace_size(
                cfgs[j].B, cfgs[j].H, cfgs[j].G, cfgs[j].d, cfgs[j].Lmax)], scale=float(inps[j].scale),
                stream=s).clone()))
    s.synchronize()
    for j, o in outs:
        check_close(o.cpu().numpy(), refs[j], what=f"back to back {j}")


def test_out_of_range_seq_lens_are_clamped_and_flagged():
    cfg = DecodeConfig("clamp", 52, B=3, H=8, G=2, d=64, Lmax=256)
    inp = make_decode_inputs(cfg, seq_lens=[256, 10, 0])
    q, k, v, _ = to_device(inp)
    bad = torch.tensor([1000, 10, -5], dtype=torch.int32, device="cuda")
    ws = gqa.alloc_workspace(3, 8, 2, 64, 256)
    got = gqa.decode(q, k, v, bad, workspace=ws, scale=float(inp.scale)).cpu().numpy()
    check_close(got, oracle_out(inp), what="clamped")
    assert gqa.read_flags(ws, clear=True) == gqa.FLAG_SEQ_LEN_CLAMPED
    assert gqa.read_flags(ws) == 0


def test_guard_regions_untouched():
    """out is written exactly in [B, H, d]; canaries around it stay."""
    cfg = DecodeConfig("guard", 53, B=2, H=8, G=2, d=128, Lmax=300)
    inp = make_decode_inputs(cfg, seq_lens=[300, 0])
    q, k, v, sl = to_device(inp)
    pad = 4096
    buf = torch.full((pad + 2 * 8 * 128 + pad,), 12345.0, dtype=torch.float32, device="cuda")
    out = buf[pad:pad + 2 * 8 * 128].view(2, 8, 128)
    gqa.decode(q, k, v, sl, out=out, scale=float(inp.scale))
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 12345.0) and np.all(b[-pad:] == 12345.0)
    check_close(out.cpu().numpy(), oracle_out(inp), what="guard")


def test_all_empty_sequences_give_zero():
    cfg = DecodeConfig("empty", 54, B=3, H=8, G=2, d=64, Lmax=128)
    inp = make_decode_inputs(cfg, seq_lens=[0, 0, 0])
    got = run(inp)
    assert np.array_equal(got, np.zeros_like(got))


def test_meanpool_bit_exact_tiny_workload():
    from kv_cache_decode_06_b300.inputs import MEANPOOL_TINY, make_meanpool_input
    c = MEANPOOL_TINY
    w = make_meanpool_input(c["H"], c["G"], c["h"], c["d_model"])
    got = gqa.meanpool_kv(torch.from_numpy(w).cuda(), c["G"]).cpu().numpy()
    ref = oracle.meanpool_f32(w, c["H"], c["G"])
    assert got.shape == (2, 64, 512)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("H,G,h,dm", [(8, 8, 16, 32), (8, 1, 16, 32), (12, 4, 8, 24), (6, 2, 5, 7), (64, 8, 128, 64),
                                      (20, 2, 4, 16), (24, 2, 5, 7), (64, 4, 8, 16), (64, 1, 8, 16), (72, 1, 3, 5)])
def test_meanpool_bit_exact_shapes(H, G, h, dm):
    from kv_cache_decode_06_b300.inputs import make_meanpool_input
    w = make_meanpool_input(H, G, h, dm, config_id=7)
    got = gqa.meanpool_kv(torch.from_numpy(w).cuda(), G).cpu().numpy()
    ref = oracle.meanpool_f32(w, H, G)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("G", [8, 1])
def test_meanpool_bit_exact_t5xxl_checkpoint(G):
    """One T5-XXL-sized projection [64, 64, 4096] (64 MiB), pooled to 8 groups and to 1."""
    from kv_cache_decode_06_b300.inputs import MEANPOOL_T5XXL, make_meanpool_input
    c = MEANPOOL_T5XXL
    w = make_meanpool_input(c["H"], G, c["h"], c["d_model"], c["config_id"])
    got = gqa.meanpool_kv(torch.from_numpy(w).cuda(), G).cpu().numpy()
    ref = oracle.meanpool_f32(w, c["H"], G)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.slow
def test_meanpool_bit_exact_whole_checkpoint():
    """Every K and V projection of a T5-XXL-shaped checkpoint, 144 x [64, 64, 4096] fp32 (9.66 GB),
    pooled to 8 groups in one strided call as the benchmark times it: the first, a middle and the
    last projection bit-exact against the oracle, and the rest checked as finite means of their heads."""
    from kv_cache_decode_06_b300.inputs import MEANPOOL_T5XXL_CHECKPOINT, make_meanpool_input
    c = MEANPOOL_T5XXL_CHECKPOINT
    H, G, h, dm, outer = c["H"], c["G"], c["h"], c["d_model"], c["outer"]
    w = make_meanpool_input(H, G, h, dm, c["config_id"], outer=outer)
    dw = torch.from_numpy(w).cuda()
    got = gqa.meanpool_kv_strided(dw, G)
    torch.cuda.synchronize()
    for o in (0, outer // 2, outer - 1):
        ref = oracle.meanpool_f32(np.ascontiguousarray(w[o]).reshape(H, h, dm), H, G)
        mine = got[o].cpu().numpy().reshape(G, h, dm)
        assert np.array_equal(mine.view(np.uint32), ref.view(np.uint32)), o
    # every projection: each group's output equals the fp32 mean of its heads to within rounding
    n = H // G
    approx = dw.view(outer, G, n, h * dm).sum(dim=2, dtype=torch.float64) / n
    assert torch.allclose(got.double(), approx, rtol=0, atol=1e-5)


@pytest.mark.parametrize("H,G", [(4, 1), (16, 1), (12, 2)])
def test_meanpool_special_values(H, G):
    """Signed zeros, infinities, NaN and subnormals: the same IEEE results as the fp32 sequence."""
    rng = np.random.default_rng(H * 10 + G)
    specials = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-40, -1e-40, 3.4e38, 1.0], dtype=np.float32)
    w = specials[rng.integers(0, len(specials), size=(H, 8, 64))].astype(np.float32)
    w[:, 0, :] = -0.0                                  # every head -0.0: the mean keeps the sign
    got = gqa.meanpool_kv(torch.from_numpy(w).cuda(), G).cpu().numpy()
    ref = oracle.meanpool_f32(w, H, G)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.signbit(got[:, 0, :]))


@pytest.mark.parametrize("inner", [1, 4])
def test_meanpool_fp32_head_order(inner):
    """Heads 1e8, 1, -1e8, 1 pool to 0.25 only when summed in head order with fp32 rounding
    after every addition (reverse order gives 0, an exact sum 0.5); inner 1 takes the scalar
    kernel, inner 4 the float4 one."""
    w = np.repeat(np.array([1e8, 1.0, -1e8, 1.0], dtype=np.float32).reshape(4, 1, 1), inner, axis=2)
    got = gqa.meanpool_kv(torch.from_numpy(np.ascontiguousarray(w)).cuda(), 1).cpu().numpy()
    assert np.all(got == np.float32(0.25))


def test_meanpool_pages_layout_bit_exact():
    """The pages' [d_model, H*h] projection pooled per column block."""
    from kv_cache_decode_06_b300.inputs import make_meanpool_input
    H, G, h, dm = 8, 2, 64, 512
    w = make_meanpool_input(H, G, h, 1, outer=dm)          # [d_model, H, h] = [d_model, H*h]
    got = gqa.meanpool_kv_strided(torch.from_numpy(w).cuda(), G).cpu().numpy()
    ref = oracle.meanpool_f32(w, H, G, head_axis=1)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------ full workloads

def test_tiny_workload():
    inp = make_decode_inputs(CONFIGS["tiny"])
    for path in (gqa.PATH_AUTO, gqa.PATH_SIMT):
        check_close(run(inp, path=path), oracle_out(inp), what="tiny")


@pytest.mark.slow
def test_mistral7b_workload_full():
    inp = make_decode_inputs(CONFIGS["mistral7b"])
    check_close(run(inp), oracle_out(inp), what="mistral7b")


@pytest.mark.slow
@pytest.mark.parametrize("G", T5XXL_SWEEP_GS)
def test_t5xxl_sweep_workload(G):
    inp = make_decode_inputs(CONFIGS["t5xxl_sweep"].with_G(G))
    check_close(run(inp), oracle_out(inp), what=f"t5xxl G={G}")


@pytest.mark.slow
def test_llama3_70b_workload():
    cfg = CONFIGS["llama3_70b"]
    inp = make_decode_inputs(cfg)
    got = run(inp)
    check_close(got, oracle_out(inp), what="llama3_70b")


@pytest.mark.slow
def test_long_ragged_workload():
    inp = make_decode_inputs(CONFIGS["long_ragged"])
    check_close(run(inp), oracle_out(inp), what="long_ragged")


def test_wait_timeout_sets_flag_and_context_survives():
    """Failure detection without a fault: a K copy that is never made (test-hooks build) leaves a
    barrier that nothing completes; block 0's bounded wait runs out after about a second, the call
    sets GQA_FLAG_WAIT_TIMEOUT and returns, and after the workspace is zeroed the next call is exact."""
    import time
    from kv_cache_decode_06_b300 import build_lib
    build_lib.build(test_hooks=True)
    cfg = CONFIGS["mistral7b"].with_(B=4)
    inp = make_decode_inputs(cfg)
    q, k, v, sl = to_device(inp)
    with gqa.using_library(gqa.load_test_hooks()):
        ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
        gqa.debug_withhold_copy(1)
        t0 = time.time()
        gqa.decode(q, k, v, sl, workspace=ws, scale=float(inp.scale), path=gqa.PATH_TCGEN05)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
        assert gqa.read_flags(ws) & gqa.FLAG_WAIT_TIMEOUT
        assert 0.5 < elapsed < 30.0, elapsed
        ws.zero_()
        got = gqa.decode(q, k, v, sl, workspace=ws, scale=float(inp.scale))
        torch.cuda.synchronize()
        check_close(got.cpu().numpy(), oracle_out(inp), what="after a timed-out call")
        assert gqa.read_flags(ws) == 0
