"""GPU parity of the decode variants (through the C ABI) against the float64 CPU oracle.

  * cross-attention: seq_lens = NULL, every one of the Lmax positions valid;
  * sliding window: the last `window` valid positions only;
  * paged cache: pages of a shared pool named by a block table;
  * fused append: the new token's K/V rows written at position seq_lens[b] - 1
    of the cache (or of its page) and attended in the same call.

Shapes cover both tensor-core layouts (d = 128; d = 64 paired, with an even
Lmax, and unpaired, with an odd one), windows that start inside, at and past
tile edges, pages smaller than, equal to and larger than a tile, and pools whose
unused pages and out-of-range table entries hold NaN and -1, which no call may
read.  Tolerance: gpu_helpers (1e-2 absolute, 2e-3 row-relative); cache writes
are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_close, to_device
from kv_cache_decode_06_b300 import gqa
from kv_cache_decode_06_b300.inputs import BF16_QNAN, DecodeConfig, f32_to_bf16_bits, make_decode_inputs
from oracle_pins import scatter_to_pages

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(gqa_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return gqa_lib


def _cfg(name, cid, B, H, G, d, Lmax):
    return DecodeConfig(name, cid, B=B, H=H, G=G, d=d, Lmax=Lmax, seq_lo=1, seq_hi=Lmax)


# (B, H, G, d, Lmax): d=128; d=64 paired (even Lmax); d=64 unpaired (odd Lmax); H/G = 4, 16 and 64
SHAPES = [(3, 32, 8, 128, 1200), (2, 16, 4, 64, 1030), (3, 8, 2, 64, 777), (2, 64, 4, 128, 600),
          (2, 64, 1, 64, 700)]   # the last: 64 heads per group at d = 64 (heads on M)


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}G{}d{}L{}".format(*s))
def test_cross_attention_all_positions(shape):
    B, H, G, d, L = shape
    cfg = _cfg("cross", 61, B, H, G, d, L)
    inp = make_decode_inputs(cfg, seq_lens=[L] * B)
    q, k, v, _ = to_device(inp)
    got = gqa.decode(q, k, v, None, scale=float(inp.scale))
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, None, inp.scale)
    check_close(got.cpu().numpy(), ref, what=f"cross {shape}")


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}G{}d{}L{}".format(*s))
def test_sliding_window(shape):
    B, H, G, d, L = shape
    cfg = _cfg("window", 62, B, H, G, d, L)
    lens = [L, L // 3 + 5, 1][:B] + [L - 1] * max(0, B - 3)
    inp = make_decode_inputs(cfg, seq_lens=lens, poison_tail=True)
    q, k, v, sl = to_device(inp)
    for W in (1, 100, 128, 129, 255, 256, 257, 513, L):
        # positions before each window hold NaN: a read of them would show up
        kp, vp = inp.k.copy(), inp.v.copy()
        for b, T in enumerate(inp.seq_lens):
            kp[b, :, :max(0, int(T) - W)] = BF16_QNAN
            vp[b, :, :max(0, int(T) - W)] = BF16_QNAN
        kd, vd = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16)
        for ctas in (0, 3):
            got = gqa.decode(q, kd, vd, sl, scale=float(inp.scale), window=W, num_ctas=ctas)
            torch.cuda.synchronize()
            ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, window=W)
            check_close(got.cpu().numpy(), ref, what=f"window {W} ctas {ctas} {shape}")


def _paged_inputs(shape, page_size, lens, seed, cid):
    B, H, G, d, L = shape
    L = -(-L // page_size) * page_size              # the capacity is whole pages
    cfg = _cfg("paged", cid, B, H, G, d, L)
    inp = make_decode_inputs(cfg, seq_lens=lens, poison_tail=True)
    (kp, vp), table = scatter_to_pages([inp.k, inp.v], inp.seq_lens, page_size, np.random.default_rng(seed))
    return cfg, inp, kp, vp, table


# page sizes are powers of two, so Lmax is even: d = 64 is paired up to H/G = 16 and
# unpaired above (H/G = 32, 64); d = 128 at H/G = 4, 16, 32 and 64 takes every softmax
# form of the paged instances, whose tiles use the page-interleaved shared-memory layout
PAGED_SHAPES = SHAPES[:3] + [(2, 64, 2, 64, 500), (2, 64, 1, 64, 500), (2, 64, 4, 128, 600),
                             (2, 64, 2, 128, 500), (1, 64, 1, 128, 700)]


@pytest.mark.parametrize("page_size", [16, 32, 64, 128, 256, 1024])
@pytest.mark.parametrize("shape", PAGED_SHAPES, ids=lambda s: "B{}H{}G{}d{}L{}".format(*s))
def test_paged_cache(shape, page_size):
    B = shape[0]
    lens = [shape[4], 1, shape[4] // 2 + 3][:B]
    cfg, inp, kp, vp, table = _paged_inputs(shape, page_size, lens, seed=page_size, cid=63)
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    sl = _dev(inp.seq_lens)
    kd, vd, td = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16), _dev(table)
    ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale)
    for ctas in (0, 2, 5):
        got = gqa.decode_paged(q, kd, vd, td, sl, workspace=ws, scale=float(inp.scale), num_ctas=ctas)
        torch.cuda.synchronize()
        check_close(got.cpu().numpy(), ref, what=f"paged ps={page_size} ctas={ctas} {shape}")
    # with a window: pages wholly before it are neither read nor looked up
    W = 3 * page_size // 2 + 7
    t2 = table.copy()
    for b, T in enumerate(inp.seq_lens):
        first = max(0, int(T) - W) // page_size
        t2[b, :first] = -1
    got = gqa.decode_paged(q, kd, vd, _dev(t2), sl, workspace=ws, scale=float(inp.scale), window=W)
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, window=W)
    check_close(got.cpu().numpy(), ref, what=f"paged window ps={page_size} {shape}")
    assert gqa.read_flags(ws) == 0


@pytest.mark.parametrize("page_size", [16, 128])
def test_paged_large_batch(page_size):
    """B = 600: T_b does not fit beside the tile prefix, so the page-id warp reads it from seq_lens."""
    shape = (600, 16, 4, 128, 256)
    lens = [(29 * i + 3) % 257 for i in range(600)]
    cfg, inp, kp, vp, table = _paged_inputs(shape, page_size, lens, seed=page_size + 1, cid=68)
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    kd, vd, td = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16), _dev(table)
    got = gqa.decode_paged(q, kd, vd, td, _dev(inp.seq_lens), scale=float(inp.scale))
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale)
    check_close(got.cpu().numpy(), ref, what=f"paged B=600 ps={page_size}")


def test_paged_cross_attention_and_bad_page_flag():
    shape = (2, 16, 4, 128, 640)
    cfg, inp, kp, vp, table = _paged_inputs(shape, 64, [640, 640], seed=5, cid=64)
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    kd, vd = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16)
    ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    got = gqa.decode_paged(q, kd, vd, _dev(table), None, workspace=ws, scale=float(inp.scale))
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, None, inp.scale)
    check_close(got.cpu().numpy(), ref, what="paged cross")
    assert gqa.read_flags(ws) == 0
    # an entry outside the pool reads zeros (keys and values 0) and is flagged
    bad = table.copy()
    bad[1, 3] = kp.shape[0] + 7
    got = gqa.decode_paged(q, kd, vd, _dev(bad), None, workspace=ws, scale=float(inp.scale))
    torch.cuda.synchronize()
    assert gqa.read_flags(ws, clear=True) & gqa.FLAG_BAD_PAGE
    k0, v0 = inp.k.copy(), inp.v.copy()
    k0[1, :, 3 * 64:4 * 64] = 0
    v0[1, :, 3 * 64:4 * 64] = 0
    ref = oracle.gqa_decode_f64(inp.q, k0, v0, None, inp.scale)
    check_close(got.cpu().numpy(), ref, what="paged bad page")


def _new_rows(cfg, seed):
    rng = np.random.default_rng(seed)
    return (f32_to_bf16_bits(rng.standard_normal((cfg.B, cfg.G, cfg.d)).astype(np.float32)),
            f32_to_bf16_bits(rng.standard_normal((cfg.B, cfg.G, cfg.d)).astype(np.float32)))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B{}H{}G{}d{}L{}".format(*s))
def test_fused_append(shape):
    B, H, G, d, L = shape
    cfg = _cfg("append", 65, B, H, G, d, L)
    lens = [L, 1, 129][:B] + [0] * max(0, B - 3)
    inp = make_decode_inputs(cfg, seq_lens=lens, poison_tail=True)
    kn, vn = _new_rows(cfg, 3)
    k_ref = oracle.append_row(inp.k, kn, inp.seq_lens)
    v_ref = oracle.append_row(inp.v, vn, inp.seq_lens)
    ref = oracle.gqa_decode_f64(inp.q, k_ref, v_ref, inp.seq_lens, inp.scale)
    for ctas, window in ((0, 0), (3, 0), (0, 100)):
        q, k, v, sl = to_device(inp)
        # the old row at T-1 holds NaN: only the appended row may be attended
        for b, T in enumerate(inp.seq_lens):
            if T > 0:
                k[b, :, T - 1] = float("nan")
                v[b, :, T - 1] = float("nan")
        got = gqa.decode_append(q, _dev(kn).view(torch.bfloat16), _dev(vn).view(torch.bfloat16), k, v, sl,
                                scale=float(inp.scale), num_ctas=ctas, window=window)
        torch.cuda.synchronize()
        r = ref if window == 0 else oracle.gqa_decode_f64(inp.q, k_ref, v_ref, inp.seq_lens, inp.scale,
                                                          window=window)
        check_close(got.cpu().numpy(), r, what=f"append ctas={ctas} window={window} {shape}")
        # the caches now hold exactly the oracle's appended caches
        assert np.array_equal(k.cpu().view(torch.int16).numpy().view(np.uint16), k_ref)
        assert np.array_equal(v.cpu().view(torch.int16).numpy().view(np.uint16), v_ref)


@pytest.mark.parametrize("page_size", [16, 128, 512])
@pytest.mark.parametrize("shape", [(3, 32, 8, 128, 1000), (3, 16, 4, 64, 1000)], ids=["d128", "d64paired"])
def test_paged_fused_append(page_size, shape):
    cfg, inp, kp, vp, table = _paged_inputs(shape, page_size, [1000, 1, 300], seed=9, cid=66)
    kn, vn = _new_rows(cfg, 4)
    k_ref = oracle.append_row(inp.k, kn, inp.seq_lens)
    v_ref = oracle.append_row(inp.v, vn, inp.seq_lens)
    ref = oracle.gqa_decode_f64(inp.q, k_ref, v_ref, inp.seq_lens, inp.scale)
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    kd, vd, td, sl = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16), _dev(table), _dev(inp.seq_lens)
    got = gqa.decode_paged(q, kd, vd, td, sl, k_new=_dev(kn).view(torch.bfloat16),
                           v_new=_dev(vn).view(torch.bfloat16), scale=float(inp.scale))
    torch.cuda.synchronize()
    check_close(got.cpu().numpy(), ref, what=f"paged append ps={page_size}")
    # the pages now hold the appended rows: gathering them gives the oracle's caches
    kg = oracle.gather_pages(kd.cpu().view(torch.int16).numpy().view(np.uint16), table, inp.seq_lens, cfg.Lmax)
    vg = oracle.gather_pages(vd.cpu().view(torch.int16).numpy().view(np.uint16), table, inp.seq_lens, cfg.Lmax)
    for b, T in enumerate(inp.seq_lens):
        assert np.array_equal(kg[b, :, :T], k_ref[b, :, :T]) and np.array_equal(vg[b, :, :T], v_ref[b, :, :T])


@pytest.mark.parametrize("page_size", [16, 256])
def test_paged_append_and_window_together(page_size):
    """All three at once: paged cache, fused append and a window, with pages before the window unlisted."""
    shape = (3, 32, 8, 128, 1000)
    cfg, inp, kp, vp, table = _paged_inputs(shape, page_size, [1000, 300, 2], seed=11, cid=67)
    kn, vn = _new_rows(cfg, 5)
    W = 333
    k_ref = oracle.append_row(inp.k, kn, inp.seq_lens)
    v_ref = oracle.append_row(inp.v, vn, inp.seq_lens)
    ref = oracle.gqa_decode_f64(inp.q, k_ref, v_ref, inp.seq_lens, inp.scale, window=W)
    t2 = table.copy()
    for b, T in enumerate(inp.seq_lens):
        t2[b, :max(0, int(T) - W) // page_size] = -1
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    kd, vd = _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16)
    ws = gqa.alloc_workspace(cfg.B, cfg.H, cfg.G, cfg.d, cfg.Lmax)
    got = gqa.decode_paged(q, kd, vd, _dev(t2), _dev(inp.seq_lens), k_new=_dev(kn).view(torch.bfloat16),
                           v_new=_dev(vn).view(torch.bfloat16), workspace=ws, scale=float(inp.scale), window=W)
    torch.cuda.synchronize()
    check_close(got.cpu().numpy(), ref, what=f"paged+append+window ps={page_size}")
    assert gqa.read_flags(ws) == 0


def test_cross_attention_on_the_cuda_core_path():
    """The CUDA-core path also takes seq_lens = NULL (it rejects only the window, paging and append)."""
    cfg = _cfg("cross_simt", 68, 2, 16, 4, 128, 700)
    inp = make_decode_inputs(cfg, seq_lens=[700, 700])
    q, k, v, _ = to_device(inp)
    got = gqa.decode(q, k, v, None, scale=float(inp.scale), path=gqa.PATH_SIMT)
    torch.cuda.synchronize()
    check_close(got.cpu().numpy(), oracle.gqa_decode_f64(inp.q, inp.k, inp.v, None, inp.scale), what="simt cross")
    with pytest.raises(gqa.GQAError):
        gqa.decode(q, k, v, to_device(inp)[3], scale=float(inp.scale), path=gqa.PATH_SIMT, window=100)


# ------------------------------------------------ full-size workloads (the benchmark's launch configuration)

from kv_cache_decode_06_b300.inputs import CONFIGS, make_new_rows, make_paged_layout  # noqa: E402


def _sample_rows(cfg, every=37):
    return np.arange(0, cfg.B * cfg.H, every, dtype=np.int64)


_MISTRAL = {}


def _mistral7b_and_oracle():
    """The Mistral-7B-shaped inputs and their float64 oracle output, computed once per session."""
    if not _MISTRAL:
        inp = make_decode_inputs(CONFIGS["mistral7b"])
        _MISTRAL["inp"] = inp
        _MISTRAL["ref"] = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale)
    return _MISTRAL["inp"], _MISTRAL["ref"]


@pytest.mark.slow
@pytest.mark.parametrize("page_size", [16, 32, 64])
def test_paged_mistral7b_full(page_size):
    """The Mistral-7B-shaped step on a paged cache in random pool order, every row, at the page
    sizes the benchmark measures (one box per page, the page-interleaved tile layout)."""
    inp, ref = _mistral7b_and_oracle()
    kp, vp, table = make_paged_layout(inp, page_size)
    q = torch.from_numpy(inp.q).view(torch.bfloat16).cuda()
    got = gqa.decode_paged(q, _dev(kp).view(torch.bfloat16), _dev(vp).view(torch.bfloat16), _dev(table),
                           _dev(inp.seq_lens), scale=float(inp.scale))
    torch.cuda.synchronize()
    check_close(got.cpu().numpy(), ref, what=f"paged mistral7b ps={page_size}")


@pytest.mark.slow
def test_append_and_window_llama3_70b_full():
    """The Llama-3-70B-shaped step with the fused append, then with a 4096-position window: sampled rows."""
    cfg = CONFIGS["llama3_70b"]
    inp = make_decode_inputs(cfg)
    rows = _sample_rows(cfg)
    kn, vn = make_new_rows(cfg)
    q, k, v, sl = to_device(inp)
    got = gqa.decode_append(q, _dev(kn).view(torch.bfloat16), _dev(vn).view(torch.bfloat16), k, v, sl,
                            scale=float(inp.scale))
    torch.cuda.synchronize()
    k_ref = oracle.append_row(inp.k, kn, inp.seq_lens)
    v_ref = oracle.append_row(inp.v, vn, inp.seq_lens)
    ref = oracle.gqa_decode_f64(inp.q, k_ref, v_ref, inp.seq_lens, inp.scale, rows=rows)
    check_close(got.cpu().numpy(), ref, rows=rows, what="append llama3_70b")
    del k_ref, v_ref
    q, k, v, sl = to_device(inp)
    got = gqa.decode(q, k, v, sl, scale=float(inp.scale), window=4096)
    torch.cuda.synchronize()
    ref = oracle.gqa_decode_f64(inp.q, inp.k, inp.v, inp.seq_lens, inp.scale, rows=rows, window=4096)
    check_close(got.cpu().numpy(), ref, rows=rows, what="window llama3_70b")
