"""CPU tests of the C ABI: the library loads, exports what include/gqa.h declares,
and rejects bad arguments before touching a GPU.  No compute call runs here."""
import ctypes
import os
import re

import pytest

from kv_cache_decode_06_b300 import gqa
from kv_cache_decode_06_b300.inputs import CONFIGS, T5XXL_SWEEP_GS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")

# Any non-null, suitably aligned address: validation never dereferences it.
FAKE = 0x10000


def declared_functions(test_hooks=False):
    """Functions the header declares; with test_hooks, those under GQA_TEST_HOOKS instead."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    hooks = "".join(re.findall(r"#ifdef GQA_TEST_HOOKS(.*?)#endif", src, flags=re.S))
    if test_hooks:
        src = hooks
    else:
        src = re.sub(r"#ifdef GQA_TEST_HOOKS.*?#endif", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z_0-9]+)\s*\(", src)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(gqa.EXPORTS)
    assert declared_functions(test_hooks=True) == sorted(gqa.TEST_HOOK_EXPORTS)


def test_library_exports_every_declared_symbol(gqa_lib):
    for name in declared_functions():
        assert hasattr(gqa_lib, name), name


def test_product_library_has_no_test_hook(gqa_lib):
    """The failure-path hook lives in the test-hooks build only."""
    for name in gqa.TEST_HOOK_EXPORTS:
        assert not hasattr(gqa_lib, name), name


def test_bench_library_exports_its_header():
    """include/gqa_bench.h is the measurement helper's header (libgqa_b300_bench.so)."""
    from kv_cache_decode_06_b300 import build_lib
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "gqa_bench.h")).read(), flags=re.S)
    declared = sorted(set(re.findall(r"\b(gqa_[a-z_0-9]+)\s*\(", src)))
    assert declared == sorted(gqa.BENCH_EXPORTS)
    build_lib.build(bench=True)
    lib = gqa.load_bench()
    for name in declared:
        assert hasattr(lib, name), name
    f = ctypes.c_uint32(0)
    assert lib.gqa_bench_stream_read(None, 1, 128, 0, ctypes.byref(f), None) == 1   # null buffer
    assert lib.gqa_bench_stream_read(FAKE, 1, 100, 0, ctypes.byref(f), None) == 1   # rows not a multiple of 128
    assert lib.gqa_bench_stream_read(FAKE + 8, 1, 128, 0, ctypes.byref(f), None) == 1   # misaligned


def test_test_hooks_library_exports_the_hook():
    from kv_cache_decode_06_b300 import build_lib
    build_lib.build(test_hooks=True)
    lib = gqa.load_test_hooks()
    for name in declared_functions() + declared_functions(test_hooks=True):
        assert hasattr(lib, name), name


def test_library_does_not_link_the_oracle(gqa_lib):
    with pytest.raises(AttributeError):
        getattr(gqa_lib, "oracle_gqa_decode_f64")


def test_abi_version_matches_header(gqa_lib):
    m = re.search(r"#define GQA_ABI_VERSION (\d+)", open(HEADER).read())
    assert gqa_lib.gqa_abi_version() == int(m.group(1))


def test_status_strings(gqa_lib):
    for code, name in gqa.STATUS_NAMES.items():
        assert gqa_lib.gqa_status_string(code).decode().startswith(name)
    assert gqa_lib.gqa_status_string(99) == b"unknown gqa_status"


def _ws(*shape):
    n = ctypes.c_size_t(0)
    st = gqa.load().gqa_decode_workspace_size(*shape, ctypes.byref(n))
    return st, n.value


def test_workspace_size_for_every_workload(gqa_lib):
    cfgs = [CONFIGS[k] for k in ("tiny", "mistral7b", "llama3_70b", "long_ragged")]
    cfgs += [CONFIGS["t5xxl_sweep"].with_G(G) for G in T5XXL_SWEEP_GS]
    for c in cfgs:
        st, n = _ws(c.B, c.H, c.G, c.d, c.Lmax)
        assert st == 0 and n > 0
        # partial slots: (GQA_MAX_CTAS + B*G) * n * (d + 2) floats (plus padding), plus the header
        assert n >= (1024 + c.B * c.G) * c.n * (c.d + 2) * 4
        assert n < 64 * 2 ** 20


@pytest.mark.parametrize("shape,status", [
    ((0, 8, 2, 64, 128), 1), ((1, 8, 3, 64, 128), 1), ((1, 8, 16, 64, 128), 1), ((1, 8, 2, 96, 128), 2),
    ((1, 8, 2, 64, 0), 1), ((2048, 8, 2, 64, 128), 2), ((1, 128, 1, 64, 128), 2), ((1, 8, 2, -64, 128), 1),
    ((1, 8, 2, 64, 1 << 25), 2),
    # 1024 * 4096 K/V heads * 2^17 tiles: more 128-position tiles than the kernels index (2^30)
    ((1024, 4096, 4096, 64, 1 << 24), 2), ((1024, 64, 64, 64, 1 << 24), 2),
])
def test_workspace_size_rejects(shape, status, gqa_lib):
    assert _ws(*shape)[0] == status


def _decode(lib, ptrs=None, shape=(1, 8, 2, 64, 128), scale=0.125, ws_bytes=None, opts=None):
    q, k, v, sl, out, ws = ptrs or (FAKE,) * 6
    B, H, G, d, L = shape
    if ws_bytes is None:
        ws_bytes = _ws(*shape)[1] if _ws(*shape)[0] == 0 else 1 << 30
    o = ctypes.byref(opts) if opts is not None else None
    return lib.gqa_decode_ex(q, k, v, sl, out, ws, ws_bytes, B, H, G, d, L, scale, None, o)


def test_decode_rejects_null_pointers(gqa_lib):
    for i in (0, 1, 2, 4):   # q, k_cache, v_cache, out (seq_lens may be NULL: every position valid)
        ptrs = [FAKE] * 6
        ptrs[i] = None
        assert _decode(gqa_lib, ptrs) == 1
    ptrs = [FAKE] * 6
    ptrs[5] = None
    assert _decode(gqa_lib, ptrs) == 3


def test_decode_rejects_bad_shapes_and_values(gqa_lib):
    assert _decode(gqa_lib, shape=(1, 8, 3, 64, 128)) == 1          # H % G != 0
    assert _decode(gqa_lib, shape=(1, 8, 2, 80, 128)) == 2          # unsupported head dim
    assert _decode(gqa_lib, shape=(0, 8, 2, 64, 128)) == 1          # B = 0
    assert _decode(gqa_lib, shape=(1, 8, 2, 64, 0)) == 1            # Lmax = 0
    assert _decode(gqa_lib, scale=float("nan")) == 1
    assert _decode(gqa_lib, scale=float("inf")) == 1


def test_decode_accepts_the_default_scale_sentinel(gqa_lib):
    """GQA_SCALE_DEFAULT (0) is a valid scale: the call gets past every argument check
    (here, without a GPU, to the device check) instead of being rejected."""
    m = re.search(r"#define GQA_SCALE_DEFAULT (\S+)f", open(HEADER).read())
    assert float(m.group(1)) == gqa.SCALE_DEFAULT == 0.0
    expect = 5 if not os.path.exists("/dev/nvidia0") else 0
    if expect == 5:
        assert _decode(gqa_lib, scale=gqa.SCALE_DEFAULT) == 5
        assert _decode(gqa_lib, scale=-0.5) == 5     # any finite value is used as given


def test_binding_computes_no_scale():
    """The binding only marshals: the default scale is resolved in the library."""
    src = open(os.path.join(ROOT, "kv_cache_decode_06_b300", "gqa.py")).read()
    assert "sqrt" not in src


def test_decode_rejects_misaligned_pointers(gqa_lib):
    for i in range(5):
        ptrs = [FAKE] * 6
        ptrs[i] = FAKE + 2
        assert _decode(gqa_lib, ptrs) == 1, i
    ptrs = [FAKE] * 6
    ptrs[5] = FAKE + 16
    assert _decode(gqa_lib, ptrs) == 3


def test_decode_rejects_small_workspace(gqa_lib):
    need = _ws(1, 8, 2, 64, 128)[1]
    assert _decode(gqa_lib, ws_bytes=need - 1) == 3


def test_decode_rejects_bad_options(gqa_lib):
    o = gqa.DecodeOptions(7, 0)
    assert _decode(gqa_lib, opts=o) == 1
    o = gqa.DecodeOptions(0, 5000)
    assert _decode(gqa_lib, opts=o) == 1
    o = gqa.DecodeOptions(0, 0)
    o.reserved[2] = 1
    assert _decode(gqa_lib, opts=o) == 1
    o = gqa.DecodeOptions(gqa.PATH_SIMT, 0)                          # H/G = 16 > simt limit
    assert _decode(gqa_lib, shape=(1, 32, 2, 64, 128), opts=o) == 2
    assert _decode(gqa_lib, opts=gqa.DecodeOptions(0, 0, -1)) == 1   # negative window
    assert _decode(gqa_lib, opts=gqa.DecodeOptions(gqa.PATH_SIMT, 0, 16)) == 2   # window: tensor-core path only


def _append(lib, k_new=FAKE, v_new=FAKE, seq_lens=FAKE, shape=(1, 8, 2, 64, 128)):
    B, H, G, d, L = shape
    ws_bytes = _ws(*shape)[1]
    return lib.gqa_decode_append(FAKE, k_new, v_new, FAKE, FAKE, seq_lens, FAKE, FAKE, ws_bytes, B, H, G, d, L,
                                 0.125, None, None)


def test_append_rejects(gqa_lib):
    assert _append(gqa_lib, k_new=None) == 1
    assert _append(gqa_lib, v_new=None) == 1
    assert _append(gqa_lib, seq_lens=None) == 1      # the append position needs the lengths
    assert _append(gqa_lib, k_new=FAKE + 8) == 1     # rows are copied in 16-byte units
    assert _append(gqa_lib, shape=(1, 8, 3, 64, 128)) == 1


def _paged(lib, table=FAKE, seq_lens=FAKE, k_new=None, v_new=None, page_size=16, max_pages=8, num_pages=64,
           G=2, d=64, opts=None):
    B, H = 1, 8
    ws_bytes = _ws(B, H, G, d, max(1, max_pages * page_size))[1] if max_pages * page_size <= (1 << 24) else 1 << 30
    return lib.gqa_decode_paged(FAKE, FAKE, FAKE, table, seq_lens, k_new, v_new, FAKE, FAKE, ws_bytes, B, H, G, d,
                                page_size, max_pages, num_pages, 0.125, None,
                                ctypes.byref(opts) if opts is not None else None)


def test_paged_rejects(gqa_lib):
    assert _paged(gqa_lib, table=None) == 1
    for ps in (0, 8, 24, 100, 1 << 21):              # powers of two from 16 to 2^20 only
        assert _paged(gqa_lib, page_size=ps) == 1, ps
    assert _paged(gqa_lib, max_pages=0) == 1
    assert _paged(gqa_lib, num_pages=0) == 1
    assert _paged(gqa_lib, k_new=FAKE) == 1          # k_new without v_new
    assert _paged(gqa_lib, k_new=FAKE, v_new=FAKE, seq_lens=None) == 1
    assert _paged(gqa_lib, table=FAKE + 2) == 1      # misaligned table
    assert _paged(gqa_lib, page_size=1 << 20, max_pages=32) == 2         # capacity above 2^24 positions
    assert _paged(gqa_lib, num_pages=1 << 30, G=2) == 2                  # pool rows above 2^31
    assert _paged(gqa_lib, opts=gqa.DecodeOptions(gqa.PATH_SIMT, 0)) == 2   # tensor-core path only


def test_select_path(gqa_lib):
    assert gqa_lib.gqa_decode_select_path(16, 32, 8, 128, 4096) in (gqa.PATH_SIMT, gqa.PATH_TCGEN05)
    assert gqa_lib.gqa_decode_select_path(1, 8, 3, 64, 128) == -1
    assert gqa_lib.gqa_decode_select_path(1, 8, 2, 96, 128) == -2


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="checks the no-GPU answer")
def test_decode_without_gpu_reports_device(gqa_lib):
    assert _decode(gqa_lib) == 5


def test_meanpool_rejects(gqa_lib):
    lib = gqa_lib
    assert lib.gqa_meanpool_kv(None, FAKE, 8, 2, 64, 512, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, None, 8, 2, 64, 512, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 3, 64, 512, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 16, 64, 512, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 2, 0, 512, None) == 1
    assert lib.gqa_meanpool_kv_strided(FAKE, FAKE, 0, 8, 2, 64, None) == 1
    assert lib.gqa_meanpool_kv_strided(FAKE + 2, FAKE, 1, 8, 2, 64, None) == 1
    assert lib.gqa_meanpool_kv_strided(FAKE, FAKE + 2, 1, 8, 2, 64, None) == 1   # w_out not 4-byte aligned
    assert lib.gqa_meanpool_kv_strided(FAKE, FAKE, 1, 8, 2, 0, None) == 1
    assert lib.gqa_meanpool_kv_strided(FAKE, FAKE, 1, 8, 2, -4, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 2, 64, 0, None) == 1                 # d_model <= 0
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 2, -1, 512, None) == 1
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 0, 1, 64, 512, None) == 1               # H <= 0
    assert lib.gqa_meanpool_kv(FAKE, FAKE, 8, 0, 64, 512, None) == 1               # G <= 0
    assert lib.gqa_meanpool_kv(FAKE, FAKE, -8, -2, 64, 512, None) == 1


def test_read_flags_rejects(gqa_lib):
    f = ctypes.c_uint32(0)
    assert gqa_lib.gqa_decode_read_flags(None, ctypes.byref(f), 0, None) == 1
    assert gqa_lib.gqa_decode_read_flags(FAKE + 8, ctypes.byref(f), 0, None) == 1


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        gqa.load(str(tmp_path / "missing.so"))


def test_binding_rejects_host_tensors():
    """Host tensors never reach the library (it takes device pointers only)."""
    import torch
    from kv_cache_decode_06_b300 import gqa
    with pytest.raises(ValueError, match="CUDA tensor"):
        gqa.meanpool_kv(torch.zeros((8, 4, 16)), 2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gqa.meanpool_kv_strided(torch.zeros((3, 8, 16)), 2)
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    kv = torch.zeros((1, 2, 128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gqa.decode(q, kv, kv, torch.full((1,), 128, dtype=torch.int32))



def test_noalloc_rejects_bad_arguments_before_queueing(gqa_lib):
    """gqa_decode_noalloc runs every host-side check before it clears its scratch header, so a
    misaligned pointer or a non-finite scale returns GQA_ERR_INVALID_ARG with nothing queued."""
    shape = (2, 8, 2, 64, 256)

    def call(q=FAKE, k=FAKE, v=FAKE, sl=FAKE, out=FAKE, scale=0.125):
        return gqa_lib.gqa_decode_noalloc(q, k, v, sl, out, *shape, scale, None)

    assert call(q=FAKE + 2) == 1
    assert call(k=FAKE + 8) == 1
    assert call(v=FAKE + 8) == 1
    assert call(out=FAKE + 4) == 1
    assert call(sl=FAKE + 2) == 1
    assert call(scale=float("nan")) == 1
    assert call(scale=float("inf")) == 1
    assert call(scale=float("-inf")) == 1
