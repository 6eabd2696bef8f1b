"""Python binding of libgqa_b300.so (ctypes).  Argument marshalling only.

Every step of the decode and of the mean-pool conversion runs in the CUDA
library; this module checks tensor properties, passes raw device pointers and
the current CUDA stream, and turns status codes into exceptions.  PyTorch is
used for device memory and streams.  If the shared library is missing the
first call raises: there is no CPU fallback.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_b300.so")
TEST_HOOKS_LIB_PATH = os.path.join(_HERE, "libgqa_b300_testhooks.so")

GQA_OK = 0
STATUS_NAMES = {0: "GQA_OK", 1: "GQA_ERR_INVALID_ARG", 2: "GQA_ERR_UNSUPPORTED", 3: "GQA_ERR_WORKSPACE",
                4: "GQA_ERR_LAUNCH", 5: "GQA_ERR_DEVICE"}
PATH_AUTO, PATH_SIMT, PATH_TCGEN05 = 0, 1, 2
FLAG_SEQ_LEN_CLAMPED = 0x1
FLAG_WAIT_TIMEOUT = 0x2
FLAG_BAD_PAGE = 0x4
SCALE_DEFAULT = 0.0   # GQA_SCALE_DEFAULT: the library then uses the pages' scale for head dim d
WORKSPACE_HEADER_BYTES = 256   # GQA_WORKSPACE_HEADER_BYTES: zero them again after a timed-out call

# Every symbol include/gqa.h declares for the product library.
EXPORTS = ("gqa_status_string", "gqa_abi_version", "gqa_decode_workspace_size", "gqa_decode", "gqa_decode_ex",
           "gqa_decode_select_path", "gqa_decode_read_flags", "gqa_meanpool_kv", "gqa_meanpool_kv_strided",
           "gqa_decode_noalloc", "gqa_decode_append", "gqa_decode_paged")
# Declared in include/gqa.h under GQA_TEST_HOOKS: exported by the test-hooks build only.
TEST_HOOK_EXPORTS = ("gqa_debug_withhold_copy",)
# Declared in include/gqa_bench.h: the measurement helper library (libgqa_b300_bench.so).
BENCH_EXPORTS = ("gqa_bench_stream_read", "gqa_bench_stream_read_pages")
BENCH_LIB_PATH = os.path.join(_HERE, "libgqa_b300_bench.so")
NOALLOC_WORKSPACE_BYTES = 8 << 20

_lock = threading.Lock()
_lib = None


class GQAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


class DecodeOptions(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("num_ctas", ctypes.c_int), ("window", ctypes.c_int),
                ("reserved", ctypes.c_int * 5)]


def load(path: Optional[str] = None):
    """Load libgqa_b300.so and declare its C signatures.  Raises if it is absent."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m kv_cache_decode_06_b300.build_lib` "
                           "(the GQA decode path has no CPU fallback)")
    with _lock:
        lib = ctypes.CDLL(p)
        V, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.gqa_status_string.restype = ctypes.c_char_p
        lib.gqa_status_string.argtypes = [I]
        lib.gqa_abi_version.restype = I
        lib.gqa_abi_version.argtypes = []
        lib.gqa_decode_workspace_size.restype = I
        lib.gqa_decode_workspace_size.argtypes = [I, I, I, I, I, ctypes.POINTER(Z)]
        lib.gqa_decode.restype = I
        lib.gqa_decode.argtypes = [V, V, V, V, V, V, Z, I, I, I, I, I, F, V]
        lib.gqa_decode_ex.restype = I
        lib.gqa_decode_ex.argtypes = [V, V, V, V, V, V, Z, I, I, I, I, I, F, V, ctypes.POINTER(DecodeOptions)]
        lib.gqa_decode_append.restype = I
        lib.gqa_decode_append.argtypes = [V, V, V, V, V, V, V, V, Z, I, I, I, I, I, F, V,
                                          ctypes.POINTER(DecodeOptions)]
        lib.gqa_decode_paged.restype = I
        lib.gqa_decode_paged.argtypes = [V, V, V, V, V, V, V, V, V, Z, I, I, I, I, I, I, I, F, V,
                                         ctypes.POINTER(DecodeOptions)]
        if hasattr(lib, "gqa_debug_withhold_copy"):   # test-hooks build only
            lib.gqa_debug_withhold_copy.restype = None
            lib.gqa_debug_withhold_copy.argtypes = [I]
        lib.gqa_decode_select_path.restype = I
        lib.gqa_decode_select_path.argtypes = [I, I, I, I, I]
        lib.gqa_decode_read_flags.restype = I
        lib.gqa_decode_read_flags.argtypes = [V, ctypes.POINTER(ctypes.c_uint32), I, V]
        lib.gqa_decode_noalloc.restype = I
        lib.gqa_decode_noalloc.argtypes = [V, V, V, V, V, I, I, I, I, I, F, V]
        lib.gqa_meanpool_kv.restype = I
        lib.gqa_meanpool_kv.argtypes = [V, V, I, I, I, I, V]
        lib.gqa_meanpool_kv_strided.restype = I
        lib.gqa_meanpool_kv_strided.argtypes = [V, V, ctypes.c_int64, I, I, ctypes.c_int64, V]
        if path is None:
            _lib = lib
    return lib


def load_test_hooks():
    """Load the test-hooks build (``build_lib --test-hooks``), which also exports
    gqa_debug_withhold_copy.  It is a separate shared object with its own device
    code; the product library is not affected."""
    if not os.path.exists(TEST_HOOKS_LIB_PATH):
        raise RuntimeError(f"{TEST_HOOKS_LIB_PATH} is missing: build it with "
                           "`python -m kv_cache_decode_06_b300.build_lib --test-hooks`")
    return load(TEST_HOOKS_LIB_PATH)


_bench_lib = None


def load_bench():
    """Load libgqa_b300_bench.so (``build_lib --bench``): the read-only stream of gqa_bench.h."""
    global _bench_lib
    if _bench_lib is not None:
        return _bench_lib
    if not os.path.exists(BENCH_LIB_PATH):
        raise RuntimeError(f"{BENCH_LIB_PATH} is missing: build it with "
                           "`python -m kv_cache_decode_06_b300.build_lib --bench`")
    with _lock:
        lib = ctypes.CDLL(BENCH_LIB_PATH)
        lib.gqa_bench_stream_read.restype = ctypes.c_int
        lib.gqa_bench_stream_read.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_int,
                                              ctypes.c_void_p, ctypes.c_void_p]
        lib.gqa_bench_stream_read_pages.restype = ctypes.c_int
        lib.gqa_bench_stream_read_pages.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_longlong,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                    ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        _bench_lib = lib
    return lib


def stream_read(buf: torch.Tensor, flags: torch.Tensor, ctas: int = 0,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Read ``buf`` (bf16 [z, rows, 128], rows a multiple of 128) once with the decode's
    TMA access pattern (gqa_bench.h); ``flags`` is a zeroed int32 [1] device tensor."""
    dev = buf.device
    _require(buf, "buf", torch.bfloat16, dev)
    if buf.dim() != 3 or buf.shape[2] != 128:
        raise ValueError("buf must be [z, rows, 128]")
    _require(flags, "flags", torch.int32, dev)
    _check(load_bench().gqa_bench_stream_read(buf.data_ptr(), buf.shape[0], buf.shape[1], int(ctas),
                                               flags.data_ptr(), _stream_handle(stream, dev)),
           "gqa_bench_stream_read")


def stream_read_pages(buf: torch.Tensor, flags: torch.Tensor, page_rows: int, lanes: int = 1, scatter: bool = True,
                      one_box: bool = False, warps: int = 1, ctas: int = 0,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """Read ``buf`` once as pages of ``page_rows`` rows: ``lanes`` issuing lanes in each of
    ``warps`` warps per block, one or two boxes per page (gqa_bench.h, gqa_bench_stream_read_pages)."""
    dev = buf.device
    _require(buf, "buf", torch.bfloat16, dev)
    if buf.dim() != 3 or buf.shape[2] != 128:
        raise ValueError("buf must be [z, rows, 128]")
    _require(flags, "flags", torch.int32, dev)
    _check(load_bench().gqa_bench_stream_read_pages(buf.data_ptr(), buf.shape[0], buf.shape[1], int(page_rows),
                                                     int(lanes), 1 if scatter else 0, 1 if one_box else 0,
                                                     int(warps), int(ctas), flags.data_ptr(),
                                                     _stream_handle(stream, dev)),
           "gqa_bench_stream_read_pages")


@contextlib.contextmanager
def using_library(lib):
    """Route this module's calls through ``lib`` (a handle from :func:`load`) inside the block."""
    global _lib
    with _lock:
        saved, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = saved


def _check(status: int, what: str) -> None:
    if status != GQA_OK:
        raise GQAError(status, what)


def _stream_handle(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _require(t: torch.Tensor, name: str, dtype: torch.dtype, device: torch.device) -> None:
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda":   # the library takes device pointers only
        raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def workspace_size(B: int, H: int, G: int, d: int, Lmax: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().gqa_decode_workspace_size(B, H, G, d, Lmax, ctypes.byref(n)), "gqa_decode_workspace_size")
    return n.value


def alloc_workspace(B: int, H: int, G: int, d: int, Lmax: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of the size gqa_decode needs (256-byte aligned by the allocator)."""
    return torch.zeros(workspace_size(B, H, G, d, Lmax), dtype=torch.uint8, device=device)


def select_path(B: int, H: int, G: int, d: int, Lmax: int) -> int:
    r = load().gqa_decode_select_path(B, H, G, d, Lmax)
    if r < 0:
        raise GQAError(-r, "gqa_decode_select_path")
    return r


def _ptr_or_null(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _prepare(q, seq_lens, out, workspace, scale, G, Lmax):
    dev = q.device
    B, H, d = q.shape
    _require(q, "q", torch.bfloat16, dev)
    if seq_lens is not None:
        if tuple(seq_lens.shape) != (B,):
            raise ValueError("seq_lens must be [B]")
        _require(seq_lens, "seq_lens", torch.int32, dev)
    if out is None:
        out = torch.empty((B, H, d), dtype=torch.float32, device=dev)
    _require(out, "out", torch.float32, dev)
    if workspace is None:
        workspace = alloc_workspace(B, H, G, d, Lmax, dev)
    _require(workspace, "workspace", torch.uint8, dev)
    if scale is None:
        scale = SCALE_DEFAULT
    return out, workspace, float(scale)


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: Optional[torch.Tensor],
           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           scale: Optional[float] = None, stream: Optional[torch.cuda.Stream] = None,
           path: int = PATH_AUTO, num_ctas: int = 0, window: int = 0) -> torch.Tensor:
    """One GQA decode step: q [B,H,d] bf16, caches [B,G,Lmax,d] bf16, seq_lens [B] int32 -> out [B,H,d] fp32.

    ``seq_lens=None`` attends to all Lmax positions (cross-attention); ``window > 0``
    to the last ``window`` valid positions only.  Enqueued on ``stream`` (default:
    the current stream); returns ``out``.  ``workspace`` must come from
    :func:`alloc_workspace` (zero-filled) and may be reused by later calls of any
    shape that fits it.  ``scale=None`` passes GQA_SCALE_DEFAULT: the library
    uses the reciprocal square root of the head dim.
    """
    dev = q.device
    B, H, d = q.shape
    Bk, G, Lmax, dk = k_cache.shape
    if Bk != B or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, k_cache and v_cache")
    _require(k_cache, "k_cache", torch.bfloat16, dev)
    _require(v_cache, "v_cache", torch.bfloat16, dev)
    out, workspace, scale = _prepare(q, seq_lens, out, workspace, scale, G, Lmax)
    opts = DecodeOptions(path, num_ctas, window)
    _check(load().gqa_decode_ex(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), _ptr_or_null(seq_lens),
                                out.data_ptr(), workspace.data_ptr(), workspace.numel(), B, H, G, d, Lmax,
                                scale, _stream_handle(stream, dev), ctypes.byref(opts)),
           "gqa_decode")
    return out


def decode_append(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, seq_lens: torch.Tensor, out: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                  stream: Optional[torch.cuda.Stream] = None, num_ctas: int = 0, window: int = 0) -> torch.Tensor:
    """Decode step with the cache append fused in: writes k_new/v_new [B,G,d] at position
    seq_lens[b] - 1 of the caches (in place) and attends over seq_lens[b] positions."""
    dev = q.device
    B, H, d = q.shape
    Bk, G, Lmax, dk = k_cache.shape
    if Bk != B or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("shape mismatch between q, k_cache and v_cache")
    if tuple(k_new.shape) != (B, G, d) or tuple(v_new.shape) != (B, G, d):
        raise ValueError("k_new and v_new must be [B, G, d]")
    for t, name in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_new, "k_new"), (v_new, "v_new")):
        _require(t, name, torch.bfloat16, dev)
    out, workspace, scale = _prepare(q, seq_lens, out, workspace, scale, G, Lmax)
    opts = DecodeOptions(0, num_ctas, window)
    _check(load().gqa_decode_append(q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                                    v_cache.data_ptr(), seq_lens.data_ptr(), out.data_ptr(),
                                    workspace.data_ptr(), workspace.numel(), B, H, G, d, Lmax, scale,
                                    _stream_handle(stream, dev), ctypes.byref(opts)),
           "gqa_decode_append")
    return out


def decode_paged(q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor, block_table: torch.Tensor,
                 seq_lens: Optional[torch.Tensor], k_new: Optional[torch.Tensor] = None,
                 v_new: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, scale: Optional[float] = None,
                 stream: Optional[torch.cuda.Stream] = None, num_ctas: int = 0, window: int = 0) -> torch.Tensor:
    """Decode step over a paged cache: pages [num_pages, G, page_size, d] bf16, block_table
    [B, max_pages] int32 (position t of sequence b is row t % page_size of page
    block_table[b, t // page_size]).  Optional fused append (k_new, v_new [B, G, d])."""
    dev = q.device
    B, H, d = q.shape
    num_pages, G, page_size, dk = k_pages.shape
    if dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("shape mismatch between q, k_pages and v_pages")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    max_pages = block_table.shape[1]
    _require(k_pages, "k_pages", torch.bfloat16, dev)
    _require(v_pages, "v_pages", torch.bfloat16, dev)
    _require(block_table, "block_table", torch.int32, dev)
    for t, name in ((k_new, "k_new"), (v_new, "v_new")):
        if t is not None:
            if tuple(t.shape) != (B, G, d):
                raise ValueError(f"{name} must be [B, G, d]")
            _require(t, name, torch.bfloat16, dev)
    out, workspace, scale = _prepare(q, seq_lens, out, workspace, scale, G, max_pages * page_size)
    opts = DecodeOptions(0, num_ctas, window)
    _check(load().gqa_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), block_table.data_ptr(),
                                   _ptr_or_null(seq_lens), _ptr_or_null(k_new), _ptr_or_null(v_new),
                                   out.data_ptr(), workspace.data_ptr(), workspace.numel(), B, H, G, d,
                                   page_size, max_pages, num_pages, scale, _stream_handle(stream, dev),
                                   ctypes.byref(opts)),
           "gqa_decode_paged")
    return out


def decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: torch.Tensor,
                   out: torch.Tensor, scale: Optional[float] = None,
                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """:func:`decode` without a workspace, for callers that cannot allocate device memory.

    The library's own scratch array (8 MiB per GPU) stands in for the
    workspace, so ``out`` must be passed in.  Calls that overlap on the GPU
    share that array and race; shapes needing more scratch raise GQAError
    (GQA_ERR_WORKSPACE).
    """
    dev = q.device
    B, H, d = q.shape
    _, G, Lmax, _ = k_cache.shape
    for t, name, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                        (v_cache, "v_cache", torch.bfloat16), (out, "out", torch.float32)):
        _require(t, name, dt, dev)
    if seq_lens is not None:
        _require(seq_lens, "seq_lens", torch.int32, dev)
    if scale is None:
        scale = SCALE_DEFAULT
    _check(load().gqa_decode_noalloc(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), _ptr_or_null(seq_lens),
                                     out.data_ptr(), B, H, G, d, Lmax, float(scale),
                                     _stream_handle(stream, dev)),
           f"gqa_decode_noalloc (scratch limit {NOALLOC_WORKSPACE_BYTES} bytes)")
    return out


def debug_withhold_copy(tile: int) -> None:
    """Test hook (test-hooks build only, see :func:`load_test_hooks`): the next decode call's
    block 0 skips its K copy number ``tile`` (see gqa.h)."""
    lib = load()
    if not hasattr(lib, "gqa_debug_withhold_copy"):
        raise RuntimeError("gqa_debug_withhold_copy is exported by the test-hooks build only")
    lib.gqa_debug_withhold_copy(int(tile))


def read_flags(workspace: torch.Tensor, clear: bool = False, stream: Optional[torch.cuda.Stream] = None) -> int:
    """GQA_FLAG_* bits recorded in ``workspace`` by earlier decode calls (synchronises the stream)."""
    f = ctypes.c_uint32(0)
    _check(load().gqa_decode_read_flags(workspace.data_ptr(), ctypes.byref(f), int(clear),
                                        _stream_handle(stream, workspace.device)), "gqa_decode_read_flags")
    return f.value


def meanpool_kv(w_in: torch.Tensor, G: int, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Mean-pool a head-major projection [H, h, d_model] fp32 into [G, h, d_model]."""
    dev = w_in.device
    _require(w_in, "w_in", torch.float32, dev)
    H, h, dm = w_in.shape
    if out is None:
        out = torch.empty((G, h, dm), dtype=torch.float32, device=dev)
    _require(out, "out", torch.float32, dev)
    if tuple(out.shape) != (G, h, dm):
        raise ValueError("out must be [G, h, d_model]")
    _check(load().gqa_meanpool_kv(w_in.data_ptr(), out.data_ptr(), H, G, h, dm, _stream_handle(stream, dev)),
           "gqa_meanpool_kv")
    return out


def meanpool_kv_strided(w_in: torch.Tensor, G: int, out: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Mean-pool heads on the middle axis: [outer, H, inner] -> [outer, G, inner]."""
    dev = w_in.device
    _require(w_in, "w_in", torch.float32, dev)
    outer, H, inner = w_in.shape
    if out is None:
        out = torch.empty((outer, G, inner), dtype=torch.float32, device=dev)
    _require(out, "out", torch.float32, dev)
    if tuple(out.shape) != (outer, G, inner):
        raise ValueError("out must be [outer, G, inner]")
    _check(load().gqa_meanpool_kv_strided(w_in.data_ptr(), out.data_ptr(), outer, H, G, inner,
                                          _stream_handle(stream, dev)), "gqa_meanpool_kv_strided")
    return out
