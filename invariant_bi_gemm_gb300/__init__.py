"""Python binding of the batch-invariant GEMM library (libbi_gemm.so, C ABI in include/bi_gemm.h
and include/bi_rmsnorm.h).

Argument marshalling only: every step of y = x·W (and of the RMSNorm) runs in the CUDA kernels of
``csrc/``.  PyTorch supplies device memory and streams.  There is no CPU or
PyTorch fallback: importing this module fails if the library has not been built
(``python -m invariant_bi_gemm_gb300.build``), and every call that the library
refuses raises ``BiGemmError``.

Low-level functions carry the C names (``bi_gemm_create``, ``bi_gemm_run``, ...,
``bi_rmsnorm_run``) and take raw device pointers; ``BiGemm`` and ``BiRmsNorm`` wrap them
for torch tensors.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

BI_BF16_OUT_BF16 = 0
BI_BF16_OUT_F32 = 1
BI_MXFP8E4M3_OUT_BF16 = 2
BI_SCALES_NONE = 0
BI_SCALES_E8M0_K32 = 1
BI_GEMM_FLAG_STATIC_W = 1

BI_GEMM_OK = 0
BI_GEMM_ERR_INVALID_ARG = -1
BI_GEMM_ERR_UNSUPPORTED = -2
BI_GEMM_ERR_ALIGNMENT = -3
BI_GEMM_ERR_CUDA = -4
BI_GEMM_ERR_OOM = -5
BI_GEMM_ERR_TIMEOUT = -6
BI_GEMM_ERR_SCRATCH_LIMIT = -7

# every symbol include/bi_gemm.h declares
EXPORTED_SYMBOLS = (
    "bi_gemm_create", "bi_gemm_create_ex", "bi_gemm_run", "bi_gemm_get_device_error",
    "bi_gemm_destroy", "bi_gemm_get_config", "bi_gemm_workspace_size", "bi_gemm_strerror",
    "bi_gemm_version", "bi_gemm_run_noalloc", "bi_gemm_run_gathered",
)
# every symbol include/bi_rmsnorm.h declares
RMSNORM_EXPORTED_SYMBOLS = ("bi_rmsnorm_create", "bi_rmsnorm_run", "bi_rmsnorm_get_config", "bi_rmsnorm_destroy")
# every symbol include/bi_prenorm.h declares
PRENORM_EXPORTED_SYMBOLS = ("bi_prenorm_create", "bi_prenorm_run", "bi_prenorm_get_config", "bi_prenorm_destroy")
# every symbol include/bi_attention.h declares
ATTENTION_EXPORTED_SYMBOLS = ("bi_attention_create", "bi_attention_run", "bi_attention_workspace_size",
                              "bi_attention_get_device_error", "bi_attention_get_config", "bi_attention_destroy")


class BiGemmError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {bi_gemm_strerror(code)} ({code})")


class bi_gemm_scales(ctypes.Structure):
    _fields_ = [("sx", ctypes.c_void_p), ("sw", ctypes.c_void_p)]


class bi_gemm_block(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("sx", ctypes.c_void_p), ("rows", ctypes.c_int64)]


class bi_gemm_options(ctypes.Structure):
    _fields_ = [("split_k", ctypes.c_int32), ("max_ctas", ctypes.c_int32), ("timeout_ns", ctypes.c_uint64),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class bi_gemm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "block_m", "block_n", "block_k", "mma_m", "mma_n", "mma_k", "stages", "split_k",
        "num_sms", "max_ctas", "threads", "smem_bytes", "tmem_cols", "ctas_per_tile", "max_groups")]


class bi_rmsnorm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("d", "threads", "vectors_per_thread", "max_ctas", "num_sms")]


class bi_attention_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_q_heads", "num_kv_heads", "head_dim", "page_size", "split_size",
                                              "threads", "stage_positions", "max_ctas", "num_sms", "tma_pages",
                                              "ring_stages")]


class bi_prenorm_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("K", "N", "chunk", "splits", "tile_rows")]


def _load() -> ctypes.CDLL:
    path = _build.lib_path("libbi_gemm.so")
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: the CUDA library has not been built "
            "(run `python -m invariant_bi_gemm_gb300.build`); there is no fallback path")
    L = ctypes.CDLL(path)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.bi_gemm_create.argtypes = [ctypes.POINTER(P), I64, I64, I32, I32]
    L.bi_gemm_create_ex.argtypes = [ctypes.POINTER(P), I64, I64, I32, I32, ctypes.POINTER(bi_gemm_options)]
    L.bi_gemm_run.argtypes = [P, P, I64, P, ctypes.POINTER(bi_gemm_scales), P, P]
    L.bi_gemm_run_noalloc.argtypes = [P, P, I64, P, ctypes.POINTER(bi_gemm_scales), P, P]
    L.bi_gemm_run_gathered.argtypes = [P, ctypes.POINTER(bi_gemm_block), ctypes.c_int32, P, P, P, P, P, P]
    L.bi_gemm_get_device_error.argtypes = [P, P]
    L.bi_gemm_destroy.argtypes = [P]
    L.bi_gemm_get_config.argtypes = [P, ctypes.POINTER(bi_gemm_config)]
    L.bi_gemm_workspace_size.argtypes = [P, I64, ctypes.POINTER(ctypes.c_uint64)]
    L.bi_gemm_strerror.argtypes = [I32]
    L.bi_gemm_strerror.restype = ctypes.c_char_p
    L.bi_gemm_version.argtypes = []
    L.bi_rmsnorm_create.argtypes = [ctypes.POINTER(P), I64, ctypes.c_float]
    L.bi_rmsnorm_run.argtypes = [P, P, I64, P, P, P]
    L.bi_rmsnorm_get_config.argtypes = [P, ctypes.POINTER(bi_rmsnorm_config)]
    L.bi_rmsnorm_destroy.argtypes = [P]
    L.bi_attention_create.argtypes = [ctypes.POINTER(P), I64, I64, I64, I64, ctypes.c_float, I64]
    L.bi_attention_run.argtypes = [P, P, I64, P, P, P, P, I64, P, I64, I64, I64, P, P]
    L.bi_attention_workspace_size.argtypes = [P, I64, I64, ctypes.POINTER(ctypes.c_uint64)]
    L.bi_attention_get_device_error.argtypes = [P, P]
    L.bi_attention_get_config.argtypes = [P, ctypes.POINTER(bi_attention_config)]
    L.bi_attention_destroy.argtypes = [P]
    L.bi_prenorm_create.argtypes = [ctypes.POINTER(P), I64, I64, ctypes.c_float, I64]
    L.bi_prenorm_run.argtypes = [P, P, I64, P, P, P]
    L.bi_prenorm_get_config.argtypes = [P, ctypes.POINTER(bi_prenorm_config)]
    L.bi_prenorm_destroy.argtypes = [P]
    for n in ("bi_gemm_create", "bi_gemm_create_ex", "bi_gemm_run", "bi_gemm_run_noalloc", "bi_gemm_run_gathered",
              "bi_gemm_get_device_error",
              "bi_gemm_destroy", "bi_gemm_get_config", "bi_gemm_workspace_size", "bi_gemm_version") + \
            RMSNORM_EXPORTED_SYMBOLS + ATTENTION_EXPORTED_SYMBOLS + PRENORM_EXPORTED_SYMBOLS:
        getattr(L, n).restype = I32
    return L


_lib = None
LIB_PATH = _build.lib_path("libbi_gemm.so")


def library() -> ctypes.CDLL:
    """The loaded libbi_gemm.so (loaded on first use; ImportError if it was never built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != BI_GEMM_OK:
        raise BiGemmError(rc, where)


# --------------------------------------------------------------------- C names

def bi_gemm_strerror(code: int) -> str:
    return library().bi_gemm_strerror(int(code)).decode()


def bi_gemm_version() -> int:
    return library().bi_gemm_version()


def bi_gemm_create(K: int, N: int, dtype: int, scale_layout: int = BI_SCALES_NONE,
                   options: bi_gemm_options | None = None) -> int:
    """Returns the handle (an opaque integer); raises BiGemmError on refusal."""
    h = ctypes.c_void_p()
    if options is None:
        rc = library().bi_gemm_create(ctypes.byref(h), int(K), int(N), int(dtype), int(scale_layout))
    else:
        rc = library().bi_gemm_create_ex(ctypes.byref(h), int(K), int(N), int(dtype), int(scale_layout),
                                   ctypes.byref(options))
    _check(rc, "bi_gemm_create")
    return h.value


def bi_gemm_run(h: int, x: int, M: int, W: int, scales: bi_gemm_scales | None, y: int, stream: int) -> None:
    """Raw-pointer call: x, W, y device addresses, stream a cudaStream_t value."""
    rc = library().bi_gemm_run(ctypes.c_void_p(h), ctypes.c_void_p(x), int(M), ctypes.c_void_p(W),
                         ctypes.byref(scales) if scales is not None else None, ctypes.c_void_p(y),
                         ctypes.c_void_p(stream))
    _check(rc, "bi_gemm_run")


def bi_gemm_run_noalloc(h: int, x: int, M: int, W: int, scales: bi_gemm_scales | None, y: int,
                        stream: int) -> None:
    """bi_gemm_run for callers that may not allocate device memory: a split count > 1 keeps its
    scratch in the library's fixed 8 MiB per-device array; too large a run raises
    BiGemmError(BI_GEMM_ERR_SCRATCH_LIMIT).  Calls that overlap on the GPU race on that array."""
    rc = library().bi_gemm_run_noalloc(ctypes.c_void_p(h), ctypes.c_void_p(x), int(M), ctypes.c_void_p(W),
                                       ctypes.byref(scales) if scales is not None else None, ctypes.c_void_p(y),
                                       ctypes.c_void_p(stream))
    _check(rc, "bi_gemm_run_noalloc")


def bi_gemm_get_device_error(h: int, stream: int = 0) -> int:
    return library().bi_gemm_get_device_error(ctypes.c_void_p(h), ctypes.c_void_p(stream))


def bi_gemm_destroy(h: int) -> None:
    _check(library().bi_gemm_destroy(ctypes.c_void_p(h)), "bi_gemm_destroy")


def bi_gemm_get_config(h: int) -> dict:
    c = bi_gemm_config()
    _check(library().bi_gemm_get_config(ctypes.c_void_p(h), ctypes.byref(c)), "bi_gemm_get_config")
    return {n: getattr(c, n) for n, _ in bi_gemm_config._fields_}


def bi_gemm_workspace_size(h: int, M: int) -> int:
    b = ctypes.c_uint64()
    _check(library().bi_gemm_workspace_size(ctypes.c_void_p(h), int(M), ctypes.byref(b)), "bi_gemm_workspace_size")
    return b.value


def bi_rmsnorm_create(d: int, eps: float) -> int:
    """Returns the handle (an opaque integer); raises BiGemmError on refusal."""
    h = ctypes.c_void_p()
    _check(library().bi_rmsnorm_create(ctypes.byref(h), int(d), float(eps)), "bi_rmsnorm_create")
    return h.value


def bi_rmsnorm_run(h: int, x: int, M: int, g: int, y: int, stream: int) -> None:
    """Raw-pointer call: x, g, y device addresses, stream a cudaStream_t value."""
    rc = library().bi_rmsnorm_run(ctypes.c_void_p(h), ctypes.c_void_p(x), int(M), ctypes.c_void_p(g),
                                  ctypes.c_void_p(y), ctypes.c_void_p(stream))
    _check(rc, "bi_rmsnorm_run")


def bi_rmsnorm_get_config(h: int) -> dict:
    c = bi_rmsnorm_config()
    _check(library().bi_rmsnorm_get_config(ctypes.c_void_p(h), ctypes.byref(c)), "bi_rmsnorm_get_config")
    return {n: getattr(c, n) for n, _ in bi_rmsnorm_config._fields_}


def bi_rmsnorm_destroy(h: int) -> None:
    _check(library().bi_rmsnorm_destroy(ctypes.c_void_p(h)), "bi_rmsnorm_destroy")


def bi_attention_create(num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int, scale: float,
                        split_size: int = 0) -> int:
    """Returns the handle (an opaque integer); raises BiGemmError on refusal."""
    h = ctypes.c_void_p()
    _check(library().bi_attention_create(ctypes.byref(h), int(num_q_heads), int(num_kv_heads), int(head_dim),
                                         int(page_size), float(scale), int(split_size)), "bi_attention_create")
    return h.value


def bi_attention_run(h: int, q: int, T: int, q_seq: int, q_pos: int, k_cache: int, v_cache: int, num_pages: int,
                     page_table: int, num_seqs: int, max_pages: int, max_pos: int, o: int, stream: int) -> None:
    """Raw-pointer call (device addresses, stream a cudaStream_t value)."""
    V = ctypes.c_void_p
    rc = library().bi_attention_run(V(h), V(q), int(T), V(q_seq), V(q_pos), V(k_cache), V(v_cache), int(num_pages),
                                     V(page_table), int(num_seqs), int(max_pages), int(max_pos), V(o), V(stream))
    _check(rc, "bi_attention_run")


def bi_attention_get_config(h: int) -> dict:
    c = bi_attention_config()
    _check(library().bi_attention_get_config(ctypes.c_void_p(h), ctypes.byref(c)), "bi_attention_get_config")
    return {n: getattr(c, n) for n, _ in bi_attention_config._fields_}


def bi_attention_workspace_size(h: int, T: int, max_pos: int) -> int:
    b = ctypes.c_uint64()
    _check(library().bi_attention_workspace_size(ctypes.c_void_p(h), int(T), int(max_pos), ctypes.byref(b)),
           "bi_attention_workspace_size")
    return b.value


def bi_attention_get_device_error(h: int, stream: int = 0) -> int:
    return library().bi_attention_get_device_error(ctypes.c_void_p(h), ctypes.c_void_p(stream))


def bi_attention_destroy(h: int) -> None:
    _check(library().bi_attention_destroy(ctypes.c_void_p(h)), "bi_attention_destroy")


def bi_prenorm_create(K: int, N: int, eps: float, chunk: int = 0) -> int:
    """Returns the handle (an opaque integer); raises BiGemmError on refusal."""
    h = ctypes.c_void_p()
    _check(library().bi_prenorm_create(ctypes.byref(h), int(K), int(N), float(eps), int(chunk)), "bi_prenorm_create")
    return h.value


def bi_prenorm_run(h: int, x: int, M: int, W: int, y: int, stream: int) -> None:
    """Raw-pointer call: x, W, y device addresses, stream a cudaStream_t value."""
    V = ctypes.c_void_p
    _check(library().bi_prenorm_run(V(h), V(x), int(M), V(W), V(y), V(stream)), "bi_prenorm_run")


def bi_prenorm_get_config(h: int) -> dict:
    c = bi_prenorm_config()
    _check(library().bi_prenorm_get_config(ctypes.c_void_p(h), ctypes.byref(c)), "bi_prenorm_get_config")
    return {n: getattr(c, n) for n, _ in bi_prenorm_config._fields_}


def bi_prenorm_destroy(h: int) -> None:
    _check(library().bi_prenorm_destroy(ctypes.c_void_p(h)), "bi_prenorm_destroy")


# --------------------------------------------------------------------- torch wrappers

_DTYPES = {"bf16": BI_BF16_OUT_BF16, "bf16_f32": BI_BF16_OUT_F32, "mxfp8": BI_MXFP8E4M3_OUT_BF16}


class BiGemm:
    """y = x·W for fixed (K, N) on torch tensors.

    kind: "bf16" (bf16 in/out), "bf16_f32" (bf16 in, fp32 out) or "mxfp8" (E4M3 codes as
    uint8 / float8_e4m3fn tensors, E8M0 scales as uint8, bf16 out).
    """

    def __init__(self, K: int, N: int, kind: str = "bf16", split_k: int = 0, max_ctas: int = 0,
                 timeout_ns: int = 0, static_w: bool = False):
        self.K, self.N, self.kind = int(K), int(N), kind
        self.dtype = _DTYPES[kind]
        layout = BI_SCALES_E8M0_K32 if kind == "mxfp8" else BI_SCALES_NONE
        opts = None
        flags = BI_GEMM_FLAG_STATIC_W if static_w else 0
        if split_k or max_ctas or timeout_ns or flags:
            opts = bi_gemm_options(int(split_k), int(max_ctas), int(timeout_ns), flags, 0)
        self.handle = bi_gemm_create(self.K, self.N, self.dtype, layout, opts)

    @property
    def config(self) -> dict:
        return bi_gemm_get_config(self.handle)

    def out_dtype(self):
        import torch
        return torch.float32 if self.kind == "bf16_f32" else torch.bfloat16

    def run(self, x, W, y=None, sx=None, sw=None, stream=None):
        import torch
        M = int(x.shape[0])
        if x.dim() != 2 or x.shape[1] != self.K or tuple(W.shape) != (self.K, self.N):
            raise ValueError("shape mismatch: x [M, K], W [K, N] expected")
        if not (x.is_cuda and W.is_cuda and x.is_contiguous() and W.is_contiguous()):
            raise ValueError("x and W must be contiguous CUDA tensors")
        want = torch.bfloat16 if self.kind != "mxfp8" else None
        if want is not None and (x.dtype != want or W.dtype != want):
            raise ValueError("bf16 inputs expected")
        if want is None and (x.element_size() != 1 or W.element_size() != 1):
            raise ValueError("E4M3 inputs (1 byte per element) expected")
        if y is None:
            y = torch.empty((M, self.N), dtype=self.out_dtype(), device=x.device)
        if tuple(y.shape) != (M, self.N) or y.dtype != self.out_dtype() or not y.is_contiguous():
            raise ValueError("y must be a contiguous [M, N] tensor of the output dtype")
        scales = None
        if self.kind == "mxfp8":
            if sx is None or sw is None:
                raise ValueError("MXFP8 needs sx [M, K/32] and sw [K/32, N] E8M0 tensors")
            if tuple(sx.shape) != (M, self.K // 32) or tuple(sw.shape) != (self.K // 32, self.N):
                raise ValueError("scale shapes: sx [M, K/32], sw [K/32, N]")
            if sx.element_size() != 1 or sw.element_size() != 1 or not (sx.is_contiguous() and sw.is_contiguous()):
                raise ValueError("scales must be contiguous uint8 tensors")
            scales = bi_gemm_scales(sx.data_ptr(), sw.data_ptr())
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        bi_gemm_run(self.handle, x.data_ptr(), M, W.data_ptr(), scales, y.data_ptr(), s)
        return y

    __call__ = run

    def run_gathered(self, blocks, W, x_out=None, y=None, sx_blocks=None, sx_out=None, sw=None, stream=None):
        """y = concat(blocks) · W through bi_gemm_run_gathered: the row blocks (contiguous [rows, K]
        CUDA tensors, in order; for MXFP8 with their scales sx_blocks) are gathered into x_out
        (and sx_out), then multiplied with the same kernel configuration as every other row.
        Returns (y, x_out, sx_out)."""
        import torch
        nb = len(blocks)
        if nb < 1 or (sx_blocks is not None and len(sx_blocks) != nb):
            raise ValueError("one or more blocks (and one scale block per block for MXFP8)")
        fp8 = self.kind == "mxfp8"
        for b in blocks:
            if b.dim() != 2 or b.shape[1] != self.K or not (b.is_cuda and b.is_contiguous()):
                raise ValueError("blocks must be contiguous [rows, K] CUDA tensors")
        M = sum(int(b.shape[0]) for b in blocks)
        dev = blocks[0].device
        if x_out is None:
            x_out = torch.empty((M, self.K), dtype=blocks[0].dtype, device=dev)
        if fp8:
            if sx_blocks is None or sw is None:
                raise ValueError("MXFP8 needs sx_blocks and sw")
            if sx_out is None:
                sx_out = torch.empty((M, self.K // 32), dtype=torch.uint8, device=dev)
        if y is None:
            y = torch.empty((M, self.N), dtype=self.out_dtype(), device=dev)
        if tuple(x_out.shape) != (M, self.K) or tuple(y.shape) != (M, self.N):
            raise ValueError("x_out [M, K] and y [M, N] expected")
        arr = (bi_gemm_block * nb)()
        for i, b in enumerate(blocks):
            arr[i].x = b.data_ptr()
            arr[i].sx = sx_blocks[i].data_ptr() if fp8 else None
            arr[i].rows = int(b.shape[0])
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        rc = library().bi_gemm_run_gathered(ctypes.c_void_p(self.handle), arr, nb, ctypes.c_void_p(x_out.data_ptr()),
                                            ctypes.c_void_p(sx_out.data_ptr() if fp8 else None),
                                            ctypes.c_void_p(W.data_ptr()),
                                            ctypes.c_void_p(sw.data_ptr() if fp8 else None),
                                            ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(s))
        _check(rc, "bi_gemm_run_gathered")
        return y, x_out, sx_out

    def device_error(self, stream=None) -> int:
        s = 0
        if stream is not None:
            s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        return bi_gemm_get_device_error(self.handle, s)

    def workspace_size(self, M: int) -> int:
        return bi_gemm_workspace_size(self.handle, M)

    def close(self) -> None:
        if getattr(self, "handle", None):
            bi_gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BiRmsNorm:
    """y = RMSNorm(x) * g over rows of length d on torch bf16 tensors (x [M, d], g [d])."""

    def __init__(self, d: int, eps: float = 1e-6):
        self.d, self.eps = int(d), float(eps)
        self.handle = bi_rmsnorm_create(self.d, self.eps)

    @property
    def config(self) -> dict:
        return bi_rmsnorm_get_config(self.handle)

    def run(self, x, g, y=None, stream=None):
        import torch
        if x.dim() != 2 or x.shape[1] != self.d or tuple(g.shape) != (self.d,):
            raise ValueError("shape mismatch: x [M, d], g [d] expected")
        if x.dtype != torch.bfloat16 or g.dtype != torch.bfloat16:
            raise ValueError("bf16 inputs expected")
        if not (x.is_cuda and g.is_cuda and x.is_contiguous() and g.is_contiguous()):
            raise ValueError("x and g must be contiguous CUDA tensors")
        M = int(x.shape[0])
        if y is None:
            y = torch.empty((M, self.d), dtype=torch.bfloat16, device=x.device)
        if tuple(y.shape) != (M, self.d) or y.dtype != torch.bfloat16 or not y.is_contiguous():
            raise ValueError("y must be a contiguous [M, d] bf16 tensor")
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        bi_rmsnorm_run(self.handle, x.data_ptr(), M, g.data_ptr(), y.data_ptr(), s)
        return y

    __call__ = run

    def close(self) -> None:
        if getattr(self, "handle", None):
            bi_rmsnorm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BiAttention:
    """Batch-invariant decode attention over a paged KV cache on torch tensors.

    q [T, Hq, D] bf16; k_cache, v_cache [pages, page_size, Hkv, D] bf16; page_table int32
    [num_seqs, max_pages]; q_seq, q_pos int32 [T] (request and position of each query token).
    """

    def __init__(self, num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 scale: float | None = None, split_size: int = 0):
        self.Hq, self.Hkv, self.D, self.page_size = int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size)
        self.scale = float(scale) if scale is not None else float(head_dim) ** -0.5
        self.handle = bi_attention_create(self.Hq, self.Hkv, self.D, self.page_size, self.scale, split_size)

    @property
    def config(self) -> dict:
        return bi_attention_get_config(self.handle)

    def run(self, q, q_seq, q_pos, k_cache, v_cache, page_table, max_pos: int, o=None, stream=None):
        import torch
        T = int(q.shape[0])
        if q.dim() != 3 or q.shape[1] != self.Hq or q.shape[2] != self.D:
            raise ValueError("q must be [T, num_q_heads, head_dim]")
        if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (self.page_size, self.Hkv, self.D) or \
                v_cache.shape != k_cache.shape:
            raise ValueError("k_cache, v_cache must be [pages, page_size, num_kv_heads, head_dim]")
        for name, tns in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
            if tns.dtype != torch.bfloat16 or not tns.is_cuda or not tns.is_contiguous():
                raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
        for name, tns in (("q_seq", q_seq), ("q_pos", q_pos), ("page_table", page_table)):
            if tns.dtype != torch.int32 or not tns.is_cuda or not tns.is_contiguous():
                raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
        if tuple(q_seq.shape) != (T,) or tuple(q_pos.shape) != (T,) or page_table.dim() != 2:
            raise ValueError("q_seq, q_pos [T]; page_table [num_seqs, max_pages]")
        if o is None:
            o = torch.empty_like(q)
        if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
            raise ValueError("o must be a contiguous bf16 tensor shaped like q")
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        bi_attention_run(self.handle, q.data_ptr(), T, q_seq.data_ptr(), q_pos.data_ptr(), k_cache.data_ptr(),
                         v_cache.data_ptr(), int(k_cache.shape[0]), page_table.data_ptr(), int(page_table.shape[0]),
                         int(page_table.shape[1]), int(max_pos), o.data_ptr(), s)
        return o

    __call__ = run

    def device_error(self, stream=None) -> int:
        s = 0
        if stream is not None:
            s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        return bi_attention_get_device_error(self.handle, s)

    def workspace_size(self, T: int, max_pos: int) -> int:
        return bi_attention_workspace_size(self.handle, T, max_pos)

    def close(self) -> None:
        if getattr(self, "handle", None):
            bi_attention_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class BiPreNorm:
    """mHC pre-norm projection y = RMSNorm(x) . W (fp32 out) on torch tensors: x [M, K] bf16,
    W [K, N] bf16 (a norm weight folded into W's rows)."""

    def __init__(self, K: int, N: int, eps: float = 1e-6, chunk: int = 0):
        self.K, self.N, self.eps = int(K), int(N), float(eps)
        self.handle = bi_prenorm_create(self.K, self.N, self.eps, chunk)

    @property
    def config(self) -> dict:
        return bi_prenorm_get_config(self.handle)

    def run(self, x, W, y=None, stream=None):
        import torch
        if x.dim() != 2 or x.shape[1] != self.K or tuple(W.shape) != (self.K, self.N):
            raise ValueError("shape mismatch: x [M, K], W [K, N] expected")
        if x.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
            raise ValueError("bf16 inputs expected")
        if not (x.is_cuda and W.is_cuda and x.is_contiguous() and W.is_contiguous()):
            raise ValueError("x and W must be contiguous CUDA tensors")
        M = int(x.shape[0])
        if y is None:
            y = torch.empty((M, self.N), dtype=torch.float32, device=x.device)
        if tuple(y.shape) != (M, self.N) or y.dtype != torch.float32 or not y.is_contiguous():
            raise ValueError("y must be a contiguous [M, N] fp32 tensor")
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        bi_prenorm_run(self.handle, x.data_ptr(), M, W.data_ptr(), y.data_ptr(), s)
        return y

    __call__ = run

    def close(self) -> None:
        if getattr(self, "handle", None):
            bi_prenorm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


__all__ = [
    "BiPreNorm", "bi_prenorm_create", "bi_prenorm_run", "bi_prenorm_get_config", "bi_prenorm_destroy",
    "bi_prenorm_config", "PRENORM_EXPORTED_SYMBOLS",
    "BiAttention", "bi_attention_create", "bi_attention_run", "bi_attention_get_config", "bi_attention_workspace_size",
    "bi_attention_get_device_error", "bi_attention_destroy", "bi_attention_config", "ATTENTION_EXPORTED_SYMBOLS",
    "BiRmsNorm", "bi_rmsnorm_create", "bi_rmsnorm_run", "bi_rmsnorm_get_config", "bi_rmsnorm_destroy",
    "bi_rmsnorm_config", "RMSNORM_EXPORTED_SYMBOLS",
    "BiGemm", "BiGemmError", "bi_gemm_create", "bi_gemm_run", "bi_gemm_run_noalloc", "bi_gemm_get_device_error",
    "bi_gemm_destroy", "bi_gemm_get_config", "bi_gemm_workspace_size", "bi_gemm_strerror",
    "bi_gemm_version", "bi_gemm_scales", "bi_gemm_options", "bi_gemm_block", "EXPORTED_SYMBOLS", "LIB_PATH", "library",
]
