"""Thin ctypes binding of libq8 (include/q8.h): argument marshalling only.

Every entry point takes torch CUDA tensors, passes their device pointers and
the current (or given) CUDA stream to the C ABI, and raises ``Q8Error`` on a
non-OK status.  There is no fallback: if ``libq8.so`` is missing or a call
fails, the call raises.  Outputs may be pre-allocated by the caller or are
allocated here with torch (device memory is the only thing torch is used for).

Tensor conventions (raw bits are accepted in any 16-bit dtype):
  q  int8 [N, K]           codes
  s  16-bit [N, K/32]      binary16 scale bits (torch.float16 or int16/uint16)
  x  16-bit [M, K]         bf16 activation bits (torch.bfloat16 or int16/uint16)
  y  float32 [M, N]        (bf16 [M, N] for q8_gemm)
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq8.so")

Q8_OK = 0
Q8_ERR_ARG, Q8_ERR_ALIGN, Q8_ERR_SHAPE, Q8_ERR_WORKSPACE, Q8_ERR_ARCH, Q8_ERR_CUDA, Q8_ERR_UNSUPPORTED = range(1, 8)
Q8_DEV_NONFINITE = 0x1
Q8_DEV_SCALE_OVF = 0x2
Q8_DEV_TIMEOUT = 0x4
Q8_SKINNY_MAX_M = 32
Q8_MAX_BATCH = 64
Q8_VARIANT_AUTO, Q8_VARIANT_SIMT, Q8_VARIANT_MMA, Q8_VARIANT_BATCH_INVARIANT, Q8_VARIANT_W8A8 = 0, 1, 2, 3, 4
Q8_GEMM_TILE_AUTO, Q8_GEMM_TILE_256x128, Q8_GEMM_TILE_128x128, Q8_GEMM_TILE_64x128 = 0, 1, 2, 3
Q8_GEMM_MAX_SPLITS = 8
Q8_QUANT_EXACT, Q8_QUANT_FL32 = 0, 1

EXPORTS = ("q8_quantize_rows", "q8_gemv", "q8_gemm_skinny", "q8_linear_batch", "q8_linear_batch_ex",
           "q8_linear_batch_chained", "q8_workspace_size", "q8_linear_batch_workspace_size", "q8_linear_batch_workspace_size_ex", "q8_gemm", "q8_status_str",
           "q8_abi_version", "q8_gemm_skinny_noalloc", "q8_gemm_ex", "q8_gguf_to_planar",
           "q8_planar_to_gguf", "q8_quantize_rows_ex", "q8_selftest_wait_timeout",
           "q8_stream_read", "q8_stream_read_out_words", "q8_linear_chain", "q8_linear_chain_workspace_size",
           "q8_gemm_w8a8", "q8_gemm_w8a8_workspace_size")
Q8_NOALLOC_SCRATCH_BYTES = 4 << 20


class Q8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} (status {status})")


class LinearDesc(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("ldy", ctypes.c_int64)]


class ChainStep(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("ldy", ctypes.c_int64), ("next", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


# how the next step of a chain takes its x from this step's y
Q8_CHAIN_END = 0
Q8_CHAIN_RMSNORM = 1
Q8_CHAIN_SWIGLU_RMSNORM = 2
Q8_MAX_CHAIN = 4096

_lib = None


def lib():
    """Load libq8.so from the package directory (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m block_quantized_int8_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, SZ, U32P = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t, ctypes.c_void_p
        L.q8_quantize_rows.argtypes = [P, I64, I64, P, P, U32P, P]
        L.q8_quantize_rows_ex.argtypes = [P, I64, I64, P, P, I32, U32P, P]
        L.q8_gemv.argtypes = [P, P, I64, I64, P, P, P, SZ, U32P, P]
        L.q8_gemm_skinny.argtypes = [P, P, I64, I64, P, I64, I32, P, I64, P, SZ, U32P, P]
        L.q8_linear_batch.argtypes = [ctypes.POINTER(LinearDesc), I32, I32, P, SZ, U32P, P]
        L.q8_linear_batch_ex.argtypes = [ctypes.POINTER(LinearDesc), I32, I32, I32, P, SZ, U32P, P]
        L.q8_linear_batch_chained.argtypes = [ctypes.POINTER(LinearDesc), I32, I32, P, SZ, U32P, P]
        L.q8_workspace_size.argtypes = [I64, I64, I32]
        L.q8_workspace_size.restype = SZ
        L.q8_linear_batch_workspace_size.argtypes = [ctypes.POINTER(LinearDesc), I32, I32]
        L.q8_linear_batch_workspace_size.restype = SZ
        L.q8_linear_batch_workspace_size_ex.argtypes = [ctypes.POINTER(LinearDesc), I32, I32, I32]
        L.q8_linear_batch_workspace_size_ex.restype = SZ
        L.q8_linear_chain.argtypes = [ctypes.POINTER(ChainStep), I32, I32, P, SZ, U32P, P]
        L.q8_linear_chain_workspace_size.argtypes = [ctypes.POINTER(ChainStep), I32, I32]
        L.q8_linear_chain_workspace_size.restype = SZ
        L.q8_gemm_w8a8.argtypes = [P, P, I64, I64, P, I64, I32, P, I64, P, SZ, U32P, P]
        L.q8_gemm_w8a8_workspace_size.argtypes = [I64, I64, I32]
        L.q8_gemm_w8a8_workspace_size.restype = SZ
        L.q8_gemm.argtypes = [P, P, I64, I64, P, I64, I32, P, I64, U32P, P]
        L.q8_gemm_ex.argtypes = [P, P, I64, I64, P, I64, I32, P, I64, I32, I32, U32P, P]
        L.q8_gemm_skinny_noalloc.argtypes = [P, P, I64, I64, P, I64, I32, P, I64, U32P, P]
        L.q8_gguf_to_planar.argtypes = [P, I64, I64, P, P, P]
        L.q8_planar_to_gguf.argtypes = [P, P, I64, I64, P, P]
        L.q8_selftest_wait_timeout.argtypes = [ctypes.c_uint64, U32P, P, P]
        L.q8_selftest_wait_timeout.restype = ctypes.c_int
        L.q8_stream_read.argtypes = [P, SZ, P, P]
        L.q8_stream_read.restype = ctypes.c_int
        L.q8_stream_read_out_words.restype = SZ
        L.q8_status_str.argtypes = [ctypes.c_int]
        L.q8_status_str.restype = ctypes.c_char_p
        L.q8_abi_version.restype = I32
        for name in ("q8_quantize_rows", "q8_quantize_rows_ex", "q8_gemv", "q8_gemm_skinny", "q8_linear_batch",
                     "q8_linear_batch_ex", "q8_linear_batch_chained", "q8_gguf_to_planar",
                     "q8_planar_to_gguf", "q8_gemm", "q8_gemm_ex", "q8_gemm_skinny_noalloc", "q8_linear_chain", "q8_gemm_w8a8"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def status_str(st: int) -> str:
    return lib().q8_status_str(int(st)).decode()


def _check(st: int, what: str):
    if st != Q8_OK:
        raise Q8Error(st, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(t, name, dtypes, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    return t


_B16 = (torch.bfloat16, torch.float16, torch.int16, torch.uint16)


def workspace(nbytes: int, device=None) -> torch.Tensor | None:
    """A zeroed workspace of ``nbytes`` (None if 0).  Zero once, reuse freely."""
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


# ---------------------------------------------------------------------------
def q8_quantize_rows(w, q=None, s=None, dev_status=None, stream=None, mode=Q8_QUANT_EXACT):
    """Q8_0-quantize float32 w[rows, K] -> (q int8 [rows, K], s float16 [rows, K/32]);
    ``mode`` picks the code rule (Q8_QUANT_EXACT or Q8_QUANT_FL32)."""
    _cuda(w, "w", (torch.float32,), 2)
    if not w.is_contiguous():
        raise ValueError("w must be contiguous")
    rows, K = w.shape
    if q is None:
        q = torch.empty((rows, K), dtype=torch.int8, device=w.device)
    if s is None:
        s = torch.empty((rows, max(K // 32, 0)), dtype=torch.float16, device=w.device)
    st = lib().q8_quantize_rows_ex(_p(w), rows, K, _p(q), _p(s), int(mode), _p(dev_status), _stream(stream))
    _check(st, "q8_quantize_rows")
    return q, s


def q8_gguf_to_planar(blocks, rows: int, K: int, q=None, s=None, stream=None):
    """GGUF Q8_0 bytes (uint8, rows * K/32 blocks of 34 bytes) -> (q int8 [rows, K],
    s float16 [rows, K/32])."""
    _cuda(blocks, "blocks", (torch.uint8,))
    if not blocks.is_contiguous() or blocks.numel() != rows * (K // 32) * 34:
        raise ValueError("blocks must be contiguous and hold rows * K/32 blocks of 34 bytes")
    if q is None:
        q = torch.empty((rows, K), dtype=torch.int8, device=blocks.device)
    if s is None:
        s = torch.empty((rows, K // 32), dtype=torch.float16, device=blocks.device)
    st = lib().q8_gguf_to_planar(_p(blocks), rows, K, _p(q), _p(s), _stream(stream))
    _check(st, "q8_gguf_to_planar")
    return q, s


def q8_planar_to_gguf(q, s, blocks=None, stream=None):
    """(q int8 [rows, K], s binary16 [rows, K/32]) -> GGUF Q8_0 bytes (uint8)."""
    _cuda(q, "q", (torch.int8,), 2)
    _cuda(s, "s", _B16, 2)
    rows, K = q.shape
    if blocks is None:
        blocks = torch.empty(rows * (K // 32) * 34, dtype=torch.uint8, device=q.device)
    st = lib().q8_planar_to_gguf(_p(q), _p(s), rows, K, _p(blocks), _stream(stream))
    _check(st, "q8_planar_to_gguf")
    return blocks


def q8_workspace_size(N: int, K: int, M: int) -> int:
    return int(lib().q8_workspace_size(N, K, M))


def _desc(q, s, x, y):
    _cuda(q, "q", (torch.int8,), 2)
    _cuda(s, "s", _B16, 2)
    _cuda(x, "x", _B16)
    _cuda(y, "y", (torch.float32,))
    N, K = q.shape
    x2 = x if x.dim() == 2 else x.view(1, -1)
    y2 = y if y.dim() == 2 else y.view(1, -1)
    if x2.stride(1) != 1 or y2.stride(1) != 1 or not q.is_contiguous() or not s.is_contiguous():
        raise ValueError("q, s must be contiguous; x, y must have unit inner stride")
    return LinearDesc(q.data_ptr(), s.data_ptr(), x2.data_ptr(), y2.data_ptr(), N, K,
                      x2.stride(0) if x2.shape[0] > 1 else K, y2.stride(0) if y2.shape[0] > 1 else max(N, 1)), x2.shape[0]


def q8_gemv(q, s, x, y=None, ws=None, dev_status=None, stream=None):
    """y[N] = dequant(q, s) @ x[K] (fp32)."""
    N, K = q.shape
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=q.device)
    need = q8_workspace_size(N, K, 1)
    if ws is None and need:
        ws = workspace(need, q.device)
    st = lib().q8_gemv(_p(q), _p(s), N, K, _p(x), _p(y), _p(ws), 0 if ws is None else ws.numel(),
                       _p(dev_status), _stream(stream))
    _check(st, "q8_gemv")
    return y


def q8_gemm_skinny(q, s, x, y=None, ws=None, dev_status=None, stream=None):
    """y[M, N] = x[M, K] @ dequant(q, s)^T (fp32), 1 <= M <= 32."""
    N, K = q.shape
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    d, _ = _desc(q, s, x, y)
    need = q8_workspace_size(N, K, M)
    if ws is None and need:
        ws = workspace(need, q.device)
    st = lib().q8_gemm_skinny(_p(q), _p(s), N, K, _p(x), d.ldx, M, _p(y), d.ldy, _p(ws),
                              0 if ws is None else ws.numel(), _p(dev_status), _stream(stream))
    _check(st, "q8_gemm_skinny")
    return y


def q8_gemm_skinny_noalloc(q, s, x, y=None, dev_status=None, stream=None):
    """As q8_gemm_skinny, for callers that cannot allocate device memory: the
    split-K scratch is the library's built-in device array (shapes needing more
    than Q8_NOALLOC_SCRATCH_BYTES are rejected).  Calls that may overlap on the
    GPU must not use it concurrently."""
    N, K = q.shape
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    d, _ = _desc(q, s, x, y)
    st = lib().q8_gemm_skinny_noalloc(_p(q), _p(s), N, K, _p(x), d.ldx, M, _p(y), d.ldy,
                                      _p(dev_status), _stream(stream))
    _check(st, "q8_gemm_skinny_noalloc")
    return y


def make_descs(mats):
    """[(q, s, x, y), ...] -> (ctypes array of LinearDesc, M)."""
    arr = (LinearDesc * len(mats))()
    M = None
    for i, (q, s, x, y) in enumerate(mats):
        arr[i], m = _desc(q, s, x, y)
        if M is not None and m != M:
            raise ValueError("all matrices of a batch share M")
        M = m
    return arr, (M or 0)


def q8_linear_batch_workspace_size(descs, M: int) -> int:
    return int(lib().q8_linear_batch_workspace_size(descs, len(descs), M))


def q8_linear_batch(mats=None, ws=None, variant=Q8_VARIANT_AUTO, dev_status=None, stream=None,
                    descs=None, M=None, chained=False):
    """Run several skinny matmuls in one launch.  ``mats`` = [(q, s, x, y), ...],
    or pass prepared ``descs`` (from make_descs) and ``M``.  ``chained=True``
    calls q8_linear_batch_chained (no earlier work in the stream may write
    the weights; the variant is then automatic)."""
    if descs is None:
        descs, M = make_descs(mats)
    need = int(lib().q8_linear_batch_workspace_size_ex(descs, len(descs), M, variant))
    if ws is None and need:
        ws = workspace(need)
    nbytes = 0 if ws is None else ws.numel()
    if chained:
        if variant != Q8_VARIANT_AUTO:
            raise ValueError("a chained call uses the automatic variant")
        st = lib().q8_linear_batch_chained(descs, len(descs), M, _p(ws), nbytes, _p(dev_status), _stream(stream))
    else:
        st = lib().q8_linear_batch_ex(descs, len(descs), M, variant, _p(ws), nbytes, _p(dev_status),
                                      _stream(stream))
    _check(st, "q8_linear_batch")


def make_chain(steps):
    """[(q, s, x, y, next), ...] -> (ctypes array of ChainStep, M).  Step 0's
    x is the input; every later x is a buffer the chain writes (bf16 [M][K]);
    y is fp32 [M][N]; `next` is a Q8_CHAIN_* code (Q8_CHAIN_END last)."""
    arr = (ChainStep * len(steps))()
    M = None
    for i, (q, s, x, y, nxt) in enumerate(steps):
        d, m = _desc(q, s, x, y)
        if M is not None and m != M:
            raise ValueError("all steps of a chain share M")
        M = m
        arr[i] = ChainStep(d.q, d.s, d.x, d.y, d.N, d.K, d.ldx, d.ldy, int(nxt), 0)
    return arr, (M or 0)


def q8_linear_chain_workspace_size(steps, M: int) -> int:
    return int(lib().q8_linear_chain_workspace_size(steps, len(steps), M))


def q8_linear_chain(steps, M, ws=None, dev_status=None, stream=None):
    """Run a chain from make_chain(): each step's matmul, then the next
    step's x made from its y on the device (q8_linear_chain)."""
    need = q8_linear_chain_workspace_size(steps, M)
    if ws is None and need:
        ws = workspace(need)
    nbytes = 0 if ws is None else ws.numel()
    st = lib().q8_linear_chain(steps, len(steps), M, _p(ws), nbytes, _p(dev_status), _stream(stream))
    _check(st, "q8_linear_chain")


def q8_gemm_w8a8(q, s, x, y=None, ws=None, dev_status=None, stream=None):
    """y[M, N] (fp32) = the W8A8 product of x[M, K] (bf16, rows quantized to
    Q8_0) and dequant(q, s)^T, any M (q8_gemm_w8a8)."""
    _cuda(q, "q", (torch.int8,), 2)
    _cuda(x, "x", _B16, 2)
    N, K = q.shape
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=q.device)
    need = int(lib().q8_gemm_w8a8_workspace_size(N, K, M))
    if ws is None and need:
        ws = workspace(need, q.device)
    st = lib().q8_gemm_w8a8(_p(q), _p(s), N, K, _p(x), x.stride(0), M, _p(y), y.stride(0), _p(ws),
                            0 if ws is None else ws.numel(), _p(dev_status), _stream(stream))
    _check(st, "q8_gemm_w8a8")
    return y


def q8_gemm(q, s, x, y=None, dev_status=None, stream=None, tile=0, splits=0):
    """y[M, N] (bf16) = x[M, K] @ dequant(q, s)^T for M > 32 (tcgen05 path);
    `tile` is one of the Q8_GEMM_TILE_* shapes and `splits` the number of
    CTAs sharing a tile's K range (0: automatic for either)."""
    _cuda(q, "q", (torch.int8,), 2)
    _cuda(x, "x", _B16, 2)
    N, K = q.shape
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=q.device)
    st = lib().q8_gemm_ex(_p(q), _p(s), N, K, _p(x), x.stride(0), M, _p(y), y.stride(0), int(tile), int(splits),
                          _p(dev_status), _stream(stream))
    _check(st, "q8_gemm")
    return y
