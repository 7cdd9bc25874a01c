"""libq8 C ABI: the library loads, exports every function include/q8.h
declares, and rejects bad arguments on the host before any CUDA call (so
these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8.h")


@pytest.fixture(scope="module")
def L():
    from block_quantized_int8_gb300 import build, q8
    build.build()
    return q8.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q8_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["q8_quantize_rows", "q8_gemv", "q8_gemm_skinny", "q8_linear_batch", "q8_gemm"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    from block_quantized_int8_gb300 import q8
    for n in declared_functions():
        assert hasattr(L, n), n
    assert set(q8.EXPORTS) <= set(declared_functions())
    assert L.q8_abi_version() == 2


def test_status_strings(L):
    from block_quantized_int8_gb300 import q8
    for st in range(0, 8):
        assert q8.status_str(st)
    assert q8.status_str(99) == "unknown status"


# Fake, well-aligned device addresses: the calls below must fail validation
# before touching them.
A = 1 << 20


def call_gemv(L, q=A, s=A, N=128, K=64, x=A, y=A, ws=None, wsb=0):
    return L.q8_gemv(q, s, N, K, x, y, ws, wsb, None, None)


def test_gemv_validation(L):
    from block_quantized_int8_gb300 import q8
    assert call_gemv(L, K=33) == q8.Q8_ERR_SHAPE
    assert call_gemv(L, K=0) == q8.Q8_ERR_SHAPE
    assert call_gemv(L, K=-32) == q8.Q8_ERR_SHAPE
    assert call_gemv(L, N=-1) == q8.Q8_ERR_SHAPE
    assert call_gemv(L, q=None) == q8.Q8_ERR_ARG
    assert call_gemv(L, x=None) == q8.Q8_ERR_ARG
    assert call_gemv(L, y=None) == q8.Q8_ERR_ARG
    assert call_gemv(L, q=A + 8) == q8.Q8_ERR_ALIGN
    assert call_gemv(L, s=A + 2) == q8.Q8_ERR_ALIGN
    assert call_gemv(L, x=A + 4) == q8.Q8_ERR_ALIGN
    assert call_gemv(L, y=A + 2) == q8.Q8_ERR_ALIGN
    assert call_gemv(L, N=0) == q8.Q8_OK          # empty: no-op, no CUDA call


def test_skinny_validation(L):
    from block_quantized_int8_gb300 import q8
    f = L.q8_gemm_skinny
    assert f(A, A, 64, 64, A, 64, 33, A, 64, None, 0, None, None) == q8.Q8_ERR_SHAPE   # M > 32
    assert f(A, A, 64, 64, A, 64, -1, A, 64, None, 0, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 64, 64, A, 60, 2, A, 64, None, 0, None, None) == q8.Q8_ERR_SHAPE    # ldx < K
    assert f(A, A, 64, 64, A, 64, 2, A, 63, None, 0, None, None) == q8.Q8_ERR_SHAPE    # ldy < N
    assert f(A, A, 64, 64, A, 68, 2, A, 64, None, 0, None, None) == q8.Q8_ERR_ALIGN    # ldx % 8
    assert f(A, A, 64, 64, A, 64, 0, A, 64, None, 0, None, None) == q8.Q8_OK           # M == 0
    assert f(A, A, 64, 64, A, 64, 2, A, 64, None, 0, A + 1, None) == q8.Q8_ERR_ALIGN   # dev_status


def test_batch_validation(L):
    from block_quantized_int8_gb300 import q8
    d = (q8.LinearDesc * 2)()
    for i in range(2):
        d[i] = q8.LinearDesc(A, A, A, A, 64, 64, 64, 64)
    assert L.q8_linear_batch(d, 65, 1, None, 0, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_batch(None, 1, 1, None, 0, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_batch_ex(d, 2, 1, 7, None, 0, None, None) == q8.Q8_ERR_ARG
    # every variant takes any K that is a multiple of 32 (checked before
    # anything touches the device)
    d[0].K = 40
    assert L.q8_linear_batch_ex(d, 2, 3, q8.Q8_VARIANT_W8A8, None, 0, None, None) == q8.Q8_ERR_SHAPE
    assert L.q8_linear_batch_ex(d, 2, 3, q8.Q8_VARIANT_BATCH_INVARIANT, None, 0, None, None) == q8.Q8_ERR_SHAPE
    d[0].K = 64
    assert L.q8_linear_batch_ex(d, 2, 3, 5, None, 0, None, None) == q8.Q8_ERR_ARG
    # workspace by variant: none for batch-invariant; W8A8 holds x as binary32
    # blocks, codes and scales (per 256-wide chunk and 8-row group: 9 blocks)
    w = (q8.LinearDesc * 1)()
    w[0] = q8.LinearDesc(A, A, A, A, 1536, 4096, 4096, 1536)
    assert L.q8_linear_batch_workspace_size_ex(w, 1, 4, q8.Q8_VARIANT_BATCH_INVARIANT) == 0
    # off the 256 grid the batch-invariant variant keeps partial sums: K = 2080
    # in ceil(2080 / 512) = 5 ranges, 4 rows of 1536 fp32 each, 256-byte rounded
    odd = (q8.LinearDesc * 1)()
    odd[0] = q8.LinearDesc(A, A, A, A, 1536, 2080, 2080, 1536)
    inv = L.q8_linear_batch_workspace_size_ex(odd, 1, 4, q8.Q8_VARIANT_BATCH_INVARIANT)
    assert inv >= 5 * 4 * 1536 * 4 and inv % 256 == 0
    # W8A8 off the 256 grid: x as binary32, codes and scales (M = 4 rows)
    w8odd = L.q8_linear_batch_workspace_size_ex(odd, 1, 4, q8.Q8_VARIANT_W8A8)
    assert w8odd >= 4 * 2080 * 4 + 4 * 2080 + 4 * 65 * 2 and w8odd % 256 == 0
    assert L.q8_linear_batch_workspace_size_ex(w, 1, 4, 0) == L.q8_linear_batch_workspace_size(w, 1, 4)
    w8 = L.q8_linear_batch_workspace_size_ex(w, 1, 4, q8.Q8_VARIANT_W8A8)
    assert w8 >= 16 * 8 * 288 * 4 + 16 * 8 * (288 + 18) and w8 % 256 == 0
    d[1].K = 48
    assert L.q8_linear_batch(d, 2, 1, None, 0, None, None) == q8.Q8_ERR_SHAPE
    d[1].K = 64
    d[1].x = A + 2
    assert L.q8_linear_batch(d, 2, 1, None, 0, None, None) == q8.Q8_ERR_ALIGN
    assert L.q8_linear_batch(d, 0, 1, None, 0, None, None) == q8.Q8_OK
    # the chained entry point checks the same way before anything is launched
    assert L.q8_linear_batch_chained(d, 65, 1, None, 0, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_batch_chained(None, 1, 1, None, 0, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_batch_chained(d, 2, 1, None, 0, None, None) == q8.Q8_ERR_ALIGN
    assert L.q8_linear_batch_chained(d, 0, 1, None, 0, None, None) == q8.Q8_OK


def test_chain_validation(L):
    """q8_linear_chain checks the whole chain on the host before anything is
    enqueued: the `next` codes (the last step ends the chain), each step's K
    against the previous step's N (N >= K for RMSNORM, N >= 2 K for SwiGLU),
    M, the count, alignment and the workspace."""
    from block_quantized_int8_gb300 import q8

    def chain(*steps):
        arr = (q8.ChainStep * len(steps))()
        for i, (N, K, nxt) in enumerate(steps):
            arr[i] = q8.ChainStep(A, A, A, A, N, K, K, N, nxt, 0)
        return arr

    ok = chain((4608, 1536, q8.Q8_CHAIN_RMSNORM), (8192, 1536, q8.Q8_CHAIN_SWIGLU_RMSNORM),
               (1536, 4096, q8.Q8_CHAIN_END))
    need = L.q8_linear_chain_workspace_size(ok, 3, 1)
    # one 256-byte rounded region per distinct (N, K): a region always holds
    # the same layout, so its counters stay zero from step to step
    up = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert need == sum(up(L.q8_workspace_size(N, K, 1)) for (N, K) in [(4608, 1536), (8192, 1536), (1536, 4096)])
    twice = chain((4608, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 4608, q8.Q8_CHAIN_RMSNORM),
                  (4608, 1536, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain_workspace_size(twice, 3, 4) == sum(
        up(L.q8_workspace_size(N, K, 4)) for (N, K) in [(4608, 1536), (1536, 4608)])
    assert L.q8_linear_chain(ok, 3, 1, None, 0, None, None) == q8.Q8_ERR_WORKSPACE
    assert L.q8_linear_chain(ok, 3, 1, A + 16, 1 << 20, None, None) == q8.Q8_ERR_ALIGN
    assert L.q8_linear_chain(ok, 3, 33, A, 1 << 20, None, None) == q8.Q8_ERR_SHAPE
    assert L.q8_linear_chain(ok, 0, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_chain(None, 1, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ARG
    assert L.q8_linear_chain_workspace_size(ok, 3, 33) == 0
    # the last step must end the chain; a middle step must not
    bad = chain((1536, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 1536, q8.Q8_CHAIN_RMSNORM))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ARG
    bad = chain((1536, 1536, q8.Q8_CHAIN_END), (1536, 1536, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ARG
    bad = chain((1536, 1536, 7), (1536, 1536, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ARG
    # the next K must fit this step's N (twice over for SwiGLU)
    bad = chain((1536, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 2048, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_SHAPE
    bad = chain((4096, 1536, q8.Q8_CHAIN_SWIGLU_RMSNORM), (1536, 4096, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_SHAPE
    # an empty step and a K off the 32 grid
    bad = chain((0, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 1536, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_SHAPE
    bad = chain((1536, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 1540, q8.Q8_CHAIN_END))
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_SHAPE
    # a misaligned x of a later step
    bad = chain((1536, 1536, q8.Q8_CHAIN_RMSNORM), (1536, 1536, q8.Q8_CHAIN_END))
    bad[1].x = A + 2
    assert L.q8_linear_chain(bad, 2, 1, A, 1 << 20, None, None) == q8.Q8_ERR_ALIGN


def test_gemm_w8a8_validation(L):
    """q8_gemm_w8a8 (any M, W8A8 in 32-row slices) checks its arguments on the
    host; its workspace covers the largest launch (a group of up to 64 full
    slices, or the remaining rows)."""
    from block_quantized_int8_gb300 import q8
    f = L.q8_gemm_w8a8
    ws = L.q8_gemm_w8a8_workspace_size
    assert ws(8192, 1536, 512) > 0 and ws(8192, 1536, 512) % 256 == 0
    assert ws(8192, 1536, 512) >= ws(8192, 1536, 32) and ws(8192, 1536, 100) >= ws(8192, 1536, 4)
    # 16 slices in one launch hold 16 quantized copies of x; one slice holds one
    assert ws(8192, 1536, 512) > 8 * ws(8192, 1536, 32) // 2
    assert ws(8192, 1540, 512) == 0 and ws(0, 1536, 512) == 0 and ws(8192, 1536, 0) == 0
    need = ws(1536, 1536, 64)
    assert f(A, A, 1536, 1536, A, 1536, -1, A, 1536, A, need, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 1536, 1540, A, 1540, 64, A, 1536, A, need, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 1536, 1536, A + 2, 1536, 64, A, 1536, A, need, None, None) == q8.Q8_ERR_ALIGN
    assert f(A, A, 1536, 1536, A, 1536, 64, A, 1000, A, need, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 1536, 1536, A, 1536, 64, A, 1536, None, 0, None, None) == q8.Q8_ERR_WORKSPACE
    assert f(A, A, 1536, 1536, A, 1536, 64, A, 1536, A + 16, need, None, None) == q8.Q8_ERR_ALIGN
    assert f(A, A, 1536, 1536, A, 1536, 0, A, 1536, None, 0, None, None) == q8.Q8_OK


def test_quantize_validation(L):
    from block_quantized_int8_gb300 import q8
    f = L.q8_quantize_rows
    assert f(A, 4, 40, A, A, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, -1, 64, A, A, None, None) == q8.Q8_ERR_SHAPE
    assert f(None, 4, 64, A, A, None, None) == q8.Q8_ERR_ARG
    assert f(A + 4, 4, 64, A, A, None, None) == q8.Q8_ERR_ALIGN
    assert f(A, 0, 64, A, A, None, None) == q8.Q8_OK


def test_gemm_validation(L):
    from block_quantized_int8_gb300 import q8
    f = L.q8_gemm
    assert f(A, A, 64, 48, A, 64, 64, A, 64, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 64, 64, A, 64, 64, A, 60, None, None) == q8.Q8_ERR_SHAPE
    assert f(A, A, 64, 64, A, 64, 64, A + 8, 64, None, None) == q8.Q8_ERR_ALIGN
    g = L.q8_gemm_ex
    for tile in (-1, 4, 99):
        assert g(A, A, 64, 64, A, 64, 64, A, 64, tile, 0, None, None) == q8.Q8_ERR_ARG
    for splits in (-1, q8.Q8_GEMM_MAX_SPLITS + 1):
        assert g(A, A, 64, 64, A, 64, 64, A, 64, 0, splits, None, None) == q8.Q8_ERR_ARG
    assert g(A, A, 64, 48, A, 64, 64, A, 64, q8.Q8_GEMM_TILE_64x128, 1, None, None) == q8.Q8_ERR_SHAPE


def test_quantize_ex_validation(L):
    from block_quantized_int8_gb300 import q8
    assert L.q8_quantize_rows_ex(A, 1, 32, A, A, 2, None, None) == q8.Q8_ERR_ARG
    assert L.q8_quantize_rows_ex(A, 1, 32, A, A, -1, None, None) == q8.Q8_ERR_ARG
    assert L.q8_quantize_rows_ex(A, 1, 48, A, A, q8.Q8_QUANT_FL32, None, None) == q8.Q8_ERR_SHAPE
    assert L.q8_quantize_rows_ex(A + 4, 1, 32, A, A, q8.Q8_QUANT_FL32, None, None) == q8.Q8_ERR_ALIGN
    assert L.q8_quantize_rows_ex(A, 0, 32, A, A, q8.Q8_QUANT_FL32, None, None) == q8.Q8_OK


def test_selftest_validation(L):
    from block_quantized_int8_gb300 import q8
    assert L.q8_selftest_wait_timeout(0, None, None, None) == q8.Q8_ERR_ARG
    assert L.q8_selftest_wait_timeout(2_000_000_000, None, None, None) == q8.Q8_ERR_ARG
    assert L.q8_selftest_wait_timeout(1000, A + 2, None, None) == q8.Q8_ERR_ALIGN
    assert L.q8_selftest_wait_timeout(1000, None, A + 4, None) == q8.Q8_ERR_ALIGN


def test_gguf_validation(L):
    """Argument checks of the GGUF repack happen on the host, before any CUDA call."""
    from block_quantized_int8_gb300 import q8
    assert L.q8_gguf_to_planar(A, 2, 48, A, A, None) == q8.Q8_ERR_SHAPE
    assert L.q8_gguf_to_planar(A, -1, 64, A, A, None) == q8.Q8_ERR_SHAPE
    assert L.q8_gguf_to_planar(None, 2, 64, A, A, None) == q8.Q8_ERR_ARG
    assert L.q8_gguf_to_planar(A + 2, 2, 64, A, A, None) == q8.Q8_ERR_ALIGN
    assert L.q8_gguf_to_planar(A, 2, 64, A + 8, A, None) == q8.Q8_ERR_ALIGN
    assert L.q8_gguf_to_planar(A, 0, 64, None, None, None) == q8.Q8_OK
    assert L.q8_planar_to_gguf(A, A, 2, 64, None, None) == q8.Q8_ERR_ARG
    assert L.q8_planar_to_gguf(A, A, 2, 64, A + 2, None) == q8.Q8_ERR_ALIGN
    assert L.q8_planar_to_gguf(A, A, 2, 40, A, None) == q8.Q8_ERR_SHAPE


def test_workspace_sizes(L):
    from block_quantized_int8_gb300 import q8
    # invalid shapes need nothing
    assert L.q8_workspace_size(0, 64, 1) == 0
    assert L.q8_workspace_size(64, 33, 1) == 0
    assert L.q8_workspace_size(64, 64, 33) == 0
    # a huge N needs no split, only (at M = 1) the 256-byte block of the
    # GEMV's pool counter; a short-N, long-K matrix splits K as well
    assert L.q8_workspace_size(262144, 1536, 1) == 256
    assert L.q8_workspace_size(262144, 1536, 2) == 0
    w = L.q8_workspace_size(1536, 4096, 1)
    assert w > 256 and w % 256 == 0
    # a batch needs the sum of its members' split workspaces and one counter block
    d = (q8.LinearDesc * 2)()
    d[0] = q8.LinearDesc(A, A, A, A, 1536, 4096, 4096, 1536)
    d[1] = q8.LinearDesc(A, A, A, A, 262144, 1536, 1536, 262144)
    assert L.q8_linear_batch_workspace_size(d, 2, 1) == w
    # and the size does not depend on which device is current (host arithmetic)
    assert L.q8_workspace_size(1536, 4096, 32) >= L.q8_workspace_size(1536, 4096, 1)
