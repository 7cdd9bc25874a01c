"""M <= 32 matmul kernels (q8_gemv, q8_gemm_skinny, q8_linear_batch) vs the
oracle.  Exactly representable inputs must match bit for bit; random Q8_0
inputs must satisfy |y - y_ref| <= 2e-3 * sum|w'x| + 1e-6 per output."""
import numpy as np
import pytest
import torch

import synth
from helpers import check_tol, dev, weights_dev, x_dev

pytestmark = pytest.mark.gpu

VARIANTS = [0, 1, 2]  # Q8_VARIANT_AUTO, Q8_VARIANT_SIMT, Q8_VARIANT_MMA


def run_batch(mats_np, M, variant, ws_extra=0):
    """mats_np = [(q, s, x_bits)]; returns list of y (numpy fp32)."""
    from block_quantized_int8_gb300 import q8
    mats = []
    outs = []
    for (qn, sn, xn) in mats_np:
        q, s = weights_dev(qn, sn)
        x = x_dev(xn)
        y = torch.full((M, qn.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
        mats.append((q, s, x, y))
        outs.append(y)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch(mats, variant=variant, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return [y.cpu().numpy() for y in outs]


# ---------------------------------------------------------------------------
# exact cases: every product and sum is exact in fp32 -> bit-exact
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,K", [(1, 32), (7, 64), (128, 96), (129, 1536), (300, 4096), (1536, 1536),
                                 (129, 2080), (130, 4384)])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16, 17, 32])
def test_exact_cases_bit_exact(oracle, variant, N, K, M):
    q, s, x = synth.exact_case(N, K, M, 0, f"ex{N}.{K}.{M}")
    y_ref, _ = oracle.matmul(q, s, x)
    (y,) = run_batch([(q, s, x)], M, variant)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("variant", VARIANTS)
def test_unit_vectors(oracle, variant):
    N, K = 200, 1536
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, "uvec"))
    for k in [0, 31, 32, 700, 1535]:
        x = synth.unit_vector_x(K, k)
        (y,) = run_batch([(q, s, x)], 1, variant)
        expect = s[:, k // 32].view(np.float16).astype(np.float64) * q[:, k]
        assert np.array_equal(y[0].astype(np.float64), expect)


# ---------------------------------------------------------------------------
# random Q8_0 weights, tolerance; sizes span several tiles, splits and a tail
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,K", [(300, 1536), (1536, 4096), (4097, 1536), (33, 32)])
@pytest.mark.parametrize("M", [1, 2, 5, 8, 13, 32])
def test_random_tolerance(oracle, variant, N, K, M):
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"rt{N}.{K}"))
    x = synth.activations(M, K, 0, f"rtx{M}.{K}")
    y_ref, B = oracle.matmul(q, s, x, threads=8)
    (y,) = run_batch([(q, s, x)], M, variant)
    check_tol(y, y_ref, B, f"N={N} K={K} M={M} variant={variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("N,K", [(300, 1536), (77, 4096), (130, 2048)])
@pytest.mark.parametrize("M", [1, 2, 8, 16])
def test_wide_range_activations(oracle, variant, N, K, M):
    """Activations spanning the whole bf16 range, subnormals and zeros: the
    binary16 fast path of the M <= 8 kernel has to hand such blocks to its
    exact bf16 path, and every kernel stays within the tolerance."""
    q, s, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"wr{N}.{K}"))
    x = synth.wide_range_activations(M, K, 0, f"wrx{M}.{K}")
    y_ref, B = oracle.matmul(q, s, x, threads=8)
    (y,) = run_batch([(q, s, x)], M, variant)
    check_tol(y, y_ref, B, f"wide range N={N} K={K} M={M} variant={variant}")


def test_gemv_and_skinny_entry_points(oracle):
    from block_quantized_int8_gb300 import q8
    N, K = 1536, 4096
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "ep"))
    xn = synth.activations(4, K, 0, "epx")
    y_ref, B = oracle.matmul(qn, sn, xn)
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    y1 = q8.q8_gemv(q, s, x[0].contiguous())
    y4 = q8.q8_gemm_skinny(q, s, x)
    torch.cuda.synchronize()
    check_tol(y1.cpu().numpy()[None], y_ref[:1], B[:1], "gemv")
    check_tol(y4.cpu().numpy(), y_ref, B, "skinny")


def test_strided_x_and_y(oracle):
    from block_quantized_int8_gb300 import q8
    N, K, M = 520, 1536, 3
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "strided"))
    xn = synth.activations(M, K, 0, "stridedx")
    y_ref, B = oracle.matmul(qn, sn, xn)
    q, s = weights_dev(qn, sn)
    xb = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    xb[:, :K] = x_dev(xn)
    yb = torch.full((M, N + 40), -7.0, dtype=torch.float32, device="cuda")
    q8.q8_gemm_skinny(q, s, xb[:, :K], yb[:, :N])
    torch.cuda.synchronize()
    out = yb.cpu().numpy()
    check_tol(out[:, :N], y_ref, B, "strided")
    assert np.all(out[:, N:] == -7.0)  # nothing written past ldy's live columns


# ---------------------------------------------------------------------------
# full-size workloads of the benchmark (sampled or full comparisons)
# ---------------------------------------------------------------------------
def test_tiny_gemv_full(oracle):
    N, K = 4096, 1536
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "tiny"))
    xn = synth.activations(1, K, 0, "tinyx")
    y_ref, B = oracle.matmul(qn, sn, xn, threads=8)
    for v in VARIANTS:
        (y,) = run_batch([(qn, sn, xn)], 1, v)
        check_tol(y, y_ref, B, f"tiny v{v}")


def test_vocab_gemv_sampled(oracle):
    from block_quantized_int8_gb300 import q8
    N, K = synth.VOCAB, synth.HIDDEN
    w = synth.weights(N, K, 0, "vocab")
    q, s = q8.q8_quantize_rows(dev(w))
    xn = synth.unit_activation(K, 0)
    y = q8.q8_gemv(q, s, x_dev(xn)[0].contiguous())
    torch.cuda.synchronize()
    rows = np.sort(synth.rng(0, "vocab.rows").choice(N, 4096, replace=False))
    rows = np.unique(np.concatenate([rows, [0, N - 1]]))
    qn, sn, _ = oracle.quantize_rows(w[rows])
    y_ref, B = oracle.matmul(qn, sn, xn)
    check_tol(y.cpu().numpy()[rows][None], y_ref, B, "vocab")


@pytest.mark.parametrize("K,N", synth.SWEEP_SHAPES)
@pytest.mark.parametrize("M", synth.SWEEP_M)
def test_sweep_full(oracle, K, N, M):
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"sweep{K}.{N}"))
    xn = synth.activations(M, K, 0, f"sweepx{M}.{K}")
    rows = np.arange(N) if M <= 8 else np.unique(np.concatenate(
        [synth.rng(0, "sweep.rows").choice(N, 1024, replace=False), [0, N - 1]]))
    y_ref, B = oracle.matmul(qn[rows], sn[rows], xn, threads=8)
    for v in VARIANTS:
        (y,) = run_batch([(qn, sn, xn)], M, v)
        check_tol(y[:, rows], y_ref, B, f"sweep K={K} N={N} M={M} v{v}")


def test_layer_set_batch_sampled(oracle):
    """One pass of the decode layer set (16 layers x 4 matrices) as one batch."""
    from block_quantized_int8_gb300 import q8
    mats, refs = [], []
    xs = {K: synth.activations(1, K, 0, synth.layer_x_tag(0, K)) for K in (synth.HIDDEN, synth.INTER)}
    for layer in range(synth.LAYERS):
        for (name, K, N) in synth.LAYER_MATRICES:
            w = synth.weights(N, K, 0, synth.layer_weight_tag(layer, name))
            q, s = q8.q8_quantize_rows(dev(w))
            y = torch.empty((1, N), dtype=torch.float32, device="cuda")
            mats.append((q, s, x_dev(xs[K]), y))
            rows = np.unique(np.concatenate([synth.rng(layer, name).choice(N, 48, replace=False), [0, N - 1]]))
            refs.append((w, rows, xs[K]))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch(mats, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for (q, s, x, y), (w, rows, xn) in zip(mats, refs):
        qn, sn, _ = oracle.quantize_rows(w[rows])
        y_ref, B = oracle.matmul(qn, sn, xn)
        check_tol(y.cpu().numpy()[:, rows], y_ref, B, "layer set")


@pytest.mark.parametrize("M", [1, 8, 16])
def test_chained_calls_keep_write_order(oracle, M):
    """Chained calls that write the same outputs from different activations,
    back to back: the last call's values must be what remains (a dependent
    launch writes y only after the calls before it have completed)."""
    from block_quantized_int8_gb300 import q8
    N, K = 1536, 4096
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "wo"))
    q, s = weights_dev(qn, sn)
    xs = [x_dev(synth.activations(M, K, 0, f"wox{i}")) for i in range(5)]
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = q8.workspace(q8.q8_linear_batch_workspace_size(q8.make_descs([(q, s, xs[0], y)])[0], M))
    want = torch.empty_like(y)
    q8.q8_linear_batch([(q, s, xs[-1], want)], ws=ws)
    for rep in range(3):
        for x in xs:
            q8.q8_linear_batch([(q, s, x, y)], ws=ws, chained=True)
        torch.cuda.synchronize()
        assert torch.equal(y, want)


def test_layer_set_bench_step_sampled(oracle):
    """The benchmark's own step: the layer set built by bench.py, 8 passes
    launched with q8_linear_batch_chained as it times them, twice in a row on
    one workspace; sampled outputs of every pass and matrix against the
    oracle, and the second step bit-identical to the first."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from block_quantized_int8_gb300 import q8
    ls = bench.LayerSet(torch, q8)
    ls.y_all.fill_(float("nan"))
    ls.step(chained=True)
    torch.cuda.synchronize()
    first = ls.y_all.clone()
    ls.y_all.fill_(float("nan"))
    ls.step(chained=True)
    torch.cuda.synchronize()
    assert torch.equal(ls.y_all, first)
    assert int(ls.ws.view(-1)[-256:].count_nonzero()) == 0
    for layer in range(synth.LAYERS):
        for (name, K, N) in synth.LAYER_MATRICES:
            w = synth.weights(N, K, 0, synth.layer_weight_tag(layer, name))
            rows = np.unique(np.concatenate([synth.rng(layer, "step." + name).choice(N, 16, replace=False),
                                             [0, N - 1]]))
            qn, sn, _ = oracle.quantize_rows(w[rows])
            for p in (0, synth.PASSES - 1, layer % synth.PASSES):
                y_ref, B = oracle.matmul(qn, sn, ls.x_host[(p, K)])
                y = ls.y[p][layer][name].cpu().numpy()[:, rows]
                check_tol(y, y_ref, B, f"bench step pass {p} layer {layer} {name}")


# ---------------------------------------------------------------------------
# determinism, graph replay, batch == separate calls
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M", [1, 3, 8, 12, 20])
@pytest.mark.parametrize("variant", VARIANTS)
def test_batch_equals_separate_calls_bitwise(oracle, variant, M):
    # shapes that the automatic routing sends to different kernels: K = 1536
    # or K % 256 != 0 (pipeline for M <= 8), other K % 256 == 0 (tiles for
    # M >= 2), K > 4096 off the 256 grid and K > 12288 (general)
    # (the tiles' K classes: 4 at K = 4096, 3 at K = 1536, 2 of 5 chunks at
    # K = 2560, 1 at K = 256; a lone matrix shares its row blocks between
    # CTAs, a batch mostly does not)
    shapes = [(4608, 1536), (1536, 1536), (8192, 1536), (1536, 4096), (77, 256),
              (130, 2080), (300, 4128), (96, 12800), (300, 2560)]
    mats_np = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"bs{i}"))
        mats_np.append((qn, sn, synth.activations(M, K, 0, f"bsx{i}")))
    together = run_batch(mats_np, M, variant)
    for m_np, y_t in zip(mats_np, together):
        (y_s,) = run_batch([m_np], M, variant)
        assert np.array_equal(y_s, y_t)


@pytest.mark.parametrize("M", [4, 12, 24, 32])
@pytest.mark.parametrize("K", [1536, 4096])
def test_tile_k_split_keeps_bits(oracle, M, K):
    """A lone small matrix has its row blocks' K classes spread over several
    CTAs (to fill the GPU), so its row blocks are added through the
    workspace; in a launch with many rows most are not.  Its result must not
    change.  (M > 16 at K = 4096: four classes, the running sums kept in
    the workspace.)"""
    if M <= 8 and K == 1536:
        pytest.skip("served by the pipeline kernel, not the tiles")
    qn, sn, _ = oracle.quantize_rows(synth.weights(1536, K, 0, "ks"))
    mat = (qn, sn, synth.activations(M, K, 0, "ksx"))
    (alone,) = run_batch([mat], M, 0)
    big_q, big_s, _ = oracle.quantize_rows(synth.weights(8192, K, 0, "ksb"))
    big = (big_q, big_s, synth.activations(M, K, 0, "ksbx"))
    together = run_batch([mat] + [big] * 6, M, 0)
    assert np.array_equal(alone, together[0])
    y_ref, B = oracle.matmul(qn, sn, mat[2], threads=8)
    check_tol(alone, y_ref, B, f"K split N=1536 K={K} M={M}")


@pytest.mark.parametrize("M", [2, 9, 16, 17, 32])
@pytest.mark.parametrize("K", [288, 800, 2080, 4128, 6176, 12800])
def test_tile_partial_chunk(oracle, K, M):
    """K not a multiple of 256 on the tile kernel (M = 9..32, and M = 2..8
    beyond the pipeline's K <= 4096): the last chunk is partial, the blocks
    past K add exact zeros.  Within the tolerance of the oracle at 300 rows
    (a partial last row block); a lone matrix (its row blocks' classes spread
    over CTAs) gives the same bits as beside six large ones."""
    qn, sn, _ = oracle.quantize_rows(synth.weights(300, K, 0, f"pc{K}"))
    mat = (qn, sn, synth.activations(M, K, 0, f"pcx{K}.{M}"))
    (alone,) = run_batch([mat], M, 0)
    y_ref, B = oracle.matmul(qn, sn, mat[2], threads=8)
    check_tol(alone, y_ref, B, f"partial chunk K={K} M={M}")
    big_q, big_s, _ = oracle.quantize_rows(synth.weights(4096, K, 0, f"pcb{K}"))
    big = (big_q, big_s, synth.activations(M, K, 0, f"pcbx{K}.{M}"))
    together = run_batch([mat] + [big] * 6, M, 0)
    assert np.array_equal(alone, together[0])


@pytest.mark.parametrize("M", [1, 4, 16, 32])
def test_workspace_shared_by_other_shapes(oracle, M):
    """One workspace serving calls of different shapes in turn: the split-K
    tickets and counters of one call sit where another call's partial sums
    went, so the library clears a call's counter words when the workspace
    last held another layout.  Each result equals, bit for bit, the result
    on a fresh workspace, through several alternations (QKV-shaped, then
    gate+up-shaped matmuls: their tile tickets and partials overlap), and
    also after a W8A8 call on the same workspace."""
    from block_quantized_int8_gb300 import q8
    shapes = [(4608, 1536), (8192, 1536), (1536, 1536), (1536, 4096)]
    mats = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"wsx{i}"))
        q, s = weights_dev(qn, sn)
        x = x_dev(synth.activations(M, K, 0, f"wsxx{i}.{M}"))
        mats.append((q, s, x))
    fresh = []
    for (q, s, x) in mats:
        y = torch.empty((M, q.shape[0]), dtype=torch.float32, device="cuda")
        q8.q8_linear_batch([(q, s, x, y)])
        fresh.append(y)
    need = 0
    for (q, s, x) in mats:
        d, _ = q8.make_descs([(q, s, x, torch.empty((M, q.shape[0]), dtype=torch.float32, device="cuda"))])
        need = max(need, q8.q8_linear_batch_workspace_size(d, M),
                   int(q8.lib().q8_linear_batch_workspace_size_ex(d, 1, M, q8.Q8_VARIANT_W8A8)))
    ws = q8.workspace(need)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rnd in range(3):
        for i in [0, 1, 2, 1, 3, 0, 1]:
            q, s, x = mats[i]
            y = torch.full((M, q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
            q8.q8_linear_batch([(q, s, x, y)], ws=ws, dev_status=st)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int32), fresh[i].view(torch.int32)), f"round {rnd} shape {shapes[i]}"
        q, s, x = mats[rnd % len(mats)]
        y8 = torch.empty((M, q.shape[0]), dtype=torch.float32, device="cuda")
        q8.q8_linear_batch([(q, s, x, y8)], ws=ws, variant=q8.Q8_VARIANT_W8A8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_gemv_pool_counter_returns_to_zero(oracle):
    """The M = 1 kernel hands out its last stages through a counter in the
    workspace; every launch must leave it zero, or the next launch on the same
    workspace would skip stages.  Repeated calls and graph replays on one
    workspace give the same bits, and the counter block reads zero after."""
    from block_quantized_int8_gb300 import q8
    mats, ys, host = [], [], []
    for i, (N, K) in enumerate([(4608, 1536), (1536, 1536), (8192, 1536), (1536, 4096)] * 4):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"pc{i % 4}"))
        xn = synth.activations(1, K, 0, f"pcx{i}")
        host.append((qn, sn, xn))
        q, s = weights_dev(qn, sn)
        x = x_dev(xn)
        y = torch.empty((1, N), dtype=torch.float32, device="cuda")
        mats.append((q, s, x, y))
        ys.append(y)
    descs, M = q8.make_descs(mats)
    need = q8.q8_linear_batch_workspace_size(descs, M)
    assert need >= 256
    ws = q8.workspace(need)
    q8.q8_linear_batch(descs=descs, M=M, ws=ws)
    torch.cuda.synchronize()
    first = [y.clone() for y in ys]
    assert int(ws.view(-1)[-256:].count_nonzero()) == 0
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        q8.q8_linear_batch(descs=descs, M=M, ws=ws)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ys, first))
        assert int(ws.view(-1)[-256:].count_nonzero()) == 0
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        q8.q8_linear_batch(descs=descs, M=M, ws=ws)
    stream.synchronize()
    with torch.cuda.graph(g, stream=stream):
        q8.q8_linear_batch(descs=descs, M=M, ws=ws)
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(ys, first))
    assert int(ws.view(-1)[-256:].count_nonzero()) == 0
    # and the result is right
    for (qn, sn, xn), y in zip(host[:4], ys[:4]):
        y_ref, B = oracle.matmul(qn, sn, xn, threads=8)
        check_tol(y.cpu().numpy(), y_ref, B, "pooled GEMV")


@pytest.mark.parametrize("M", [1, 4, 12, 24])
def test_chained_calls_match_plain_calls(oracle, M):
    """q8_linear_batch_chained over a stream of passes (new x each pass, one
    workspace, weights fixed) gives the same bits as q8_linear_batch, also in
    a CUDA graph, and leaves the M = 1 pool counter zero.  The shapes reach
    every kernel family (GEMV, pipeline, tiles, general)."""
    from block_quantized_int8_gb300 import q8
    shapes = [(4608, 1536), (1536, 1536), (8192, 1536), (1536, 4096), (300, 2080)]
    w = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"ch{i}"))
        w.append(weights_dev(qn, sn))
    passes = 6
    xs = [[x_dev(synth.activations(M, K, 0, f"chx{p}.{i}")) for i, (N, K) in enumerate(shapes)]
          for p in range(passes)]

    def run(chained, graph=False):
        ys = [[torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for (N, K) in shapes]
              for _ in range(passes)]
        descs = [q8.make_descs([(w[i][0], w[i][1], xs[p][i], ys[p][i]) for i in range(len(shapes))])[0]
                 for p in range(passes)]
        ws = q8.workspace(max(q8.q8_linear_batch_workspace_size(d, M) for d in descs))
        st = torch.zeros(1, dtype=torch.int32, device="cuda")

        def step():
            for d in descs:
                q8.q8_linear_batch(descs=d, M=M, ws=ws, dev_status=st, chained=chained)
        if graph:
            stream = torch.cuda.Stream()
            with torch.cuda.stream(stream):
                step()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            for _ in range(2):
                g.replay()
        else:
            for _ in range(3):
                step()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        if ws is not None and M == 1:
            assert int(ws.view(-1)[-256:].count_nonzero()) == 0
        return [[y.cpu() for y in row] for row in ys]

    plain = run(False)
    for got in (run(True), run(True, graph=True)):
        for p in range(passes):
            for a, b in zip(plain[p], got[p]):
                assert torch.equal(a, b)
    qn, sn, _ = oracle.quantize_rows(synth.weights(1536, 4096, 0, "ch3"))
    y_ref, B = oracle.matmul(qn, sn, synth.activations(M, 4096, 0, "chx5.3"), threads=8)
    check_tol(plain[5][3].numpy(), y_ref, B, "chained pass 5")


@pytest.mark.parametrize("variant", VARIANTS)
def test_deterministic_and_graph_replay(oracle, variant):
    from block_quantized_int8_gb300 import q8
    N, K, M = 1536, 4096, 4   # split-K path
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, "det"))
    q, s = weights_dev(qn, sn)
    x = x_dev(synth.activations(M, K, 0, "detx"))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    descs, _ = q8.make_descs([(q, s, x, y)])
    ws = q8.workspace(q8.q8_linear_batch_workspace_size(descs, M))
    assert ws is not None   # this shape is split along K
    q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=variant)
    torch.cuda.synchronize()
    first = y.clone()
    for _ in range(3):
        y.zero_()
        q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=variant)
        torch.cuda.synchronize()
        assert torch.equal(y, first)
    # capture into a CUDA graph and replay
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=variant)  # warm on the capture stream
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=variant)
    for _ in range(3):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, first)
    # the split-K tickets (first words of the workspace) are reset after every call
    tiles = (N + 127) // 128
    assert int(ws[: 4 * tiles].ne(0).sum().item()) == 0


def test_workspace_too_small_is_rejected(oracle):
    from block_quantized_int8_gb300 import q8
    N, K = 1536, 4096
    q = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((N, K // 32), dtype=torch.float16, device="cuda")
    x = torch.zeros((16, K), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((16, N), dtype=torch.float32, device="cuda")
    need = q8.q8_workspace_size(N, K, 16)
    assert need > 256   # M = 16 on this short-N, long-K shape splits K
    ws = q8.workspace(need - 256)
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_gemm_skinny(q, s, x, y, ws=ws)
    assert e.value.status == q8.Q8_ERR_WORKSPACE


def test_empty_shapes_noop():
    from block_quantized_int8_gb300 import q8
    q = torch.zeros((0, 64), dtype=torch.int8, device="cuda")
    s = torch.zeros((0, 2), dtype=torch.float16, device="cuda")
    x = torch.zeros((2, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((2, 0), dtype=torch.float32, device="cuda")
    q8.q8_gemm_skinny(q, s, x, y)
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# the M = 1 pipeline: K slicing (1, 2, 4, 8 slices), scale tails that are not
# a multiple of 16 bytes, and the fallback beyond its largest K
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("K", [32, 96, 1568, 2080, 4096, 6176, 8192, 12320, 16384, 16416])
@pytest.mark.parametrize("N", [1, 7, 33, 300])
def test_gemv_k_slicing_exact(oracle, K, N):
    q, s, x = synth.exact_case(N, K, 1, 0, f"gk{N}.{K}")
    y_ref, _ = oracle.matmul(q, s, x)
    for v in VARIANTS:
        (y,) = run_batch([(q, s, x)], 1, v)
        assert np.array_equal(y.astype(np.float64), y_ref), f"variant {v}"


def test_gemv_mixed_batch_tolerance(oracle):
    """Matrices of different K (different slice counts) in one M = 1 launch."""
    shapes = [(300, 96), (1000, 1536), (77, 4096), (513, 8192), (5, 32), (129, 2080)]
    mats_np = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"mix{i}"))
        mats_np.append((qn, sn, synth.activations(1, K, 0, f"mixx{i}")))
    ys = run_batch(mats_np, 1, 0)
    for (qn, sn, xn), y in zip(mats_np, ys):
        y_ref, B = oracle.matmul(qn, sn, xn)
        check_tol(y, y_ref, B, f"mixed N={qn.shape[0]} K={qn.shape[1]}")
    # and each matrix alone gives the same bits
    for m_np, y in zip(mats_np, ys):
        (y1,) = run_batch([m_np], 1, 0)
        assert np.array_equal(y1, y)


@pytest.mark.parametrize("N,K,M", [(300, 1024, 12), (130, 2048, 3), (96, 1536, 16), (130, 2080, 12),
                                   (77, 4384, 5)])
def test_tile_x_copy_chunks(oracle, N, K, M):
    """The tile kernel (M <= 16) reads x from a copy in the workspace: each 256-column
    chunk (all M rows) as binary16 when binary16 holds every value of the
    chunk exactly (zero, or magnitude in [2^-17, 65504]), else as the bf16
    bits, with one flag word per chunk (0 = binary16).  For K not a multiple
    of 256 the copy's rows are K rounded up to 256 long, zero past K.
    Checked against that rule restated on the float values, then the result
    against the oracle."""
    from block_quantized_int8_gb300 import q8
    KC = (K + 255) // 256
    Kp = KC * 256
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"xc{N}.{K}"))
    xn = synth.activations(M, K, 0, f"xcx{M}.{K}").copy()
    # chunk 1 gets a value below binary16's exact range in its last row,
    # chunk 3 (if any) one above it in its first row; the rest stay N(0, 1)
    tiny = np.array([3e-7], dtype=np.float32).view(np.uint32)[0] >> 16
    huge = np.array([1e5], dtype=np.float32).view(np.uint32)[0] >> 16
    xn[M - 1, 256 + 17] = tiny
    if KC > 3:
        xn[0, 3 * 256 + 200] = huge
    xf = (xn.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    a = np.abs(xf)
    fits = (a == 0) | ((a >= 2.0 ** -17) & (a <= 65504.0))
    want_flags = np.array([0 if fits[:, 256 * c:min(K, 256 * (c + 1))].all() else 1 for c in range(KC)], np.uint32)
    assert want_flags[1] == 1 and 0 in want_flags

    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    need = q8.q8_workspace_size(N, K, M)
    up = lambda b: (b + 255) // 256 * 256
    copy_bytes = up(M * Kp * 2)
    # after the copy and its flags: the tickets and partials of row blocks
    # that CTAs share, for at most min(320, row blocks) of them
    MT = 1 if M <= 8 else 2
    ms = min(320, (N + 127) // 128)
    split_bytes = up(ms * 8 * 4) + ms * 4 * 8 * 32 * MT * 16
    tile_bytes = copy_bytes + up(KC * 4) + split_bytes
    assert need >= tile_bytes
    ws = q8.workspace(need)
    y = q8.q8_gemm_skinny(q, s, x, ws=ws)
    torch.cuda.synchronize()
    w = ws.cpu().numpy()
    off = need - tile_bytes
    got_copy = w[off:off + M * Kp * 2].view(np.uint16).reshape(M, Kp)
    got_flags = w[off + copy_bytes:off + copy_bytes + KC * 4].view(np.uint32)
    assert np.array_equal(got_flags, want_flags)
    assert not got_copy[:, K:].any()
    for c in range(KC):
        cols = slice(256 * c, min(K, 256 * (c + 1)))
        if want_flags[c]:
            want = xn[:, cols]
        else:
            want = xf[:, cols].astype(np.float16).view(np.uint16)
        assert np.array_equal(got_copy[:, cols], want), f"chunk {c}"
    y_ref, B = oracle.matmul(qn, sn, xn, threads=8)
    check_tol(y.cpu().numpy(), y_ref, B, f"x copy N={N} K={K} M={M}")


def test_batch_invariant_rows(oracle):
    """Q8_VARIANT_BATCH_INVARIANT: row m of Y is the same, bit for bit, for
    every M that includes it, alone or in a batch of matrices, and within
    the tolerance of the oracle."""
    from block_quantized_int8_gb300 import q8
    shapes = [(300, 4096), (1536, 1536), (130, 256), (4100, 2048)]
    mats = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"inv{i}"))
        mats.append((qn, sn, synth.activations(32, K, 0, f"invx{i}")))
    dev_w = [weights_dev(qn, sn) for (qn, sn, _) in mats]

    def run(M, which):
        outs, ms = [], []
        for i in which:
            q, s = dev_w[i]
            x = x_dev(np.ascontiguousarray(mats[i][2][:M]))
            y = torch.full((M, q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
            ms.append((q, s, x, y))
            outs.append(y)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q8.q8_linear_batch(ms, variant=q8.Q8_VARIANT_BATCH_INVARIANT, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return [y.cpu().numpy() for y in outs]

    everything = list(range(len(mats)))
    full = run(32, everything)
    for i, (qn, sn, xn) in enumerate(mats):
        y_ref, B = oracle.matmul(qn, sn, xn, threads=8)
        check_tol(full[i], y_ref, B, f"invariant N={qn.shape[0]} K={qn.shape[1]}")
    for M in (1, 2, 3, 5, 8, 9, 12, 16, 17, 24, 31):
        part = run(M, everything)
        for i in everything:
            assert np.array_equal(part[i], full[i][:M]), f"matrix {i} at M={M}"
        (alone,) = run(M, [1])
        assert np.array_equal(alone, full[1][:M])


@pytest.mark.parametrize("K", [2080, 4128, 12800])
def test_batch_invariant_rows_any_k(oracle, K):
    """The batch-invariant variant at K % 256 != 0 (the general kernel, one K
    range per row tile): row m is the same, bit for bit, for every M that
    includes it, alone or beside a K % 256 == 0 matrix, and within the
    tolerance of the oracle."""
    from block_quantized_int8_gb300 import q8
    shapes = [(300, K), (1000, 4096)]
    mats = []
    for i, (N, Kk) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, Kk, 0, f"invk{K}.{i}"))
        mats.append((qn, sn, synth.activations(32, Kk, 0, f"invkx{K}.{i}")))
    dev_w = [weights_dev(qn, sn) for (qn, sn, _) in mats]

    def run(M, which):
        outs, ms = [], []
        for i in which:
            q, s = dev_w[i]
            x = x_dev(np.ascontiguousarray(mats[i][2][:M]))
            y = torch.full((M, q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
            ms.append((q, s, x, y))
            outs.append(y)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        q8.q8_linear_batch(ms, variant=q8.Q8_VARIANT_BATCH_INVARIANT, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return [y.cpu().numpy() for y in outs]

    full = run(32, [0, 1])
    qn, sn, xn = mats[0]
    y_ref, B = oracle.matmul(qn, sn, xn, threads=8)
    check_tol(full[0], y_ref, B, f"invariant N=300 K={K}")
    for M in (1, 2, 5, 8, 9, 16, 17, 31):
        part = run(M, [0, 1])
        for i in (0, 1):
            assert np.array_equal(part[i], full[i][:M]), f"matrix {i} at M={M}"
        (alone,) = run(M, [0])
        assert np.array_equal(alone, full[0][:M])


def _w8a8_run(mats_np, M):
    from block_quantized_int8_gb300 import q8
    mats, outs = [], []
    for (qn, sn, xn) in mats_np:
        q, s = weights_dev(qn, sn)
        y = torch.full((M, qn.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
        mats.append((q, s, x_dev(np.ascontiguousarray(xn)), y))
        outs.append(y)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch(mats, variant=q8.Q8_VARIANT_W8A8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return [y.cpu().numpy() for y in outs]


@pytest.mark.parametrize("M", [1, 3, 8, 12, 16, 32])
def test_w8a8_tolerance_and_batch(oracle, M):
    """W8A8 (activations quantized to Q8_0 per row, int8 block dots) against
    the oracle's W8A8 definition; a batch gives the same bits as separate calls."""
    shapes = [(300, 4096), (1536, 1536), (130, 256), (4100, 2048)]
    mats = []
    for i, (N, K) in enumerate(shapes):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"w8{i}"))
        mats.append((qn, sn, synth.activations(M, K, 0, f"w8x{i}.{M}")))
    together = _w8a8_run(mats, M)
    for m_np, y in zip(mats, together):
        y_ref, B = oracle.matmul_w8a8(*m_np)
        check_tol(y, y_ref, B, f"W8A8 N={m_np[0].shape[0]} K={m_np[0].shape[1]} M={M}")
        (alone,) = _w8a8_run([m_np], M)
        assert np.array_equal(alone, y)


def test_w8a8_exact_case(oracle):
    """Integer activations with 127 in every block quantize to themselves;
    with small codes and power-of-two weight scales every sum is exact in
    fp32, so the kernel matches the W8A8 definition bit for bit."""
    N, K, M = 300, 1536, 9
    q, s, _ = synth.exact_case(N, K, M, 0, "w8ex")
    rng = np.random.default_rng(11)
    xv = rng.integers(-126, 127, size=(M, K)).astype(np.float32)
    xv[:, ::32] = 127.0
    xb = (xv.view(np.uint32) >> 16).astype(np.uint16)
    (y,) = _w8a8_run([(q, s, xb)], M)
    y_ref, _ = oracle.matmul_w8a8(q, s, xb)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("M", [1, 12, 32])
@pytest.mark.parametrize("K", [2080, 4128, 12800])
def test_w8a8_any_k(oracle, K, M):
    """W8A8 at K % 256 != 0 (the general kernel: x quantized to Q8_0 rows in
    the workspace, one int8 MMA per block): within the tolerance of the
    oracle's W8A8 definition, and the same bits alone as beside a K % 256
    == 0 matrix (which the tile kernel serves)."""
    mats = []
    for i, (N, Kk) in enumerate([(300, K), (1536, 4096)]):
        qn, sn, _ = oracle.quantize_rows(synth.weights(N, Kk, 0, f"w8k{K}.{i}"))
        mats.append((qn, sn, synth.activations(M, Kk, 0, f"w8kx{K}.{i}.{M}")))
    together = _w8a8_run(mats, M)
    y_ref, B = oracle.matmul_w8a8(*mats[0])
    check_tol(together[0], y_ref, B, f"W8A8 N=300 K={K} M={M}")
    (alone,) = _w8a8_run([mats[0]], M)
    assert np.array_equal(alone, together[0])


def test_w8a8_exact_case_any_k(oracle):
    """The exact case of test_w8a8_exact_case at K = 2080 (general kernel):
    bit for bit the W8A8 definition."""
    N, K, M = 300, 2080, 9
    q, s, _ = synth.exact_case(N, K, M, 0, "w8exk")
    rng = np.random.default_rng(12)
    xv = rng.integers(-126, 127, size=(M, K)).astype(np.float32)
    xv[:, ::32] = 127.0
    xb = (xv.view(np.uint32) >> 16).astype(np.uint16)
    (y,) = _w8a8_run([(q, s, xb)], M)
    y_ref, _ = oracle.matmul_w8a8(q, s, xb)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("M,kind", [(5, "normal"), (17, "wide"), (32, "small")])
def test_w8a8_activation_codes_any_k(oracle, M, kind):
    """At K % 256 != 0 the W8A8 activations are quantized into the workspace
    as binary32 rows [M][K], then codes [M][K] and binary16 scales
    [M][K / 32] (each region rounded up to 256 bytes).  Read back, the codes
    and scales equal the oracle's quantize_rows of the binary32 activations
    bit for bit, and the device status equals the oracle's flags."""
    from block_quantized_int8_gb300 import q8
    N, K = 130, 2080
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"w8qk{M}"))
    if kind == "normal":
        xn = synth.activations(M, K, 0, f"w8qkx{M}")
    elif kind == "wide":
        xn = synth.wide_range_activations(M, K, 0, f"w8qkw{M}")
    else:
        xn = _small_scale_activations(M, K, f"w8qks{M}")
    q, s = weights_dev(qn, sn)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    x = x_dev(xn)  # the descriptor holds a bare pointer: keep x alive
    descs, _ = q8.make_descs([(q, s, x, y)])
    need = int(q8.lib().q8_linear_batch_workspace_size_ex(descs, 1, M, q8.Q8_VARIANT_W8A8))
    up = lambda b: (b + 255) // 256 * 256  # noqa: E731
    assert need >= up(M * K * 4) + up(M * K) + up(M * (K // 32) * 2)
    ws = q8.workspace(need)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=q8.Q8_VARIANT_W8A8, dev_status=st)
    torch.cuda.synchronize()
    raw = ws.cpu().numpy().view(np.uint8)
    o_q = up(M * K * 4)
    o_s = o_q + up(M * K)
    codes = raw[o_q:o_q + M * K].view(np.int8).reshape(M, K)
    scales = raw[o_s:o_s + M * (K // 32) * 2].view(np.uint16).reshape(M, K // 32)
    xf = synth.bf16_bits_to_f32(xn)
    ref_q, ref_s, flags = oracle.quantize_rows(xf)
    assert np.array_equal(codes, ref_q)
    assert np.array_equal(scales, ref_s)
    assert int(st.item()) == int(flags)
    if int(flags) == 0:
        y_ref, B = oracle.matmul_w8a8(qn, sn, xn)
        check_tol(y.cpu().numpy(), y_ref, B, f"W8A8 codes case M={M} {kind}")


def _small_scale_activations(M, K, tag):
    """bf16 bits [M][K]: N(0, 1) draws times one magnitude per 32-block,
    cycling over 2^-8 .. 2^-24, 0 and 1, so that blocks get normal,
    binary16-subnormal and zero activation scales (amax / 127 below 2^-14
    is subnormal in binary16, below 2^-25 it rounds to zero)."""
    g = synth.normal_f32((M, K), 0, tag).astype(np.float64)
    mags = np.array([2.0 ** -8, 2.0 ** -12, 2.0 ** -16, 2.0 ** -20, 2.0 ** -24, 0.0, 1.0])
    blk = np.arange(K) // 32
    pick = (blk[None, :] + np.arange(M)[:, None]) % len(mags)
    return synth.f32_to_bf16_bits((g * mags[pick]).astype(np.float32))


@pytest.mark.parametrize("N,K,M,kind", [(300, 1536, 3, "normal"), (130, 4096, 12, "wide"),
                                        (96, 2048, 32, "wide"), (200, 1024, 8, "small"),
                                        (77, 2560, 17, "small")])
def test_w8a8_activation_codes_bit_exact(oracle, N, K, M, kind):
    """The W8A8 variant quantizes each activation row to Q8_0 in the
    workspace with the weights' quantizer.  Read back, the codes and binary16
    scales equal the oracle's quantize_rows of the binary32 activations bit
    for bit, rows past M and each chunk's ninth (padding) block are zero, and
    the device status equals the oracle's flags (wide-range rows hold blocks
    whose scale overflows binary16).  Layout of the region: binary32 blocks
    [K/256][MP][9 x 32], then codes [K/256][MP][9 x 32] and scales
    [K/256][MP][9], MP = M rounded up to 8, 16 or 32.  The result then
    satisfies the tolerance against the oracle's W8A8 reference."""
    from block_quantized_int8_gb300 import q8
    qn, sn, _ = oracle.quantize_rows(synth.weights(N, K, 0, f"w8q{N}.{K}"))
    if kind == "normal":
        xn = synth.activations(M, K, 0, f"w8qx{M}.{K}")
    elif kind == "wide":
        xn = synth.wide_range_activations(M, K, 0, f"w8qw{M}.{K}")
    else:
        xn = _small_scale_activations(M, K, f"w8qs{M}.{K}")
    xf = synth.bf16_bits_to_f32(xn)
    qx, sx, flags = oracle.quantize_rows(xf)
    if kind == "small":
        sxf = oracle.f16_to_f64(sx)
        assert (sxf == 0).any() and ((sxf > 0) & (sxf < 2.0 ** -14)).any() and (sxf >= 2.0 ** -14).any()
    q, s = weights_dev(qn, sn)
    x = x_dev(xn)
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    descs, _ = q8.make_descs([(q, s, x, y)])
    need = int(q8.lib().q8_linear_batch_workspace_size_ex(descs, 1, M, q8.Q8_VARIANT_W8A8))
    ws = q8.workspace(need)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q8.q8_linear_batch(descs=descs, M=M, ws=ws, variant=q8.Q8_VARIANT_W8A8, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == flags
    KC = K // 256
    MP = 8 if M <= 8 else (16 if M <= 16 else 32)
    up = lambda b: (b + 255) // 256 * 256  # noqa: E731
    w = ws.cpu().numpy()
    off = up(KC * MP * 288 * 4)
    got_q = w[off:off + KC * MP * 288].view(np.int8).reshape(KC, MP, 9, 32)
    got_s = w[off + KC * MP * 288:off + KC * MP * 288 + KC * MP * 9 * 2].view(np.uint16).reshape(KC, MP, 9)
    want_q = np.zeros((KC, MP, 9, 32), np.int8)
    want_q[:, :M, :8, :] = qx.reshape(M, KC, 8, 32).transpose(1, 0, 2, 3)
    want_s = np.zeros((KC, MP, 9), np.uint16)
    want_s[:, :M, :8] = sx.reshape(M, KC, 8).transpose(1, 0, 2)
    assert np.array_equal(got_s, want_s)
    assert np.array_equal(got_q, want_q)
    y_ref, B = oracle.matmul_w8a8(qn, sn, xn)
    check_tol(y.cpu().numpy(), y_ref, B, f"W8A8 {kind} N={N} K={K} M={M}")
