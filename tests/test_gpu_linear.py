"""Parity of the whole layer (convrot_linear / convrot_prepare_weight) with the
oracle, on the five workloads and the edge cases.

Y must lie within 1e-3 * |Y_ref| + 1e-3 of the oracle's fp32-epilogue result
(plus the LoRA term in fp64), widened only by what +-1 flips of near-tie
activation codes can change (the oracle computes that bound from its own
values).  Where the oracle would need minutes (the large configs), the GPU
runs the full shape and the oracle checks a seeded sample of rows: every
output row depends only on its own input row.
"""
import functools

import numpy as np
import pytest

import oracle
import workloads
import w8a8_hadamard_rotated_gb300 as cr

from . import gpu_util as gu
from . import report

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=8)
def _prep(N, K, seed):
    W = workloads.make_w(N, K, seed)
    return oracle.prepare_weight(W)


def _sample_rows(M, n, seed):
    if M <= n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    rows = rng.choice(M, size=n - 2, replace=False)
    return np.unique(np.concatenate([[0, M - 1], rows]))


def _check_config(cfg, n_rows=None, with_img=True):
    X, W, down, up = workloads.make_inputs(cfg)
    prep = _prep(cfg.N, cfg.K, cfg.seed)
    img = prep["Q_W"].astype(np.float16) if with_img else None
    Y = gu.linear(X, prep["Q_W"], prep["s_W"], img, down, up, cfg.lora_scale)
    rows = _sample_rows(cfg.M, n_rows, cfg.seed) if n_rows else np.arange(cfg.M)
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], down, up, cfg.lora_scale, rows=rows)
    err = gu.compare_y(Y[rows], ref)
    _record_quant_error(cfg.name, X[rows], W, down, up, cfg.lora_scale, Y[rows])
    return Y, ref, rows, err


def _record_quant_error(name, X, W, down, up, scale, Y):
    """Relative L2 and max-abs error of the fp16 Y against the unquantized
    fp64 product on the same rows (the error the W8A8 quantization costs),
    printed in the run's summary."""
    x = X.astype(np.float64)
    exact = oracle.matmul_nt(x, W.astype(np.float64))
    if down is not None:
        exact = exact + scale * oracle.matmul_nt(oracle.matmul_nt(x, down.astype(np.float64)),
                                                  up.astype(np.float64))
    d = Y.astype(np.float64) - exact
    report.QUANT_ERRORS.append((name, int(X.shape[0]),
                                float(np.linalg.norm(d) / np.linalg.norm(exact)),
                                float(np.abs(d).max()), float(np.abs(exact).max())))


def test_tiny_config():
    gu.require_gpu()
    cfg = workloads.TINY
    Y, ref, rows, err = _check_config(cfg)
    X, W, _, _ = workloads.make_inputs(cfg)
    exact = oracle.matmul_nt(X.astype(np.float64), W.astype(np.float64))
    qerr = np.linalg.norm(Y.astype(np.float64) - exact) / np.linalg.norm(exact)
    print(f"tiny: max |Y - Y_ref| = {err:.3g}; quant error vs fp64 XW^T = {qerr:.3g}")
    assert qerr < 0.02


def test_attn_config():
    gu.require_gpu()
    Y, ref, rows, err = _check_config(workloads.ATTN, n_rows=256)
    print(f"attn: max |Y - Y_ref| = {err:.3g}")


@pytest.mark.parametrize("i", range(len(workloads.SWEEP_SHAPES)))
def test_sweep_shapes(i):
    gu.require_gpu()
    cfg, _ = workloads.sweep_configs()[i]
    _check_config(cfg, n_rows=48)


@pytest.mark.parametrize("cfg", workloads.m_sweep_configs(), ids=lambda c: c.name)
def test_m_sweep(cfg):
    gu.require_gpu()
    _check_config(cfg, n_rows=32)


def test_lora_config():
    gu.require_gpu()
    _check_config(workloads.LORA, n_rows=32)


@pytest.mark.parametrize("M", [1, 3, 16, 40, 300])
def test_weight_image_optional_and_host_variant(M):
    gu.require_gpu()
    cfg = workloads.Config("t", M, 320, 1024, seed=M)
    X, W, _, _ = workloads.make_inputs(cfg)
    prep = _prep(cfg.N, cfg.K, cfg.seed)
    y_img = gu.linear(X, prep["Q_W"], prep["s_W"], prep["Q_W"].astype(np.float16))
    y_noimg = gu.linear(X, prep["Q_W"], prep["s_W"], None)
    assert np.array_equal(y_img.view(np.uint16), y_noimg.view(np.uint16))
    # Host-buffer entry point: same bits.
    torch = gu.torch
    Xh = torch.from_numpy(X).pin_memory()
    Yh = torch.empty((M, cfg.N), dtype=torch.float16).pin_memory()
    ws = gu.workspace(cr.convrot_linear_host_workspace_bytes(M, cfg.N, cfg.K, 0, False))
    cr.convrot_linear_host(Xh, gu.dev(prep["Q_W"]), gu.dev(prep["s_W"]), Yh, ws)
    gu.check_no_device_error()
    assert np.array_equal(Yh.numpy().view(np.uint16), y_noimg.view(np.uint16))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"])
    gu.compare_y(y_img, ref)


@pytest.mark.parametrize("M", [2, 100])
def test_lora_cancelling_and_zero_scale(M):
    gu.require_gpu()
    cfg = workloads.Config("t", M, 264, 512, seed=5, R=12, lora_scale=0.8)
    X, W, down, up = workloads.make_inputs(cfg)
    prep = _prep(cfg.N, cfg.K, cfg.seed)
    base = gu.linear(X, prep["Q_W"], prep["s_W"])
    # lora_scale = 0 and lora_up = 0: the base result bit for bit.
    y0 = gu.linear(X, prep["Q_W"], prep["s_W"], None, down, up, 0.0)
    yz = gu.linear(X, prep["Q_W"], prep["s_W"], None, down, np.zeros_like(up), 0.8)
    assert np.array_equal(y0.view(np.uint16), base.view(np.uint16))
    assert np.array_equal(yz.view(np.uint16), base.view(np.uint16))
    # A real LoRA at a rank that is not a multiple of 8 (rank tail).
    y = gu.linear(X, prep["Q_W"], prep["s_W"], None, down, up, 0.8)
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], down, up, 0.8)
    gu.compare_y(y, ref)


@pytest.mark.parametrize("M,N,K,R", [(4096, 2048, 8192, 32), (300, 256, 2048, 12), (7, 512, 1024, 32)])
def test_lora_layer_is_bit_reproducible(M, N, K, R):
    # The down-projection's K slices are added in a fixed order (a cluster
    # reduction, no atomics), so Y is the same bits on every run, and on a
    # workspace left dirty by another call.
    gu.require_gpu()
    torch = gu.torch
    X = workloads.make_x(M, K, seed=R + K, n_out=workloads.n_outliers(K))
    down, up = workloads.make_lora(N, K, R, seed=R)
    prep = _prep(N, K, 3)
    Xd, dd, ud = gu.dev(X), gu.dev(down), gu.dev(up)
    Qd, sd = gu.dev(prep["Q_W"]), gu.dev(prep["s_W"])
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, R, False))
    outs = []
    for fill in (0x00, 0x7F, 0xFF):
        ws.fill_(fill)
        Y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        cr.convrot_linear(Xd, Qd, sd, Y, ws, lora_down=dd, lora_up=ud, lora_scale=0.8)
        gu.check_no_device_error()
        outs.append(gu.host(Y).view(np.uint16))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    rows = np.unique(np.linspace(0, M - 1, min(M, 24)).astype(np.int64))
    ref = oracle.linear(X, prep["Q_W"], prep["s_W"], down, up, 0.8, rows=rows)
    gu.compare_y(outs[0].view(np.float16)[rows], ref)


def test_lora_layers_chained_in_a_graph():
    # Chained LoRA layers (each layer's Y the next one's X, one shared
    # workspace) captured in one graph on a side stream of the caller:
    # replays give the eager results bit for bit, also twice back to back.
    gu.require_gpu()
    torch = gu.torch
    M, N, K, R = 512, 1024, 1024, 32
    layers = []
    for i in range(3):
        down, up = workloads.make_lora(N, K, R, seed=40 + i)
        prep = _prep(N, K, 40 + i)
        layers.append((gu.dev(prep["Q_W"]), gu.dev(prep["s_W"]), gu.dev(down), gu.dev(up)))
    X0 = gu.dev(workloads.make_x(M, K, seed=40, n_out=workloads.n_outliers(K)))
    ws = gu.workspace(cr.convrot_linear_workspace_bytes(M, N, K, R, False))
    ys = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in layers]

    def chain():
        x = X0
        for (Q, s, d, u), y in zip(layers, ys):
            cr.convrot_linear(x, Q, s, y, ws, lora_down=d, lora_up=u, lora_scale=0.5)
            x = y

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        chain()
    stream.synchronize()
    gu.check_no_device_error()
    ref = [gu.host(y).view(np.uint16).copy() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        chain()
    for _ in range(2):
        for y in ys:
            y.zero_()
        with torch.cuda.stream(stream):
            g.replay()
            g.replay()
        stream.synchronize()
        gu.check_no_device_error()
        for y, r in zip(ys, ref):
            assert np.array_equal(gu.host(y).view(np.uint16), r)


def test_lora_only_when_weight_is_zero():
    gu.require_gpu()
    M, N, K, R = 24, 96, 512, 16
    X = workloads.make_x(M, K, seed=21)
    down, up = workloads.make_lora(N, K, R, seed=21)
    Q_W = np.zeros((N, K), np.int8)
    s_W = np.zeros((N,), np.float32)
    y = gu.linear(X, Q_W, s_W, None, down, up, 1.5)
    exact = oracle.lora(X.astype(np.float64), down, up, 1.5)
    np.testing.assert_allclose(y.astype(np.float64), exact, rtol=1e-3, atol=1e-4)


def test_zero_rows_and_column_tail():
    gu.require_gpu()
    M, N, K = 50, 77, 768
    X = workloads.make_x(M, K, seed=13)
    X[7] = 0
    prep = _prep(N, K, 13)
    y = gu.linear(X, prep["Q_W"], prep["s_W"])
    assert np.all(y[7] == 0)
    gu.compare_y(y, oracle.linear(X, prep["Q_W"], prep["s_W"]))


def test_prepare_weight_matches_oracle():
    gu.require_gpu()
    for (N, K, seed) in [(256, 256, 0), (77, 2048, 1), (40, 768, 2), (16, 8192, 3)]:
        W = workloads.make_w(N, K, seed)
        W[0] = 0.0
        Q, s, img = gu.prepare_weight(W)
        ref = oracle.prepare_weight(W)
        q = gu.host(Q)
        flips = gu.compare_q(q, ref["Q_W"], ref["pre"])
        np.testing.assert_allclose(gu.host(s), ref["s_W64"], rtol=1e-6, atol=0)
        assert np.array_equal(gu.host(img), q.astype(np.float16))
        assert np.all(q[0] == 0) and gu.host(s)[0] == 0
        print(f"prep N={N} K={K}: {flips} near-tie flips")


def test_full_gpu_pipeline_end_to_end():
    # Weight prepared on the GPU, then the layer, against the oracle layer on
    # the oracle's own prepared weight.  The two weight codes may differ by one
    # at near-tie positions; the tolerance adds what such a flip can change
    # (computed from the oracle's values only).
    gu.require_gpu()
    cfg = workloads.Config("t", 96, 512, 2048, seed=17)
    X, W, _, _ = workloads.make_inputs(cfg)
    Q, s, img = gu.prepare_weight(W)
    ref_w = oracle.prepare_weight(W)
    gu.compare_q(gu.host(Q), ref_w["Q_W"], ref_w["pre"])
    y = gu.linear(X, Q, s, img)
    ref = oracle.linear(X, ref_w["Q_W"], ref_w["s_W"])
    wnear = oracle.near_tie_mask(ref_w["pre"]).astype(np.float64)
    flips = np.abs(ref["Q_X"].astype(np.float64)) @ wnear.T
    ref["near_tie_bound"] = ref["near_tie_bound"] + flips * \
        ref["s_X"].astype(np.float64)[:, None] * ref_w["s_W"].astype(np.float64)[None, :]
    gu.compare_y(y, ref)


def test_host_entry_on_several_streams_in_one_graph():
    # The end-to-end pattern of the benchmark: layers of different shapes
    # dealt round-robin to three streams, each with its own workspace and
    # pinned output buffers, captured as one graph that forks from and joins
    # a main stream.  Every output must equal the single-call result.
    gu.require_gpu()
    torch = gu.torch
    shapes = [(512, 2048, 2048), (512, 256, 2048), (512, 6144, 256), (300, 640, 1024),
              (512, 2048, 2048), (300, 640, 1024)]
    layers = []
    for i, (M, N, K) in enumerate(shapes):
        X = workloads.make_x(M, K, 90 + i, workloads.n_outliers(K))
        Q_W, s_W, img = gu.prepare_weight(workloads.make_w(N, K, 90 + i))
        ref = gu.linear(X, Q_W, s_W, img).view(np.uint16)
        layers.append((torch.from_numpy(X).pin_memory(), Q_W, s_W, img, ref, M, N))
    ns = 3
    streams = [torch.cuda.Stream() for _ in range(ns)]
    ws = [gu.workspace(max(cr.convrot_linear_host_workspace_bytes(M, N, K, 0, True)
                           for (M, N, K) in shapes)) for _ in range(ns)]
    outs = [torch.empty((M, N), dtype=torch.float16).pin_memory() for (_, _, _, _, _, M, N) in layers]
    main = torch.cuda.Stream()

    def issue():
        fork = torch.cuda.Event()
        fork.record(main)
        for s in streams:
            s.wait_event(fork)
        for i, (Xh, Q_W, s_W, img, _, _, _) in enumerate(layers):
            with torch.cuda.stream(streams[i % ns]):
                cr.convrot_linear_host(Xh, Q_W, s_W, outs[i], ws[i % ns], W_img=img)
        for s in streams:
            join = torch.cuda.Event()
            join.record(s)
            main.wait_event(join)

    with torch.cuda.stream(main):
        issue()
    main.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=main):
        issue()
    for rep in range(3):
        for o in outs:
            o.zero_()
        with torch.cuda.stream(main):
            graph.replay()
        main.synchronize()
        gu.check_no_device_error()
        for i, (_, _, _, _, ref, _, _) in enumerate(layers):
            assert np.array_equal(outs[i].numpy().view(np.uint16), ref), (rep, i)
