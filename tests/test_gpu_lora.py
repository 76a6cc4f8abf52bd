"""GPU parity of idlm_gated_lora (the tcgen05 gated-LoRA projection) against
the oracle (marked gpu).

Tolerance: outputs are stored in bf16 after fp32 accumulation, so they are
compared with the attention bound, |gpu - oracle| <= 2e-2 + 1e-2 |oracle|,
against the oracle's float64 result on the same bf16 inputs.  Rows whose gate
is 0 must equal the same kernel's output without the adapter bit for bit
("Lossless R-ISD": verify positions keep the base model's outputs).
"""
import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from oracle import isd
from speculative_verify_accept_step_b300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def gpu_lora_status(x, w, a, b, g, s, dev="cuda"):
    M, K = x.shape
    N, r = w.shape[0], a.shape[0]
    ws = torch.empty(lib.idlm_gated_lora_workspace_size(M, K, N, r), dtype=torch.uint8,
                     device=dev)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.idlm_gated_lora(x.to(dev), w.to(dev), a.to(dev), b.to(dev), g.to(dev), s, y, ws, st)
    torch.cuda.synchronize()
    return y, int(st.item())


def gpu_lora(x, w, a, b, g, s, dev="cuda"):
    y, st = gpu_lora_status(x, w, a, b, g, s, dev)
    assert st == 0, f"device status {st}"
    return y


def case(M, K, N, r, seed, wstd=0.02):
    gen = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=gen).bfloat16()
    w = (torch.randn(N, K, generator=gen) * wstd).bfloat16()
    a = (torch.randn(r, K, generator=gen) * wstd).bfloat16()
    b = (torch.randn(N, r, generator=gen) * wstd).bfloat16()
    g = (torch.arange(M) % 7 >= 4).to(torch.uint8)
    return x, w, a, b, g


def assert_close(got, ref):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = float((err / bound).max())
    assert np.all(err <= bound), f"worst err/bound {worst:.3f}"
    return worst


@pytest.mark.parametrize("M,K,N,r", [(21, 136, 200, 16), (3, 64, 128, 8), (3, 64, 256, 8),
                                     (45, 320, 204, 8),
                                     (448, 512, 384, 16), (600, 256, 256, 16), (130, 320, 520, 64),
                                     (48, 4096, 128, 16)])
def test_against_oracle_small(cuda_device, M, K, N, r):
    x, w, a, b, g = case(M, K, N, r, seed=M + K + N)
    y = gpu_lora(x, w, a, b, g, 1.0)
    ref = isd.gated_lora(f64(x), f64(w), f64(a), f64(b), g.numpy(), 1.0)
    assert_close(f64(y), ref)


def test_lora_scale(cuda_device):
    x, w, a, b, g = case(64, 256, 256, 16, seed=5, wstd=0.2)
    y = gpu_lora(x, w, a, b, g, 0.5)
    ref = isd.gated_lora(f64(x), f64(w), f64(a), f64(b), g.numpy(), 0.5)
    assert_close(f64(y), ref)


def test_ungated_rows_bit_identical_to_the_base_projection(cuda_device):
    x, w, a, b, g = case(448, 1024, 512, 16, seed=7, wstd=0.2)
    y = gpu_lora(x, w, a, b, g, 1.0)
    y0 = gpu_lora(x, w, a, torch.zeros_like(b), g, 1.0)
    clean = g == 0
    assert torch.equal(y[clean.cuda()], y0[clean.cuda()])
    # and the adapter does change the MASK rows
    assert not torch.equal(y[~clean.cuda()], y0[~clean.cuda()])
    # every gate off: the whole output equals the base projection
    yoff = gpu_lora(x, w, a, b, torch.zeros_like(g), 1.0)
    assert torch.equal(yoff, y0)


@pytest.mark.parametrize("name", ["q", "k", "gate", "down"])
def test_layer_projection_full_size_sampled(cuda_device, name):
    """One projection of the workload's decoder layer (hidden 4096, FFN 12288,
    448 token rows, rank 16) at full size, checked on 4096 sampled outputs
    that the oracle computes one by one."""
    w_ = wl.WORKLOADS["lora_layer_m448"]
    inp = wl.lora_inputs(w_)
    pj = inp["proj"][name]
    x = inp["x"] if name != "down" else (torch.randn(448, w_.ffn, generator=torch.Generator().manual_seed(3))).bfloat16()
    y = f64(gpu_lora(x, pj["w"], pj["a"], pj["b"], inp["row_gate"], inp["lora_scale"]))
    M, N = y.shape
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, M, 4096), rng.integers(0, N, 4096)
    xs, ws_ = f64(x), None
    wf, af, bf = f64(pj["w"]), f64(pj["a"]), f64(pj["b"])
    g = inp["row_gate"].numpy()
    ref = np.array([isd.gated_lora(xs[m:m + 1], wf[n:n + 1], af, bf[n:n + 1], g[m:m + 1],
                                   inp["lora_scale"])[0, 0] for m, n in zip(ms, ns)])
    assert_close(y[ms, ns], ref)


@pytest.mark.parametrize("M,K,N,r", [(448, 640, 520, 16), (130, 4096, 256, 64), (37, 192, 384, 8)])
def test_every_grid_size_matches_the_oracle_and_repeats_bitwise(cuda_device, monkeypatch, M, K, N, r):
    """The GEMM splits the (tile, K step) work evenly over its grid; a tile
    cut by a range boundary is summed from fp32 partial tiles in CTA order.
    Every grid size (1 CTA, ranges inside one tile, ranges across several
    tiles) must match the oracle, and a repeated call with the same grid must
    give the same bits."""
    x, w, a, b, g = case(M, K, N, r, seed=11 + M)
    ref = isd.gated_lora(f64(x), f64(w), f64(a), f64(b), g.numpy(), 1.0)
    for grid in (1, 2, 3, 7, 19, 64, 148):
        monkeypatch.setenv("IDLM_LORA_GRID", str(grid))
        y1 = gpu_lora(x, w, a, b, g, 1.0)
        assert_close(f64(y1), ref)
        y2 = gpu_lora(x, w, a, b, g, 1.0)
        assert torch.equal(y1, y2), f"grid {grid} not reproducible"


def test_ungated_rows_bit_identical_under_a_split_k_sum(cuda_device, monkeypatch):
    """With tiles whose K sum is split over several CTAs, rows with g = 0 must
    still equal the base projection (lora_b = 0) bit for bit."""
    monkeypatch.setenv("IDLM_LORA_GRID", "37")
    x, w, a, b, g = case(448, 2048, 640, 16, seed=9, wstd=0.2)
    y = gpu_lora(x, w, a, b, g, 1.0)
    y0 = gpu_lora(x, w, a, torch.zeros_like(b), g, 1.0)
    clean = (g == 0).cuda()
    assert torch.equal(y[clean], y0[clean])


def test_fused_projections_match_the_separate_ones(cuda_device):
    """q|k|v as one call (weights stacked along N, adapters stacked along the
    rank with B block diagonal) gives each projection's output: compared with
    the three separate calls within the tolerance, and with the oracle on
    sampled outputs."""
    w_ = wl.WORKLOADS["lora_layer_m448"]
    inp = wl.lora_inputs(w_)
    names = ("q", "k", "v")
    f = wl.fuse_projections(inp["proj"], names)
    yf = f64(gpu_lora(inp["x"], f["w"], f["a"], f["b"], inp["row_gate"], inp["lora_scale"]))
    n0 = 0
    for n in names:
        pj = inp["proj"][n]
        ys = f64(gpu_lora(inp["x"], pj["w"], pj["a"], pj["b"], inp["row_gate"], inp["lora_scale"]))
        assert_close(yf[:, n0:n0 + ys.shape[1]], ys)
        n0 += ys.shape[1]
    assert n0 == yf.shape[1]
    M, N = yf.shape
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, M, 2048), rng.integers(0, N, 2048)
    xs, wf, af, bf = f64(inp["x"]), f64(f["w"]), f64(f["a"]), f64(f["b"])
    g = inp["row_gate"].numpy()
    ref = np.array([isd.gated_lora(xs[m:m + 1], wf[n:n + 1], af, bf[n:n + 1], g[m:m + 1],
                                   inp["lora_scale"])[0, 0] for m, n in zip(ms, ns)])
    assert_close(yf[ms, ns], ref)


def test_a_wait_that_runs_out_reports_timeout_and_the_context_survives(cuda_device, monkeypatch):
    """Failure detection without a GPU fault.  Under the test switch
    IDLM_TEST_STALL=1 every GEMM CTA first waits on an mbarrier that nothing
    arrives on; its bounded wait (20 ms) runs out, the kernel records
    TIMEOUT (5) in the status word, drains its copies, frees its tensor
    memory and returns.  The next call, without the switch, must run
    normally and match the oracle."""
    x, w, a, b, g = case(64, 1024, 256, 16, seed=13)
    monkeypatch.setenv("IDLM_LORA_GRID", "7")   # 2 tiles x 17 K steps over 7 CTAs: split
    monkeypatch.setenv("IDLM_TEST_STALL", "1")
    _, st = gpu_lora_status(x, w, a, b, g, 1.0)
    assert st == 5, f"expected TIMEOUT, device status {st}"
    monkeypatch.delenv("IDLM_TEST_STALL")
    y = gpu_lora(x, w, a, b, g, 1.0)
    ref = isd.gated_lora(f64(x), f64(w), f64(a), f64(b), g.numpy(), 1.0)
    assert_close(f64(y), ref)


@pytest.mark.parametrize("M,K,N,r", [(448, 1024, 384, 72), (448, 4096, 512, 128),
                                     (37, 320, 200, 128), (130, 2048, 256, 120)])
def test_rank_up_to_128_matches_the_oracle(cuda_device, M, K, N, r):
    """Ranks above 64 take two adapter K steps ("Lossless R-ISD": the pages'
    adapter has rank 128)."""
    x, w, a, b, g = case(M, K, N, r, seed=r + K)
    y = gpu_lora(x, w, a, b, g, 1.0)
    ref = isd.gated_lora(f64(x), f64(w), f64(a), f64(b), g.numpy(), 1.0)
    assert_close(f64(y), ref)


def test_rank_128_ungated_rows_bit_identical(cuda_device, monkeypatch):
    monkeypatch.setenv("IDLM_LORA_GRID", "37")
    x, w, a, b, g = case(448, 2048, 640, 128, seed=21, wstd=0.2)
    y = gpu_lora(x, w, a, b, g, 1.0)
    y0 = gpu_lora(x, w, a, torch.zeros_like(b), g, 1.0)
    clean = (g == 0).cuda()
    assert torch.equal(y[clean], y0[clean])
    assert not torch.equal(y[~clean], y0[~clean])


def gpu_lora_grouped(x, w, a, b, g, s, group_rows, dev="cuda"):
    M, K = x.shape
    N = w.shape[0]
    r = a.shape[0] // len(group_rows)
    ws = torch.empty(lib.idlm_gated_lora_grouped_workspace_size(M, K, N, r, len(group_rows)),
                     dtype=torch.uint8, device=dev)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.idlm_gated_lora_grouped(x.to(dev), w.to(dev), a.to(dev), b.to(dev), g.to(dev), s,
                                group_rows, y, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return y


@pytest.mark.parametrize("r", [16, 128])
def test_grouped_projections_match_the_separate_ones(cuda_device, r):
    """q|k|v in one call with one adapter per group: each group's columns
    match that projection's own call and the oracle, within the tolerance
    (the two calls may split their K sums differently)."""
    gen = torch.Generator().manual_seed(r)
    M, K = 448, 1024
    rows = [512, 256, 256]
    x = torch.randn(M, K, generator=gen).bfloat16()
    g = (torch.arange(M) % 7 >= 4).to(torch.uint8)
    ws_, as_, bs_ = [], [], []
    for n in rows:
        ws_.append((torch.randn(n, K, generator=gen) * 0.02).bfloat16())
        as_.append((torch.randn(r, K, generator=gen) * 0.02).bfloat16())
        bs_.append((torch.randn(n, r, generator=gen) * 0.02).bfloat16())
    W, A, B = torch.cat(ws_), torch.cat(as_), torch.cat(bs_)
    yg = f64(gpu_lora_grouped(x, W, A, B, g, 1.0, rows))
    n0 = 0
    for i, n in enumerate(rows):
        ys = f64(gpu_lora(x, ws_[i], as_[i], bs_[i], g, 1.0))
        assert_close(yg[:, n0:n0 + n], ys)
        ref = isd.gated_lora(f64(x), f64(ws_[i]), f64(as_[i]), f64(bs_[i]), g.numpy(), 1.0)
        assert_close(yg[:, n0:n0 + n], ref)
        n0 += n


def test_graph_replays_sum_the_adapter_slices(cuda_device):
    """Rank 16 at K = 4096 computes T = g s X A^T in several K slices, summed
    by the last slice of each block to arrive; a CUDA graph replays the
    launch with its epoch frozen, and every replay must still sum them."""
    M, K, N, r = 448, 4096, 512, 16
    x, w, a, b, g = case(M, K, N, r, seed=31)
    eager = gpu_lora(x, w, a, b, g, 1.0)
    dev = "cuda"
    xs, ws_, as_, bs, gs = (t.to(dev) for t in (x, w, a, b, g))
    ws = torch.empty(lib.idlm_gated_lora_workspace_size(M, K, N, r), dtype=torch.uint8,
                     device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            lib.idlm_gated_lora(xs, ws_, as_, bs, gs, 1.0, y, ws, st)
    for _ in range(3):
        y.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(y, eager)
