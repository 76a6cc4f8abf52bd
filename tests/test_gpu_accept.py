"""GPU parity of idlm_isd_accept against the oracle (marked gpu).

Each case runs a FRESH step (whose MASK rows propose the drafts) and then a
FULL step that verifies them, on the GPU and in the oracle, from the same
seeded logits; each side computes its own drafts and q statistics.
"""
import numpy as np
import pytest
import torch

from _gpu import compare_accept, f64, gpu_accept, run_two_steps_gpu, run_two_steps_oracle
from oracle import isd
from speculative_verify_accept_step_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _check_pair(b, N, T, pm, seed, step0, greedy=False):
    g0, g1 = run_two_steps_gpu(b, N, T, pm, seed, step0)
    o0, o1 = run_two_steps_oracle(b, N, T, pm, seed, step0)
    s0 = compare_accept(g0, o0, N, greedy)
    # the FULL step only makes sense where both sides proposed the same drafts
    assert np.array_equal(g0["next_drafts"].cpu().numpy(), o0["next_drafts"])
    s1 = compare_accept(g1, o1, N, greedy)
    return s0, s1, o1


def test_tiny_fp32_workload(cuda_device):
    w = wl.WORKLOADS["isd_tiny_c1_n2_f32"]
    b = wl.accept_inputs(w)
    for step0 in range(0, 40, 2):
        _check_pair(b, w.N, 1.0, isd.PROPOSE_ARGMAX, 0, step0)


def test_small_bf16_workload(cuda_device):
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    b = wl.accept_inputs(w)
    for step0 in (0, 10, 20):
        s0, s1, _ = _check_pair(b, w.N, 1.0, isd.PROPOSE_ARGMAX, 0, step0)
        assert s1["compared"] >= 3


def test_headline_workload_full_size(cuda_device):
    w = wl.WORKLOADS["isd_c64_n4_ctx4096"]
    b = wl.accept_inputs(w)
    s0, s1, o1 = _check_pair(b, w.N, 1.0, isd.PROPOSE_ARGMAX, 0, 0)
    assert s1["compared"] >= 60
    # the batch exercised both rejections (residual draws) and bonus draws
    kinds = set(o1["final_kind"].tolist())
    assert isd.END_RESIDUAL in kinds and isd.END_BONUS in kinds


def test_ragged_workload_mixed_targets(cuda_device):
    w = wl.WORKLOADS["isd_c64_n4_ctx1k_32k"]
    b = wl.accept_inputs(w)
    _, s1, _ = _check_pair(b, w.N, 1.0, isd.PROPOSE_ARGMAX, 3, 100)
    assert s1["compared"] >= 60


def _small_batch(C, N, V, seed, scale=2.0, noise=0.7, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    l1 = torch.randn(C * (2 * N - 1), V, generator=g) * scale
    l0 = torch.empty(C * N, V)
    for c in range(C):
        l0[c * N] = torch.randn(V, generator=g) * scale
        for k in range(1, N):
            l0[c * N + k] = l1[c * (2 * N - 1) + k - 1] + noise * torch.randn(V, generator=g)
    return dict(logits0=l0.to(dtype), logits1=l1.to(dtype),
                qo0=torch.arange(0, C * N + 1, N, dtype=torch.int32),
                qo1=torch.arange(0, C * (2 * N - 1) + 1, 2 * N - 1, dtype=torch.int32),
                mode0=torch.zeros(C, dtype=torch.uint8))


@pytest.mark.parametrize("N", [2, 3, 8, 16])
def test_other_strides(cuda_device, N):
    b = _small_batch(32, N, 4096, seed=N)
    _check_pair(b, N, 1.0, isd.PROPOSE_ARGMAX, 1, 7)


def test_sample_mode_proposals(cuda_device):
    b = _small_batch(32, 4, 20000, seed=4)
    _check_pair(b, 4, 1.0, isd.PROPOSE_SAMPLE, 5, 9)


def test_temperature_other_than_one(cuda_device):
    b = _small_batch(24, 4, 8192, seed=6)
    _check_pair(b, 4, 0.7, isd.PROPOSE_ARGMAX, 2, 3)


def test_greedy_temperature_zero(cuda_device):
    b = _small_batch(24, 4, 8192, seed=8)
    _check_pair(b, 4, 0.0, isd.PROPOSE_ARGMAX, 2, 3, greedy=True)


def test_ragged_vocab_tail(cuda_device):
    # V not a multiple of the 8192-entry chunk: 3 chunks, the last one short
    b = _small_batch(16, 4, 8192 * 2 + 136, seed=9)
    _check_pair(b, 4, 1.0, isd.PROPOSE_ARGMAX, 0, 11)


def test_mixed_full_and_fresh_batch(cuda_device):
    C, N, V = 16, 4, 4096
    g = torch.Generator().manual_seed(10)
    mode = torch.tensor([1, 0] * (C // 2), dtype=torch.uint8)
    rows = torch.where(mode == 1, 2 * N - 1, N)
    qo = torch.zeros(C + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(rows, 0).to(torch.int32)
    logits = (torch.randn(int(qo[-1]), V, generator=g) * 2).bfloat16()
    prev = (torch.randn(C * (N - 1), V, generator=g) * 2).bfloat16()
    prow = torch.arange(0, C * (N - 1), N - 1, dtype=torch.int32)
    # drafts: argmax of the previous rows (as the previous step would have proposed)
    drafts = prev.float().argmax(-1).reshape(C, N - 1).to(torch.int32)
    pm = f64(prev)
    m = pm.max(-1)
    s = np.exp(pm - m[:, None]).sum(-1)
    dq = torch.from_numpy(np.stack([m, s], -1).reshape(C, N - 1, 2).astype(np.float32))
    dev = "cuda"
    gout = gpu_accept(logits.to(dev), qo.to(dev), mode.to(dev), drafts.to(dev), dq.to(dev),
                      prev.to(dev), prow.to(dev), N, 1.0, isd.PROPOSE_ARGMAX, 0, 5)
    o = isd.isd_accept(f64(logits), qo.numpy(), mode.numpy().astype(np.int64), drafts.numpy(),
                       pm, prow.numpy(), N, 1.0, isd.PROPOSE_ARGMAX, 0, 5)
    st = compare_accept(gout, o, N)
    assert st["compared"] >= C - 2


def test_bad_draft_token_sets_status(cuda_device):
    b = _small_batch(4, 4, 4096, seed=12)
    dev = "cuda"
    C, N = 4, 4
    l0, l1 = b["logits0"].to(dev), b["logits1"].to(dev)
    drafts = torch.full((C, N - 1), 5000, dtype=torch.int32, device=dev)   # >= V
    dq = torch.ones((C, N - 1, 2), dtype=torch.float32, device=dev)
    prow = torch.arange(0, C * N, N, dtype=torch.int32, device=dev) + 1
    out = gpu_accept(l1, b["qo1"].to(dev), torch.ones(C, dtype=torch.uint8, device=dev), drafts,
                     dq, l0, prow, N, 1.0, 0, 0, 0)
    assert out["status"] == 2


def test_row_layout_mismatch_sets_status(cuda_device):
    b = _small_batch(4, 4, 4096, seed=13)
    dev = "cuda"
    C, N = 4, 4
    l1 = b["logits1"].to(dev)
    drafts = torch.zeros((C, N - 1), dtype=torch.int32, device=dev)
    dq = torch.ones((C, N - 1, 2), dtype=torch.float32, device=dev)
    prow = torch.zeros(C, dtype=torch.int32, device=dev)
    # FRESH modes but FULL-sized rows
    out = gpu_accept(l1, b["qo1"].to(dev), torch.zeros(C, dtype=torch.uint8, device=dev), drafts,
                     dq, l1, prow, N, 1.0, 0, 0, 0)
    assert out["status"] == 3


def test_more_requests_than_sms(cuda_device):
    """C = 320 requests over one CTA per SM: a CTA's request warp decides
    several requests, in the order their chunks finish."""
    C, N, V = 320, 4, 4096
    b = _small_batch(C, N, V, seed=21)
    s0, s1, _ = _check_pair(b, N, 1.0, isd.PROPOSE_ARGMAX, 2, 8)
    assert s1["compared"] >= C - 8


def test_graph_replays_with_new_logits(cuda_device):
    """One accept launch captured in a CUDA graph and replayed with new logits
    in its input buffers each time equals an eager call on those logits, bit
    for bit: the chunk tags of one replay never read as another's."""
    import speculative_verify_accept_step_b300 as lib
    from _gpu import alloc_accept, status_tensor
    C, N, V = 24, 4, 16384
    dev = "cuda"
    M = N - 1
    T = C * (2 * N - 1)
    qo = torch.arange(0, T + 1, 2 * N - 1, dtype=torch.int32, device=dev)
    mode = torch.ones(C, dtype=torch.uint8, device=dev)
    prow = torch.arange(0, C * M, M, dtype=torch.int32, device=dev)
    logits = torch.empty((T, V), dtype=torch.bfloat16, device=dev)
    prev = torch.empty((C * M, V), dtype=torch.bfloat16, device=dev)
    drafts = torch.empty((C, M), dtype=torch.int32, device=dev)
    dq = torch.empty((C, M, 2), dtype=torch.float32, device=dev)

    def fill(seed):
        g = torch.Generator().manual_seed(seed)
        pv = torch.randn(C * M, V, generator=g) * 2
        lg = torch.randn(T, V, generator=g) * 2
        for c in range(C):   # verifying rows close to the proposing rows
            lg[c * (2 * N - 1):c * (2 * N - 1) + M] = pv[c * M:(c + 1) * M] + \
                0.5 * torch.randn(M, V, generator=g)
        prev.copy_(pv.bfloat16())
        logits.copy_(lg.bfloat16())
        drafts.copy_(prev.float().argmax(-1).reshape(C, M).to(torch.int32))
        pf = prev.float()
        m = pf.max(-1).values
        dq.copy_(torch.stack([m, torch.exp(pf - m[:, None]).sum(-1)], -1).reshape(C, M, 2))

    def call(o, ws, st):
        lib.idlm_isd_accept(logits, qo, mode, drafts, dq, prev, prow, N, 1.0,
                            isd.PROPOSE_SAMPLE, 9, 4, o["n_accepted"], o["out_tokens"],
                            o["n_out"], o["n_commit"], o["next_drafts"], o["next_q_stats"],
                            o["next_mode"], o["next_mask_row0"], ws, st,
                            row_stats=o["row_stats"], dbg=o["dbg"])

    size = lib.idlm_isd_accept_workspace_size(C, T, N, V)
    ws_g = torch.empty(size, dtype=torch.uint8, device=dev)
    ws_e = torch.empty(size, dtype=torch.uint8, device=dev)
    og, oe = alloc_accept(C, N, T, dev), alloc_accept(C, N, T, dev)
    st_g, st_e = status_tensor(dev), status_tensor(dev)
    fill(100)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            call(og, ws_g, st_g)
    seen_residual = False
    for seed in (101, 102, 103, 104):
        fill(seed)
        graph.replay()
        call(oe, ws_e, st_e)
        torch.cuda.synchronize()
        assert int(st_g.item()) == 0 and int(st_e.item()) == 0
        for k in og:
            assert torch.equal(og[k], oe[k]), f"seed {seed}: {k}"
        seen_residual |= bool((oe["next_mode"] == 0).any())
    assert seen_residual
