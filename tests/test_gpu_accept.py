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
