"""GPU parity of idlm_lm_head_accept, the LM head fused with the accept step
(marked gpu).

Source: "Introspective Diffusion Language Models" (project page), section
"Inference & ISD": p (clean rows) and q (MASK rows) both come from the one
forward pass, whose last product is the LM head.

Each case runs a FRESH step and then a FULL step through the fused call,
from hidden states built so that the FULL step's verifying rows resemble the
FRESH step's proposing rows (so drafts are accepted as well as rejected):
* the logits it writes match hidden @ w_vocab^T (float64) within the bf16
  GEMM bound used for the gated-LoRA projections;
* every output of both steps matches the oracle's accept step run on those
  same logits (decisions compared up to the oracle's ambiguity margin);
* the per-row softmax statistics taken in the GEMM's epilogue equal those of
  the unfused accept (its own pass over the same logits) to fp32 rounding.
"""
import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from _gpu import alloc_accept, compare_accept, f64, gpu_accept, run_two_steps_oracle, status_tensor
from oracle import isd

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2


def _hidden_pair(C, N, H, V, seed, noise=0.35):
    """Hidden states of a FRESH step (C N rows) and the FULL step after it
    (C (2N - 1) rows, clean row k - 1 close to the FRESH step's MASK row k),
    and LM-head weights giving logits of standard deviation ~2."""
    g = torch.Generator().manual_seed(seed)
    h0 = torch.randn(C * N, H, generator=g)
    h1 = torch.randn(C * (2 * N - 1), H, generator=g)
    for c in range(C):
        for k in range(1, N):
            h1[c * (2 * N - 1) + k - 1] = h0[c * N + k] + noise * torch.randn(H, generator=g)
    w = torch.randn(V, H, generator=g) * (2.0 / H ** 0.5)
    return h0.bfloat16(), h1.bfloat16(), w.bfloat16()


def _fused(h, w, logits, qo, mode, drafts, dq, prev, prow, N, temperature, pm, seed, step,
           dev="cuda"):
    T, H = h.shape
    V = w.shape[0]
    C = mode.shape[0]
    o = alloc_accept(C, N, T, dev)
    ws = torch.empty(lib.idlm_lm_head_accept_workspace_size(C, T, N, H, V), dtype=torch.uint8,
                     device=dev)
    st = status_tensor(dev)
    lib.idlm_lm_head_accept(h, w, logits, qo, mode, drafts, dq, prev, prow, N, temperature, pm,
                            seed, step, o["n_accepted"], o["out_tokens"], o["n_out"],
                            o["n_commit"], o["next_drafts"], o["next_q_stats"], o["next_mode"],
                            o["next_mask_row0"], ws, st, row_stats=o["row_stats"], dbg=o["dbg"])
    torch.cuda.synchronize()
    o["status"] = int(st.item())
    return o


def _check_logits(logits, h, w, samples=None):
    got = f64(logits)
    hf, wf = f64(h), f64(w)
    if samples is None:
        ref = hf @ wf.T
        err, bound = np.abs(got - ref), ATOL + RTOL * np.abs(ref)
    else:
        rng = np.random.default_rng(0)
        ms = rng.integers(0, got.shape[0], samples)
        ns = rng.integers(0, got.shape[1], samples)
        ref = np.einsum("ij,ij->i", hf[ms], wf[ns])
        err, bound = np.abs(got[ms, ns] - ref), ATOL + RTOL * np.abs(ref)
    assert np.all(err <= bound), f"worst err/bound {float((err / bound).max()):.3f}"


def _run(C, N, H, V, temperature, pm, seed, step0, full_logit_check=True, greedy=False):
    dev = "cuda"
    M = N - 1
    h0, h1, w = _hidden_pair(C, N, H, V, seed)
    h0, h1, w = h0.to(dev), h1.to(dev), w.to(dev)
    qo0 = torch.arange(0, C * N + 1, N, dtype=torch.int32, device=dev)
    qo1 = torch.arange(0, C * (2 * N - 1) + 1, 2 * N - 1, dtype=torch.int32, device=dev)
    l0 = torch.empty(C * N, V, dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(C * (2 * N - 1), V, dtype=torch.bfloat16, device=dev)
    drafts = torch.full((C, M), -1, dtype=torch.int32, device=dev)
    dq = torch.zeros((C, M, 2), dtype=torch.float32, device=dev)
    prow = torch.zeros((C,), dtype=torch.int32, device=dev)
    mode0 = torch.zeros(C, dtype=torch.uint8, device=dev)
    g0 = _fused(h0, w, l0, qo0, mode0, drafts, dq, l0, prow, N, temperature, pm, seed, step0)
    g1 = _fused(h1, w, l1, qo1, g0["next_mode"], g0["next_drafts"], g0["next_q_stats"], l0,
                g0["next_mask_row0"], N, temperature, pm, seed, step0 + 1)
    assert g0["status"] == 0 and g1["status"] == 0
    samples = None if full_logit_check else 4096
    _check_logits(l0, h0, w, samples)
    _check_logits(l1, h1, w, samples)
    # the oracle's accept on the logits the fused call wrote
    b = dict(logits0=l0.cpu(), logits1=l1.cpu(), qo0=qo0.cpu(), qo1=qo1.cpu(),
             mode0=mode0.cpu())
    o0, o1 = run_two_steps_oracle(b, N, temperature, pm, seed, step0)
    compare_accept(g0, o0, N, greedy)
    assert np.array_equal(g0["next_drafts"].cpu().numpy(), o0["next_drafts"])
    s1 = compare_accept(g1, o1, N, greedy)
    # statistics from the GEMM's epilogue against the accept's own pass
    u1 = gpu_accept(l1, qo1, g0["next_mode"], g0["next_drafts"], g0["next_q_stats"], l0,
                    g0["next_mask_row0"], N, temperature, pm, seed, step0 + 1)
    a, r = g1["row_stats"].cpu().numpy(), u1["row_stats"].cpu().numpy()
    assert np.allclose(a[:, 0], r[:, 0], rtol=0, atol=1e-6)
    assert np.allclose(a[:, 1], r[:, 1], rtol=2e-5, atol=0)
    return s1, o1


def test_small_argmax(cuda_device):
    s1, o1 = _run(16, 4, 256, 8192, 1.0, isd.PROPOSE_ARGMAX, 3, 10)
    assert s1["compared"] >= 12
    kinds = set(o1["final_kind"].tolist())
    assert isd.END_RESIDUAL in kinds or isd.END_BONUS in kinds


def test_ragged_vocab_tile_sample_mode_temperature(cuda_device):
    # V = 5000: the last 128-entry tile holds 8 entries; SAMPLE proposals, T = 0.7
    s1, _ = _run(8, 4, 512, 5000, 0.7, isd.PROPOSE_SAMPLE, 5, 4)
    assert s1["compared"] >= 6


def test_greedy_temperature_zero(cuda_device):
    _run(8, 3, 256, 4096, 0.0, isd.PROPOSE_ARGMAX, 7, 2, greedy=True)


def test_more_rows_than_one_gemm_slice(cuda_device):
    # 70 requests x 7 rows = 490 rows: two slices of the GEMM's token rows
    s1, _ = _run(70, 4, 128, 2048, 1.0, isd.PROPOSE_ARGMAX, 9, 6)
    assert s1["compared"] >= 60


def test_headline_shape(cuda_device):
    """64 requests, N = 4 (448 rows), hidden 4096, V = 151936: the fused call
    at the size the accept's headline batch has; logits checked on 4096
    sampled entries, every decision against the oracle."""
    s1, _ = _run(64, 4, 4096, 151936, 1.0, isd.PROPOSE_ARGMAX, 0, 0, full_logit_check=False)
    assert s1["compared"] >= 56
