"""GPU tests of the stationary-batch decode loop (marked gpu).

Source: "Introspective Diffusion Language Models" (project page), section
"Serving (SGLang)" (stationary-batch decode loop replayed from a CUDA graph)
and the speedup panel (memory-bound TPF = (2 + p + ... + p^(N-2)) /
(2 - p^(N-1)) at per-draft acceptance p).

* The synthetic model's rows equal their CPU twin (workloads.synth_rows) bit
  for bit.
* K steps of the loop emit the same tokens as the oracle's decode loop fed
  the same synthetic model, request by request, until the first decision
  the oracle marks ambiguous (|u - min(1, ratio)| <= 1e-5 or a CDF margin
  <= 1e-5 of the total).
* One CUDA graph of K steps gives the same bits as K eager steps.
* Tokens per forward measured on the GPU over >= 10^4 request-steps match
  the closed form at the acceptance the loop realised (within 1%), and the
  closed form at the calibrated target (within 2%).
"""
import json
import os

import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from oracle import isd
from speculative_verify_accept_step_b300 import workloads as wl
from speculative_verify_accept_step_b300.loop import StationaryLoop

pytestmark = pytest.mark.gpu

AMBIG = 1e-5


def synth_sigma(target):
    path = os.path.join(os.path.dirname(wl.__file__), "synth_noise_table.json")
    with open(path) as f:
        return float(json.load(f)["sigma"][str(target)])


def test_synth_rows_bit_exact(cuda_device):
    C, N, V = 5, 4, 1024
    first = torch.tensor([3, 1, 4, 1, 5])
    start = torch.tensor([0, 7, 100, 33, 2])
    sig = [0.3, 0.5, 0.25, 1.0, 0.1]
    lp = StationaryLoop(C, N, V, first, start, sig, steps=2, seed=17)
    # step 0: every request FRESH (1 clean + N-1 MASK rows)
    lib.idlm_synth_logits(lp.logits[0], lp.qo, lp.row_req, lp.row_pos, lp.row_token,
                          lp.scale_z, lp.scale_e, 17, 9)
    torch.cuda.synchronize()
    T = int(lp.qo[-1])
    assert T == C * N
    req = lp.row_req[:T].cpu().numpy()
    pos = lp.row_pos[:T].cpu().numpy()
    tok = lp.row_token[:T].cpu().numpy()
    assert np.array_equal(pos, np.repeat(start.numpy(), N) + np.tile(np.arange(N), C))
    assert np.array_equal(tok, np.where(np.tile(np.arange(N), C) == 0,
                                        np.repeat(first.numpy(), N), -1))
    want = wl.synth_rows(req, pos, tok < 0, V, lp.scale_z, lp.scale_e.cpu().numpy(), 17, 9)
    got = lp.logits[0][:T].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def _oracle_decode(C, N, V, first, start, sig, steps, seed, T, pm):
    sz = wl.synth_scale(3.0)
    se = np.array([wl.synth_scale(s) for s in sig], dtype=np.float32)
    calls = []

    def model(row_tok, row_req, row_mask_k, row_last_clean, row_pos):
        s = len(calls)
        calls.append(s)
        bits = wl.synth_rows(row_req, row_pos, row_tok == isd.MASK_TOKEN, V, sz, se, seed, s)
        return wl.bf16_bits_to_f32(bits).astype(np.float64)

    trace = []
    orig = isd.isd_accept

    def traced(*a, **k):
        out = orig(*a, **k)
        trace.append(out)
        return out
    isd.isd_accept = traced
    try:
        emitted, n_emitted, per_step = isd.isd_decode(model, first, N, steps, T, pm, seed,
                                                      start_len=start, with_positions=True)
    finally:
        isd.isd_accept = orig
    return emitted, n_emitted, per_step, trace


def _first_ambiguous_step(trace, c, N, greedy):
    """Index of the first step whose decision for request c is ambiguous."""
    for s, o in enumerate(trace):
        if o["final_kind"][c] != isd.END_FRESH:
            for i in range(min(N - 1, int(o["n_accepted"][c]) + 1)):
                if abs(o["u"][c, i] - min(1.0, o["ratio"][c, i])) <= AMBIG:
                    return s
        if not greedy and o["final_margin"][c] <= AMBIG:
            return s
        if np.any(o["propose_margin"][c] <= AMBIG):
            return s
    return len(trace)


@pytest.mark.parametrize("N,pm,T", [(4, lib.PROPOSE_ARGMAX, 1.0), (4, lib.PROPOSE_SAMPLE, 1.0),
                                    (3, lib.PROPOSE_ARGMAX, 0.8)])
def test_loop_matches_the_oracle_decode_loop(cuda_device, N, pm, T):
    # V small enough that few draws land within 1e-5 of a CDF edge (about
    # 2e-5 V of them do): those are ambiguous, and a request is compared
    # only up to its first ambiguous decision
    C, V, steps, seed = 16, 512, 6, 5
    g = torch.Generator().manual_seed(N)
    first = torch.randint(0, V, (C,), generator=g)
    start = torch.randint(0, 300, (C,), generator=g)
    sig = [0.4 if c % 3 else 1.2 for c in range(C)]
    lp = StationaryLoop(C, N, V, first, start, sig, steps=steps, seed=seed, temperature=T,
                        proposal_mode=pm)
    lp.run()
    r = lp.results()
    assert r["status"] == 0
    emitted, n_emitted, per_step, trace = _oracle_decode(
        C, N, V, first.numpy(), start.numpy(), sig, steps, seed, T, pm)
    compared = 0
    for c in range(C):
        s_amb = _first_ambiguous_step(trace, c, N, greedy=False)
        n_ok = int(per_step[:s_amb, c].sum())
        hist = r["history"][c].numpy()
        assert np.array_equal(hist[:n_ok], emitted[c, :n_ok]), f"request {c}"
        if s_amb == steps:
            compared += 1
            assert int(r["hist_len"][c]) == int(n_emitted[c])
            assert int(r["tokens"][c]) == int(n_emitted[c])
            assert int(r["forwards"][c]) == steps
            assert int(r["seq_lens"][c]) == int(start[c]) + sum(
                int(o["n_commit"][c]) for o in trace)
    assert compared >= C // 2
    # both kinds of transition happened
    kinds = set(np.concatenate([o["final_kind"] for o in trace]).tolist())
    assert isd.END_FRESH in kinds and (isd.END_BONUS in kinds or isd.END_RESIDUAL in kinds)


def test_graph_replay_equals_eager_steps(cuda_device):
    C, N, V, steps = 16, 4, 4096, 8
    first = torch.arange(C) * 7
    start = torch.full((C,), 64)
    sig = [0.3] * C
    a = StationaryLoop(C, N, V, first, start, sig, steps=steps, seed=3,
                       attention=dict(Hq=32, Hkv=8, D=128))
    a.run(graph=False)
    ra = a.results()
    b = StationaryLoop(C, N, V, first, start, sig, steps=steps, seed=3,
                       attention=dict(Hq=32, Hkv=8, D=128))
    b.run(graph=True)
    rb = b.results()
    assert ra["status"] == 0 and rb["status"] == 0
    for k in ("tokens", "forwards", "accepted", "tested", "history", "hist_len", "seq_lens"):
        assert torch.equal(ra[k], rb[k]), k
    assert torch.equal(a.k_cache, b.k_cache)


@pytest.mark.parametrize("target,steps", [(0.5, 200), (0.9, 400), (0.99, 200)])
def test_tokens_per_forward_matches_the_closed_form(cuda_device, target, steps):
    """SAMPLE-mode proposals, so that a draft passes with probability
    sum_v min(p_v, q_v), the overlap the synthetic model's noise is set for.
    C = 64 requests x `steps` forwards (>= 12800 request-steps), N = 4,
    V = 151936, all on the device in one CUDA graph."""
    C, N, V = 64, 4, 151936
    first = torch.arange(C)
    start = torch.full((C,), 4096)
    lp = StationaryLoop(C, N, V, first, start, [synth_sigma(target)] * C, steps=steps, seed=11,
                        proposal_mode=lib.PROPOSE_SAMPLE, hist_cap=8)
    lp.run(graph=True)
    r = lp.results()
    assert r["status"] == 0
    tokens, forwards = int(r["tokens"].sum()), int(r["forwards"].sum())
    assert forwards == C * steps
    p_hat = float(r["accepted"].sum()) / float(r["tested"].sum())
    tpf = tokens / forwards
    closed_hat = isd.tpf_closed_form(p_hat, N)
    closed_target = isd.tpf_closed_form(target, N)
    assert abs(p_hat - target) < 0.01, f"realised acceptance {p_hat:.4f} vs target {target}"
    assert abs(tpf / closed_hat - 1) < 0.01, f"TPF {tpf:.4f} vs closed form {closed_hat:.4f}"
    assert abs(tpf / closed_target - 1) < 0.02, f"TPF {tpf:.4f} vs {closed_target:.4f}"


@pytest.mark.parametrize("C,N", [(1, 2), (600, 4), (300, 16)])
def test_advance_layout_over_several_ctas(cuda_device, C, N):
    """The hand-off written request by request on the CPU from the row
    layout of section "Inference & ISD": FULL rows [anchor, d_1 .. d_{N-1},
    MASK x (N-1)], FRESH rows [anchor, MASK x (N-1)], at positions L, L+1,
    ...; C = 600 spans three CTAs of requests and a ragged last one.  One
    request with no emitted token is flagged and its rows left unwritten;
    the history of a request that overflows hist_cap is cut at hist_cap."""
    g = torch.Generator().manual_seed(C + N)
    M = N - 1
    mode = torch.randint(0, 2, (C,), generator=g, dtype=torch.uint8)
    next_mode = torch.randint(0, 2, (C,), generator=g, dtype=torch.uint8)
    n_out = torch.randint(1, N + 1, (C,), generator=g, dtype=torch.int32)
    bad = C // 2 if C > 1 else -1
    if bad >= 0:
        n_out[bad] = 0
    n_acc = (n_out - 1).clamp(min=0)
    out_tokens = torch.randint(0, 1 << 20, (C, N), generator=g, dtype=torch.int32)
    drafts = torch.randint(0, 1 << 20, (C, M), generator=g, dtype=torch.int32)
    seq = torch.randint(0, 5000, (C,), generator=g, dtype=torch.int32)
    rows = torch.tensor(isd.rows_per_request(next_mode.numpy(), N), dtype=torch.int64)
    T = C * (2 * N - 1) + 5
    cap = 6
    hist_len = torch.randint(0, cap + 1, (C,), generator=g, dtype=torch.int32)
    history = torch.randint(0, 9, (C, cap), generator=g, dtype=torch.int32)
    counters = torch.randint(0, 50, (4, C), generator=g, dtype=torch.int32)
    d = lambda x: x.to(cuda_device)
    qo, rr, rp, rt = (torch.full((n,), -7, dtype=torch.int32, device=cuda_device)
                      for n in (C + 1, T, T, T))
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    cnt_d, hist_d, hl_d = d(counters.clone()), d(history.clone()), d(hist_len.clone())
    lib.idlm_isd_advance(N, d(mode), d(next_mode), d(out_tokens), d(n_out), d(n_acc), d(drafts),
                         d(seq), qo, rr, rp, rt, status, counters=cnt_d, history=hist_d,
                         hist_len=hl_d, count=True)
    torch.cuda.synchronize()
    want_qo = torch.zeros(C + 1, dtype=torch.int64)
    want_qo[1:] = torch.cumsum(rows, 0)
    assert torch.equal(qo.cpu().long(), want_qo)
    assert int(status.item()) == (3 if bad >= 0 else 0)  # 3: bad layout
    rr, rp, rt = rr.cpu(), rp.cpu(), rt.cpu()
    cnt, hist, hl = cnt_d.cpu(), hist_d.cpu(), hl_d.cpu()
    for c in range(C):
        r0, n = int(want_qo[c]), int(rows[c])
        if c == bad:
            assert torch.all(rr[r0:r0 + n] == -7) and torch.equal(cnt[:, c], counters[:, c])
            assert torch.equal(hist[c], history[c]) and int(hl[c]) == int(hist_len[c])
            continue
        no, ncl = int(n_out[c]), (N if int(next_mode[c]) == lib.MODE_FULL else 1)
        want_tok = [int(out_tokens[c, no - 1])] + [int(drafts[c, k]) for k in range(ncl - 1)]
        want_tok += [-1] * (n - ncl)
        assert rr[r0:r0 + n].tolist() == [c] * n
        assert rp[r0:r0 + n].tolist() == list(range(int(seq[c]), int(seq[c]) + n))
        assert rt[r0:r0 + n].tolist() == want_tok, f"request {c}"
        was_full = int(mode[c]) == lib.MODE_FULL
        na = int(n_acc[c])
        assert cnt[:, c].tolist() == [int(counters[0, c]) + no, int(counters[1, c]) + 1,
                                      int(counters[2, c]) + na,
                                      int(counters[3, c]) + (min(na + 1, M) if was_full else 0)]
        h = int(hist_len[c])
        want_h = history[c].clone()
        for k in range(no):
            if h + k < cap:
                want_h[h + k] = out_tokens[c, k]
        assert torch.equal(hist[c], want_h) and int(hl[c]) == min(h + no, cap)
    used = int(want_qo[C])
    assert torch.all(rr[used:] == 0) and torch.all(rp[used:] == 0) and torch.all(rt[used:] == -2)
