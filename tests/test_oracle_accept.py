"""Pins of the oracle's ISD accept step (CPU only).

* the TPF closed form against the values the pages print;
* the closed form reproduced by running the oracle's own multi-step loop on a
  toy model whose drafts pass with a known probability (within 1%);
* the emitted tokens follow p (chi-square, alpha = 0.001, ~10^6 tokens) and,
  on a Markov toy model, the first three emitted tokens follow the chain's
  law (64 cells): this checks which row verifies which draft;
* greedy (T = 0) ISD emits exactly the greedy autoregressive sequence;
* single-step special cases (ratio >= 1 always passes, p(d) = 0 always fails,
  the residual's support, FRESH rows).

The ARGMAX-proposal acceptance numbers have no value on the pages to compare
with: parity unpinned beyond the definitions above.
"""
import os

import numpy as np
import pytest

from oracle import isd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_tpf.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([float(x) for x in line.split()])
    return rows


def test_closed_form_matches_printed_values():
    rows = _golden_rows()
    assert rows
    for N, p, tpf, tol, eff, etol in rows:
        got = isd.tpf_closed_form(p, int(N))
        assert abs(got - tpf) <= tol
        assert abs(isd.compute_efficiency(got, int(N)) - eff) <= etol


@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_closed_form_limits(N):
    assert isd.tpf_closed_form(1.0, N) == pytest.approx(N)      # every draft passes
    assert isd.tpf_closed_form(0.0, N) == pytest.approx(1.0)    # autoregressive


# ---------------------------------------------------------------- toy models

def iid_model(P, Q):
    lp, lq = np.log(P), np.log(Q)

    def model(row_tok, row_req, row_mask_k, row_last_clean):
        return np.where((row_mask_k > 0)[:, None], lq[None, :], lp[None, :])
    return model


def markov_model(Mt, Qk):
    lm, lq = np.log(Mt), np.log(Qk)

    def model(row_tok, row_req, row_mask_k, row_last_clean):
        out = np.empty((row_tok.shape[0], Mt.shape[0]))
        clean = row_mask_k == 0
        out[clean] = lm[row_tok[clean]]
        out[~clean] = lq[row_mask_k[~clean] - 1, row_last_clean[~clean]]
        return out
    return model


@pytest.mark.parametrize("N", [2, 3, 4, 8])
@pytest.mark.parametrize("alpha", [0.5, 0.9, 0.99])
def test_tpf_simulation_matches_closed_form(N, alpha):
    # V = 2: P = (0.75, 0.25), Q shifted by delta: sum(min(P, Q)) = 1 - delta
    delta = 1.0 - alpha
    P = np.array([0.75, 0.25])
    Q = np.array([0.75 - delta, 0.25 + delta])
    C, steps, burn = 8192, 40, 8
    _, _, per_step = isd.isd_decode(iid_model(P, Q), np.zeros(C, dtype=np.int64), N,
                                    steps, 1.0, isd.PROPOSE_SAMPLE, seed=11, step0=0)
    tpf = per_step[burn:].mean()
    assert tpf == pytest.approx(isd.tpf_closed_form(alpha, N), rel=0.01)


def _chi2(counts, probs):
    exp = probs * counts.sum()
    return float(((counts - exp) ** 2 / exp).sum())


def test_emitted_tokens_follow_p_chi_square():
    rng = np.random.default_rng(5)
    V, N = 8, 4
    P = rng.dirichlet(np.ones(V) * 2)
    Q = rng.dirichlet(np.ones(V) * 2)
    C, steps = 120_000, 5
    emitted, n, _ = isd.isd_decode(iid_model(P, Q), np.zeros(C, dtype=np.int64), N,
                                   steps, 1.0, isd.PROPOSE_SAMPLE, seed=3)
    toks = emitted[emitted >= 0]
    assert toks.size > 1_000_000
    counts = np.bincount(toks, minlength=V)
    # 7 degrees of freedom: the 0.999 quantile is 24.32
    assert _chi2(counts, P) < 24.32


def test_argmax_proposals_are_not_distribution_preserving():
    # power check of the chi-square above: ARGMAX proposals change the law
    rng = np.random.default_rng(5)
    V, N = 8, 4
    P = rng.dirichlet(np.ones(V) * 2)
    Q = rng.dirichlet(np.ones(V) * 2)
    emitted, _, _ = isd.isd_decode(iid_model(P, Q), np.zeros(50_000, dtype=np.int64), N,
                                   5, 1.0, isd.PROPOSE_ARGMAX, seed=3)
    toks = emitted[emitted >= 0]
    assert _chi2(np.bincount(toks, minlength=V), P) > 100.0


def test_markov_chain_first_three_tokens():
    rng = np.random.default_rng(9)
    V, N = 4, 4
    Mt = rng.dirichlet(np.ones(V) * 2, size=V)
    Qk = rng.dirichlet(np.ones(V) * 2, size=(N - 1, V))
    C = 300_000
    x0 = 0
    emitted, n, _ = isd.isd_decode(markov_model(Mt, Qk), np.full(C, x0), N, 3,
                                   1.0, isd.PROPOSE_SAMPLE, seed=21)
    assert np.all(n >= 3)
    cells = emitted[:, 0] * V * V + emitted[:, 1] * V + emitted[:, 2]
    counts = np.bincount(cells, minlength=V ** 3).astype(np.float64)
    probs = np.array([Mt[x0, a] * Mt[a, b] * Mt[b, c]
                      for a in range(V) for b in range(V) for c in range(V)])
    exp = probs * C
    small = exp < 5
    if small.any():     # pool sparse cells into one bin
        counts = np.append(counts[~small], counts[small].sum())
        probs = np.append(probs[~small], probs[small].sum())
    dof = counts.size - 1
    chi2 = _chi2(counts, probs)
    # 0.999 quantile of chi-square(63) is 103.4; scale down if cells were pooled
    from scipy.stats import chi2 as chi2dist
    assert chi2 < chi2dist.ppf(0.999, dof)


def test_markov_wrong_verifier_row_is_detected():
    # planted mistake, oracle side: verifying draft i against the row of draft i
    # instead of the row before it must break the chain's law
    rng = np.random.default_rng(9)
    V, N = 4, 4
    Mt = rng.dirichlet(np.ones(V) * 2, size=V)
    Qk = rng.dirichlet(np.ones(V) * 2, size=(N - 1, V))
    good = markov_model(Mt, Qk)

    def shifted(row_tok, row_req, row_mask_k, row_last_clean):
        out = good(row_tok, row_req, row_mask_k, row_last_clean)
        # clean rows predict from the NEXT row's token: an off-by-one shift
        nxt = np.roll(out, -1, axis=0)
        clean_next = np.roll(row_mask_k == 0, -1) & (row_mask_k == 0)
        out[clean_next] = nxt[clean_next]
        return out
    C = 100_000
    emitted, _, _ = isd.isd_decode(shifted, np.zeros(C, dtype=np.int64), N, 3,
                                   1.0, isd.PROPOSE_SAMPLE, seed=21)
    cells = emitted[:, 0] * 16 + emitted[:, 1] * 4 + emitted[:, 2]
    counts = np.bincount(cells, minlength=64).astype(np.float64)
    probs = np.array([Mt[0, a] * Mt[a, b] * Mt[b, c]
                      for a in range(V) for b in range(V) for c in range(V)])
    assert _chi2(counts, probs) > 1000.0


def test_greedy_isd_equals_greedy_autoregression():
    rng = np.random.default_rng(13)
    V, N = 16, 4
    Mt = rng.random((V, V)) + 0.01
    Mt /= Mt.sum(1, keepdims=True)
    Qk = rng.random((N - 1, V, V)) + 0.01
    Qk /= Qk.sum(2, keepdims=True)
    C = 64
    start = np.arange(C) % V
    emitted, n, _ = isd.isd_decode(markov_model(Mt, Qk), start, N, 12, 0.0,
                                   isd.PROPOSE_ARGMAX, seed=0)
    for c in range(C):
        x = start[c]
        for t in range(n[c]):
            x = int(np.argmax(Mt[x]))
            assert emitted[c, t] == x
    # drafts were wrong sometimes, so the test exercised rejections
    assert n.min() < 12 * N


# ----------------------------------------------------------- single steps

def _one_step(logits, mode, drafts, prev, prev_row0, N, T=1.0, pm=isd.PROPOSE_ARGMAX,
              seed=0, step=0):
    rows = isd.rows_per_request(np.asarray(mode), N)
    qo = np.concatenate([[0], np.cumsum(rows)])
    return isd.isd_accept(logits, qo, np.asarray(mode), np.asarray(drafts), prev,
                          np.asarray(prev_row0), N, T, pm, seed, step)


def test_fresh_request_draws_one_token_and_proposes():
    rng = np.random.default_rng(0)
    N, V = 4, 50
    logits = rng.standard_normal((N, V)) * 2
    out = _one_step(logits, [isd.FRESH], np.full((1, N - 1), -1), np.zeros((1, V)), [0], N)
    assert out["n_accepted"][0] == 0 and out["n_out"][0] == 1 and out["n_commit"][0] == 1
    assert out["next_mode"][0] == isd.FULL
    assert list(out["next_drafts"][0]) == list(np.argmax(logits[1:], axis=1))
    assert out["next_mask_row0"][0] == 1
    assert out["final_kind"][0] == isd.END_FRESH


def test_ratio_at_least_one_always_passes():
    rng = np.random.default_rng(1)
    N, V = 4, 40
    C = 200
    prev = rng.standard_normal((C * (N - 1), V))
    logits = np.zeros((C * (2 * N - 1), V))
    for c in range(C):
        for i in range(1, N):
            logits[c * (2 * N - 1) + i - 1] = prev[c * (N - 1) + i - 1]   # p_i = q_i
        logits[c * (2 * N - 1) + N - 1:(c + 1) * (2 * N - 1)] = rng.standard_normal((N, V))
    drafts = rng.integers(0, V, size=(C, N - 1))
    out = _one_step(logits, np.ones(C, dtype=int), drafts, prev, np.arange(C) * (N - 1), N)
    assert np.all(out["n_accepted"] == N - 1)
    assert np.all(out["final_kind"] == isd.END_BONUS)
    assert np.array_equal(out["out_tokens"][:, :N - 1], drafts)
    assert np.all(out["n_commit"] == N)


def test_zero_anchor_probability_always_rejects_and_residual_support():
    rng = np.random.default_rng(2)
    N, V = 3, 30
    C = 300
    prev = rng.standard_normal((C * (N - 1), V))
    logits = rng.standard_normal((C * (2 * N - 1), V))
    drafts = rng.integers(0, V, size=(C, N - 1))
    for c in range(C):
        logits[c * (2 * N - 1), drafts[c, 0]] = -1e4     # p_1(d_1) = 0
    out = _one_step(logits, np.ones(C, dtype=int), drafts, prev, np.arange(C) * (N - 1), N)
    assert np.all(out["n_accepted"] == 0)
    assert np.all(out["final_kind"] == isd.END_RESIDUAL)
    P = isd.softmax_t(logits, 1.0)
    Qd = isd.softmax_t(prev, 1.0)
    for c in range(C):
        tok = out["out_tokens"][c, 0]
        assert P[c * (2 * N - 1), tok] > Qd[c * (N - 1), tok]
    assert np.all(out["next_mode"] == isd.FRESH)
    assert np.all(out["next_drafts"] == -1)
    assert np.all(out["n_commit"] == 1)


def test_bad_row_layout_is_rejected():
    with pytest.raises(ValueError):
        isd.isd_accept(np.zeros((5, 4)), np.array([0, 5]), np.array([1]), np.zeros((1, 2), int),
                       np.zeros((2, 4)), np.array([0]), 4, 1.0, 0, 0, 0)


def test_decode_positions_feed_each_slot_its_own_rows():
    """isd_decode(with_positions=True) gives the model every row's absolute
    position.  With the slot-indexed synthetic model of the workloads, a
    draft is proposed from the MASK row of its slot at one step and verified
    against the clean row of the same slot at the next, so in SAMPLE mode
    the realised acceptance equals the mean overlap sum_v min(p_v, q_v) of
    those row pairs; a position off by one would pair unrelated rows."""
    from speculative_verify_accept_step_b300 import workloads as wl
    C, N, V, steps, seed = 300, 4, 256, 8, 2
    sz = wl.synth_scale(2.0)
    se = np.full(C, wl.synth_scale(0.6), dtype=np.float32)
    step = [0]
    tested = accepted = 0

    def model(row_tok, row_req, row_mask_k, row_last_clean, row_pos):
        bits = wl.synth_rows(row_req, row_pos, row_tok == isd.MASK_TOKEN, V, sz, se, seed,
                             step[0])
        step[0] += 1
        return wl.bf16_bits_to_f32(bits).astype(np.float64)

    outs = []
    orig = isd.isd_accept

    def traced(*a, **k):
        o = orig(*a, **k)
        outs.append(o)
        return o
    isd.isd_accept = traced
    try:
        start = np.arange(C) % 50
        isd.isd_decode(model, np.zeros(C, dtype=np.int64), N, steps, 1.0, isd.PROPOSE_SAMPLE,
                       seed, start_len=start, with_positions=True)
    finally:
        isd.isd_accept = orig
    for o in outs:
        full = o["final_kind"] != isd.END_FRESH
        n = o["n_accepted"][full]
        tested += int(np.minimum(n + 1, N - 1).sum())
        accepted += int(n.sum())
    p_hat = accepted / tested
    # expected overlap of a slot's MASK row (some step) with its clean row
    slots = np.arange(400) + 7
    req = np.arange(400) % C
    p = wl.bf16_bits_to_f32(wl.synth_rows(req, slots, np.zeros(400, bool), V, sz, se, seed, 0))
    q = wl.bf16_bits_to_f32(wl.synth_rows(req, slots, np.ones(400, bool), V, sz, se, seed, 0))
    overlap = np.minimum(isd.softmax_t(p.astype(np.float64), 1.0),
                         isd.softmax_t(q.astype(np.float64), 1.0)).sum(-1).mean()
    assert 0.3 < overlap < 0.95
    assert abs(p_hat - overlap) < 0.02, (p_hat, overlap)
