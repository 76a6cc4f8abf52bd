"""Helpers shared by the GPU parity tests: run the library through its C ABI
and the oracle on the same seeded inputs, and compare them with the
tolerances of the parity contract:

* bit-exact: page indexing, KV commit, argmax proposals, accepted counts
  wherever every examined |u_i - min(1, ratio_i)| > 1e-5, sampled tokens
  wherever the oracle's CDF margin > 1e-5 of the total;
* attention outputs: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| (bf16 storage,
  fp32 accumulation); fp32 storage: 1e-4 + 1e-4 |oracle|;
* probabilities and softmax sums: 1e-5 relative.
"""
import numpy as np
import torch

import speculative_verify_accept_step_b300 as lib
from oracle import isd

AMBIG = 1e-5
PROB_RTOL = 1e-5


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64) if t.is_floating_point() \
        else t.detach().cpu().numpy()


def status_tensor(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


# ------------------------------------------------------------------ attention

def gpu_attention(a, max_rows, dev="cuda"):
    q = a["q"].to(dev)
    T, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = a["k_cache"].shape
    C = a["page_table"].shape[0]
    dt = lib.IDLM_BF16 if q.dtype == torch.bfloat16 else lib.IDLM_F32
    ws = torch.empty(max(lib.idlm_isd_attention_workspace_size(C, Hq, Hkv, D, page_size, max_rows, dt), 256),
                     dtype=torch.uint8, device=dev)
    out = torch.full_like(q, float("nan"))
    st = status_tensor(dev)
    dv = {k: a[k].to(dev) for k in ("k_new", "v_new", "k_cache", "v_cache", "page_table",
                                    "seq_lens", "qo_indptr")}
    lib.idlm_isd_attention(q, dv["k_new"], dv["v_new"], dv["k_cache"], dv["v_cache"],
                           dv["page_table"], dv["seq_lens"], dv["qo_indptr"], out, ws, st,
                           max_rows=max_rows, sm_scale=a["sm_scale"])
    torch.cuda.synchronize()
    return out, int(st.item())


def oracle_attention(a, requests=None):
    """Oracle outputs for all requests, or only `requests` (rows of others NaN)."""
    qo = a["qo_indptr"].numpy()
    C = len(qo) - 1
    req = range(C) if requests is None else requests
    T = a["q"].shape[0]
    out = np.full((T,) + tuple(a["q"].shape[1:]), np.nan)
    kc, vc = f64(a["k_cache"]), f64(a["v_cache"])
    q, kn, vn = f64(a["q"]), f64(a["k_new"]), f64(a["v_new"])
    pt, sl = a["page_table"].numpy(), a["seq_lens"].numpy()
    P = a["k_cache"].shape[2]
    for c in req:
        t0, t1 = qo[c], qo[c + 1]
        sub_qo = np.array([0, t1 - t0])
        o = isd.isd_attention(q[t0:t1], kn[t0:t1], vn[t0:t1], kc, vc, pt[c:c + 1], sl[c:c + 1],
                              sub_qo, P, a["sm_scale"])
        out[t0:t1] = o
    return out


def assert_attention_close(got, ref, bf16=True):
    g = f64(got)
    mask = ~np.isnan(ref)
    atol, rtol = (2e-2, 1e-2) if bf16 else (1e-4, 1e-4)
    err = np.abs(g[mask] - ref[mask])
    bound = atol + rtol * np.abs(ref[mask])
    worst = float((err / bound).max()) if err.size else 0.0
    assert np.all(err <= bound), f"attention mismatch: worst err/bound = {worst:.3f}"
    return worst


# --------------------------------------------------------------------- accept

def alloc_accept(C, N, T, dev="cuda"):
    M = N - 1
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(
        n_accepted=torch.full((C,), -7, **i32), out_tokens=torch.full((C, N), -7, **i32),
        n_out=torch.full((C,), -7, **i32), n_commit=torch.full((C,), -7, **i32),
        next_drafts=torch.full((C, M), -7, **i32),
        next_q_stats=torch.zeros((C, M, 2), dtype=torch.float32, device=dev),
        next_mode=torch.zeros((C,), dtype=torch.uint8, device=dev),
        next_mask_row0=torch.full((C,), -7, **i32),
        row_stats=torch.zeros((T, 2), dtype=torch.float32, device=dev),
        dbg=torch.zeros((C, M, 4), dtype=torch.float32, device=dev))


def gpu_accept(logits, qo, mode, drafts, dq, prev, prev_row0, N, temperature, pm, seed, step,
               dev="cuda"):
    T, V = logits.shape
    C = mode.shape[0]
    o = alloc_accept(C, N, T, dev)
    ws = torch.empty(lib.idlm_isd_accept_workspace_size(C, T, N, V), dtype=torch.uint8, device=dev)
    st = status_tensor(dev)
    lib.idlm_isd_accept(logits, qo, mode, drafts, dq, prev, prev_row0, N, temperature, pm, seed,
                        step, o["n_accepted"], o["out_tokens"], o["n_out"], o["n_commit"],
                        o["next_drafts"], o["next_q_stats"], o["next_mode"], o["next_mask_row0"],
                        ws, st, row_stats=o["row_stats"], dbg=o["dbg"])
    torch.cuda.synchronize()
    o["status"] = int(st.item())
    return o


def run_two_steps_gpu(b, N, temperature, pm, seed, step0, dev="cuda"):
    """FRESH step on logits0, then FULL step on logits1, all on the GPU."""
    C = b["mode0"].shape[0]
    M = N - 1
    l0, l1 = b["logits0"].to(dev), b["logits1"].to(dev)
    qo0, qo1 = b["qo0"].to(dev), b["qo1"].to(dev)
    drafts = torch.full((C, M), -1, dtype=torch.int32, device=dev)
    dq = torch.zeros((C, M, 2), dtype=torch.float32, device=dev)
    prow = torch.zeros((C,), dtype=torch.int32, device=dev)
    s0 = gpu_accept(l0, qo0, b["mode0"].to(dev), drafts, dq, l0, prow, N, temperature, pm, seed,
                    step0)
    s1 = gpu_accept(l1, qo1, s0["next_mode"], s0["next_drafts"], s0["next_q_stats"], l0,
                    s0["next_mask_row0"], N, temperature, pm, seed, step0 + 1)
    return s0, s1


def run_two_steps_oracle(b, N, temperature, pm, seed, step0):
    C = b["mode0"].shape[0]
    M = N - 1
    l0, l1 = f64(b["logits0"]), f64(b["logits1"])
    o0 = isd.isd_accept(l0, b["qo0"].numpy(), b["mode0"].numpy().astype(np.int64),
                        np.full((C, M), -1), l0, np.zeros(C, dtype=np.int64), N, temperature, pm,
                        seed, step0)
    o1 = isd.isd_accept(l1, b["qo1"].numpy(), o0["next_mode"], o0["next_drafts"], l0,
                        o0["next_mask_row0"], N, temperature, pm, seed, step0 + 1)
    return o0, o1


def compare_accept(g, o, N, greedy=False):
    """Assert GPU step outputs against the oracle's; returns counters."""
    C = o["n_accepted"].shape[0]
    M = N - 1
    stats = dict(compared=0, ambiguous_accept=0, ambiguous_token=0)
    assert g["status"] == 0, f"device status {g['status']}"
    n_acc = g["n_accepted"].cpu().numpy()
    toks = g["out_tokens"].cpu().numpy()
    nd = g["next_drafts"].cpu().numpy()
    dbg = g["dbg"].cpu().numpy()
    rs = g["row_stats"].cpu().numpy()
    # row statistics: max exact up to the fp32 round trip, sums within 1e-5
    np.testing.assert_allclose(rs[:, 0], o["row_max"], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(rs[:, 1], o["row_sum"], rtol=PROB_RTOL)
    nq = g["next_q_stats"].cpu().numpy()
    for c in range(C):
        mrow = o["next_mask_row0"][c] + np.arange(M)
        np.testing.assert_allclose(nq[c, :, 0], o["row_max"][mrow], rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(nq[c, :, 1], o["row_sum"][mrow], rtol=PROB_RTOL)
        ambiguous = False
        if o["final_kind"][c] != isd.END_FRESH:
            # uniforms bit-exact, draft probabilities within 1e-5
            assert np.array_equal(dbg[c, :, 0], o["u"][c].astype(np.float32)), "Philox uniforms"
            np.testing.assert_allclose(dbg[c, :, 1], o["p_draft"][c], rtol=PROB_RTOL, atol=1e-30)
            np.testing.assert_allclose(dbg[c, :, 2], o["q_draft"][c], rtol=PROB_RTOL, atol=1e-30)
            # decisions in order up to the first rejection
            for i in range(min(M, int(o["n_accepted"][c]) + 1)):
                if abs(o["u"][c, i] - min(1.0, o["ratio"][c, i])) <= AMBIG:
                    ambiguous = True
                    break
        if ambiguous:
            stats["ambiguous_accept"] += 1
            continue
        assert n_acc[c] == o["n_accepted"][c], f"request {c}: n_accepted"
        k = int(n_acc[c])
        assert np.array_equal(toks[c, :k], o["out_tokens"][c, :k])
        if o["final_margin"][c] <= AMBIG and not greedy:
            stats["ambiguous_token"] += 1
        else:
            assert toks[c, k] == o["out_tokens"][c, k], (
                f"request {c}: final token {toks[c, k]} vs {o['out_tokens'][c, k]} "
                f"(kind {o['final_kind'][c]})")
        assert np.all(toks[c, k + 1:] == -1)
        assert g["n_out"][c].item() == o["n_out"][c]
        assert g["n_commit"][c].item() == o["n_commit"][c]
        assert g["next_mode"][c].item() == o["next_mode"][c]
        assert g["next_mask_row0"][c].item() == o["next_mask_row0"][c]
        assert np.array_equal(nd[c], o["next_drafts"][c]), f"request {c}: proposals"
        stats["compared"] += 1
    return stats
