"""GPU parity of idlm_kv_commit against the oracle: bit-exact (marked gpu)."""
import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from oracle.isd import kv_commit
from speculative_verify_accept_step_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run(a, n_commit, dev="cuda", same_buffer=False):
    kc, vc = a["k_cache"].to(dev), a["v_cache"].to(dev)
    sl_in = a["seq_lens"].to(dev)
    sl_out = sl_in if same_buffer else torch.full_like(sl_in, -1)
    rel = torch.full_like(sl_in, -1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.idlm_kv_commit(kc, vc, a["page_table"].to(dev), sl_in, sl_out, a["k_new"].to(dev),
                       a["v_new"].to(dev), a["qo_indptr"].to(dev),
                       n_commit.to(dev).to(torch.int32), st, releasable_from=rel)
    torch.cuda.synchronize()
    return kc.cpu(), vc.cpu(), sl_out.cpu(), rel.cpu(), int(st.item())


def _oracle(a, n_commit):
    as_np = lambda t: t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()
    kc, vc, sl, rel = kv_commit(as_np(a["k_cache"]), as_np(a["v_cache"]), a["page_table"].numpy(),
                                a["seq_lens"].numpy(), as_np(a["k_new"]), as_np(a["v_new"]),
                                a["qo_indptr"].numpy(), n_commit.numpy(), a["k_cache"].shape[2])
    return kc, vc, sl, rel


@pytest.mark.parametrize("name", ["isd_tiny_c1_n2_f32", "isd_c4_n4_ctx512_2048",
                                  "isd_c64_n4_ctx4096", "isd_c64_n4_ctx1k_32k"])
def test_commit_bit_exact(cuda_device, name):
    w = wl.WORKLOADS[name]
    a = wl.attention_inputs(w)
    g = torch.Generator().manual_seed(3)
    n_commit = torch.randint(0, w.N + 1, (w.C,), generator=g)
    kc, vc, sl, rel, st = _run(a, n_commit)
    assert st == 0
    okc, ovc, osl, orel = _oracle(a, n_commit)
    view = (lambda t: t.view(torch.int16).numpy()) if kc.dtype == torch.bfloat16 else (lambda t: t.numpy())
    assert np.array_equal(view(kc), okc)
    assert np.array_equal(view(vc), ovc)
    assert np.array_equal(sl.numpy(), osl)
    assert np.array_equal(rel.numpy(), orel)


def test_commit_in_place_lengths(cuda_device):
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    a = wl.attention_inputs(w)
    n_commit = torch.tensor([1, 4, 2, 3])
    kc, vc, sl, rel, st = _run(a, n_commit, same_buffer=True)
    assert st == 0
    assert torch.equal(sl, a["seq_lens"] + n_commit.to(torch.int32))


def test_commit_errors_write_nothing(cuda_device):
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    a = wl.attention_inputs(w)
    L1 = int(a["seq_lens"][1])
    a["page_table"][1, L1 // 16] = 999_999          # the slot L1 lands on a bad page
    n_commit = torch.tensor([2, 2, 2, 2])
    kc, vc, sl, rel, st = _run(a, n_commit)
    assert st == 1
    assert sl[1].item() == -1                       # request 1 untouched
    okc, _, osl, _ = _oracle(dict(a, page_table=a["page_table"]), torch.tensor([2, 0, 2, 2]))
    assert np.array_equal(kc.view(torch.int16).numpy(), okc)
    assert sl[0].item() == osl[0] and sl[2].item() == osl[2]


@pytest.mark.parametrize("name", ["isd_c4_n4_ctx512_2048", "isd_c64_n4_ctx4096"])
def test_fused_accept_commit_equals_accept_then_commit(cuda_device, name):
    """idlm_isd_accept_commit (the commits as work items of the accept's
    residual kernel) writes the same accept outputs, cache, lengths and
    releasable pages, bit for bit, as idlm_isd_accept followed by
    idlm_kv_commit on the same inputs (whose commit is oracle-checked above)."""
    from _gpu import alloc_accept, gpu_accept
    from oracle import isd
    dev = "cuda"
    w = wl.WORKLOADS[name]
    a = wl.attention_inputs(w)
    b = wl.accept_inputs(w)
    C, N = w.C, w.N
    qo1 = b["qo1"].to(dev)
    assert torch.equal(a["qo_indptr"], b["qo1"])
    l0, l1 = b["logits0"].to(dev), b["logits1"].to(dev)
    M = N - 1
    s0 = gpu_accept(l0, b["qo0"].to(dev), b["mode0"].to(dev),
                    torch.full((C, M), -1, dtype=torch.int32, device=dev),
                    torch.zeros((C, M, 2), dtype=torch.float32, device=dev), l0,
                    torch.zeros(C, dtype=torch.int32, device=dev), N, 1.0, isd.PROPOSE_ARGMAX, 0, 0)
    args = (qo1, s0["next_mode"], s0["next_drafts"], s0["next_q_stats"], l0, s0["next_mask_row0"],
            N, 1.0, isd.PROPOSE_ARGMAX, 0, 1)
    ref = gpu_accept(l1, *args)
    kc_ref, vc_ref, sl_ref, rel_ref, st_ref = _run(a, ref["n_commit"].cpu())
    assert st_ref == 0
    T, V = l1.shape
    o = alloc_accept(C, N, T, dev)
    ws = torch.empty(lib.idlm_isd_accept_workspace_size(C, T, N, V), dtype=torch.uint8, device=dev)
    kc, vc = a["k_cache"].to(dev), a["v_cache"].to(dev)
    sl_in = a["seq_lens"].to(dev)
    sl_out = torch.full_like(sl_in, -1)
    rel = torch.full_like(sl_in, -1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    lib.idlm_isd_accept_commit(l1, *args, o["n_accepted"], o["out_tokens"], o["n_out"],
                               o["n_commit"], o["next_drafts"], o["next_q_stats"], o["next_mode"],
                               o["next_mask_row0"], kc, vc, a["page_table"].to(dev), sl_in, sl_out,
                               a["k_new"].to(dev), a["v_new"].to(dev), ws, st,
                               row_stats=o["row_stats"], dbg=o["dbg"], releasable_from=rel)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in ("n_accepted", "out_tokens", "n_out", "n_commit", "next_drafts", "next_q_stats",
              "next_mode", "next_mask_row0", "row_stats"):
        assert torch.equal(o[k], ref[k]), k
    assert torch.equal(kc.cpu(), kc_ref) and torch.equal(vc.cpu(), vc_ref)
    assert torch.equal(sl_out.cpu(), sl_ref) and torch.equal(rel.cpu(), rel_ref)


def _fused_call(a, b_logits, qo, mode, drafts, dq, prev, prow, N, step, page_table=None,
                dev="cuda"):
    from _gpu import alloc_accept
    from oracle import isd
    C = mode.shape[0]
    T, V = b_logits.shape
    o = alloc_accept(C, N, T, dev)
    ws = torch.empty(lib.idlm_isd_accept_workspace_size(C, T, N, V), dtype=torch.uint8, device=dev)
    kc, vc = a["k_cache"].to(dev), a["v_cache"].to(dev)
    sl_in = a["seq_lens"].to(dev)
    sl_out = torch.full_like(sl_in, -1)
    rel = torch.full_like(sl_in, -1)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pt = (a["page_table"] if page_table is None else page_table).to(dev)
    lib.idlm_isd_accept_commit(b_logits, qo, mode, drafts, dq, prev, prow, N, 1.0,
                               isd.PROPOSE_ARGMAX, 0, step, o["n_accepted"], o["out_tokens"],
                               o["n_out"], o["n_commit"], o["next_drafts"], o["next_q_stats"],
                               o["next_mode"], o["next_mask_row0"], kc, vc, pt, sl_in, sl_out,
                               a["k_new"].to(dev), a["v_new"].to(dev), ws, st,
                               row_stats=o["row_stats"], dbg=o["dbg"], releasable_from=rel)
    torch.cuda.synchronize()
    return o, kc.cpu(), vc.cpu(), sl_out.cpu(), rel.cpu(), int(st.item())


def test_fused_accept_commit_fresh_step(cuda_device):
    """A FRESH step through the fused call: every request commits its one
    clean row (n_commit = 1), bit for bit as idlm_kv_commit does."""
    from _gpu import gpu_accept
    from oracle import isd
    dev = "cuda"
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    b = wl.accept_inputs(w)
    C, N = w.C, w.N
    M = N - 1
    # a FRESH step's rows (N per request) with the cache inputs of the same shape
    a = wl.attention_inputs(w, mode=torch.zeros(C, dtype=torch.int64))
    assert torch.equal(a["qo_indptr"], b["qo0"])
    l0 = b["logits0"].to(dev)
    qo0 = b["qo0"].to(dev)
    args = (qo0, b["mode0"].to(dev), torch.full((C, M), -1, dtype=torch.int32, device=dev),
            torch.zeros((C, M, 2), dtype=torch.float32, device=dev), l0,
            torch.zeros(C, dtype=torch.int32, device=dev))
    ref = gpu_accept(l0, *args, N, 1.0, isd.PROPOSE_ARGMAX, 0, 0)
    assert torch.all(ref["n_commit"] == 1)
    kc_ref, vc_ref, sl_ref, rel_ref, st_ref = _run(a, ref["n_commit"].cpu())
    o, kc, vc, sl, rel, st = _fused_call(a, l0, *args, N, 0)
    assert st == 0 and st_ref == 0
    for k in ("n_accepted", "out_tokens", "n_commit", "next_drafts", "next_mode"):
        assert torch.equal(o[k], ref[k]), k
    assert torch.equal(kc, kc_ref) and torch.equal(vc, vc_ref)
    assert torch.equal(sl, sl_ref) and torch.equal(rel, rel_ref)


def test_fused_accept_commit_bad_page_writes_nothing_for_that_request(cuda_device):
    """A page id outside the pool on the slot a request would write: the
    fused call sets BAD_PAGE and leaves that request's cache rows and length
    untouched, while the other requests commit."""
    from oracle import isd
    dev = "cuda"
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    b = wl.accept_inputs(w)
    C, N = w.C, w.N
    M = N - 1
    a = wl.attention_inputs(w, mode=torch.zeros(C, dtype=torch.int64))
    L1 = int(a["seq_lens"][1])
    pt = a["page_table"].clone()
    pt[1, L1 // 16] = 999_999
    l0 = b["logits0"].to(dev)
    args = (b["qo0"].to(dev), b["mode0"].to(dev),
            torch.full((C, M), -1, dtype=torch.int32, device=dev),
            torch.zeros((C, M, 2), dtype=torch.float32, device=dev), l0,
            torch.zeros(C, dtype=torch.int32, device=dev))
    o, kc, vc, sl, rel, st = _fused_call(a, l0, *args, N, 0, page_table=pt)
    assert st == 1   # BAD_PAGE
    assert sl[1].item() == -1 and rel[1].item() == -1
    okc, _, osl, _ = _oracle(dict(a, page_table=pt), torch.tensor([1, 0, 1, 1]))
    assert np.array_equal(kc.view(torch.int16).numpy(), okc)
    assert sl[0].item() == osl[0] and sl[2].item() == osl[2] and sl[3].item() == osl[3]
