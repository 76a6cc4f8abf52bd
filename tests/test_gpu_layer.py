"""GPU parity of idlm_risd_layer (one R-ISD decoder layer) against the
oracle's layer (marked gpu).

The oracle stores every activation in bf16 where the library does (the
workload is a bf16 layer), computing each step in float64; the comparison
uses the bf16 bound |gpu - oracle| <= 2e-2 + 1e-2 |oracle|.  Clean rows
must equal the same layer without adapters (every B = 0) bit for bit:
causal attention keeps MASK rows out of clean rows ("Lossless R-ISD").
"""
import math

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


def run_layer(inp, Hq, Hkv, D, H, F, rank, dev="cuda", eps=1e-6):
    W = {k: v.to(dev) for k, v in inp["W"].items()}
    lw = lib.layer_weights(W, H, F, Hq, Hkv, D, rank, inp["lora_scale"], eps)
    x = inp["x"].to(dev)
    M = x.shape[0]
    C = inp["page_table"].shape[0]
    max_rows = int((inp["qo_indptr"][1:] - inp["qo_indptr"][:-1]).max())
    ws = torch.empty(lib.idlm_risd_layer_workspace_size(lw, M, C, 16, max_rows), dtype=torch.uint8,
                     device=dev)
    out = torch.full_like(x, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    kn = torch.empty((M, Hkv, D), dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    lib.idlm_risd_layer(lw, x, out, inp["row_gate"].to(dev), inp["k_cache"].to(dev),
                        inp["v_cache"].to(dev), inp["page_table"].to(dev),
                        inp["seq_lens"].to(dev), inp["qo_indptr"].to(dev), max_rows, ws, st,
                        k_new_out=kn, v_new_out=vn)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return out, kn, vn


def oracle_layer(inp, Hq, Hkv, D, eps=1e-6):
    W = {k: f64(v) for k, v in inp["W"].items()}
    for k in ("a_qkv", "a_o", "a_gu", "a_down"):
        W.setdefault(k, np.zeros((0, 1)))
    for k in ("b_qkv", "b_o", "b_gu", "b_down"):
        W.setdefault(k, np.zeros((1, 0)))
    W.setdefault("norm1", None)
    W.setdefault("norm2", None)
    return isd.risd_layer(f64(inp["x"]), W, inp["row_gate"].numpy(), inp["lora_scale"], eps, Hq,
                          Hkv, D, f64(inp["k_cache"]), f64(inp["v_cache"]),
                          inp["page_table"].numpy(), inp["seq_lens"].numpy(),
                          inp["qo_indptr"].numpy(), 16, store=isd.round_bf16)


def assert_close(got, ref):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = float((err / bound).max())
    assert np.all(err <= bound), f"worst err/bound {worst:.3f}"
    return worst


def small_case(rank, seed, Hq=8, Hkv=2, D=64, H=512, F=1024, C=4, N=4):
    g = torch.Generator().manual_seed(seed)
    rows = 2 * N - 1
    nq, nkv = Hq * D, Hkv * D
    mk = lambda *s: (torch.randn(*s, generator=g) * 0.05).bfloat16()
    W = dict(w_qkv=mk(nq + 2 * nkv, H), w_o=mk(H, nq), w_gu=mk(2 * F, H), w_down=mk(H, F))
    if rank:
        W.update(a_qkv=mk(3 * rank, H), b_qkv=mk(nq + 2 * nkv, rank), a_o=mk(rank, nq),
                 b_o=mk(H, rank), a_gu=mk(2 * rank, H), b_gu=mk(2 * F, rank), a_down=mk(rank, F),
                 b_down=mk(H, rank))
    lens = [0, 17, 100, 260][:C]
    P = 16
    need = [(L + rows + P - 1) // P for L in lens]
    perm = torch.randperm(sum(need), generator=g)
    table = torch.full((C, max(need)), -1, dtype=torch.int32)
    at = 0
    for c, n in enumerate(need):
        table[c, :n] = perm[at:at + n].to(torch.int32)
        at += n
    T = C * rows
    return dict(W=W, x=torch.randn(T, H, generator=g).bfloat16(),
                row_gate=(torch.arange(T) % rows >= N).to(torch.uint8),
                k_cache=torch.randn(at, Hkv, P, D, generator=g).bfloat16(),
                v_cache=torch.randn(at, Hkv, P, D, generator=g).bfloat16(),
                page_table=table, seq_lens=torch.tensor(lens, dtype=torch.int32),
                qo_indptr=torch.arange(0, T + 1, rows, dtype=torch.int32), lora_scale=1.0)


@pytest.mark.parametrize("rank", [0, 16, 128])
def test_small_layer_matches_the_oracle(cuda_device, rank):
    inp = small_case(rank, seed=rank + 1)
    out, kn, vn = run_layer(inp, 8, 2, 64, 512, 1024, rank)
    ref, rk, rv = oracle_layer(inp, 8, 2, 64)
    assert_close(f64(out), ref)
    assert_close(f64(kn), rk)
    assert_close(f64(vn), rv)


def test_clean_rows_bit_identical_without_the_adapters(cuda_device):
    inp = small_case(128, seed=7)
    out, _, _ = run_layer(inp, 8, 2, 64, 512, 1024, 128)
    zero_b = dict(inp, W={k: (torch.zeros_like(v) if k.startswith("b_") else v)
                          for k, v in inp["W"].items()})
    base, _, _ = run_layer(zero_b, 8, 2, 64, 512, 1024, 128)
    clean = (inp["row_gate"] == 0).cuda()
    assert torch.equal(out[clean], base[clean])
    assert not torch.equal(out[~clean], base[~clean])


@pytest.mark.parametrize("rank", [16, 128])
def test_full_size_layer_on_sampled_requests(cuda_device, rank):
    """The gated-LoRA workload's layer (hidden 4096, FFN 12288, 32/8 heads of
    128, 4096-token contexts), on 4 of its 64 requests (28 rows): every op
    but attention is row-wise, and attention stays inside a request."""
    w = wl.WORKLOADS["lora_layer_m448"]
    inp = wl.layer_inputs(w, rank=rank, requests=[0, 21, 42, 63])
    out, _, _ = run_layer(inp, w.Hq, w.Hkv, w.D, w.hidden, w.ffn, rank)
    ref, _, _ = oracle_layer(inp, w.Hq, w.Hkv, w.D)
    assert_close(f64(out), ref)
