"""GPU parity of idlm_risd_layer (one R-ISD decoder layer) against the
oracle's layer (marked gpu).

The oracle stores every activation in bf16 where the library does (the
workload is a bf16 layer, the adapters' rank-r intermediates included),
computing each step in float64.  A layer chains eleven stored activations;
where the GPU's fp32 and the oracle's float64 land on either side of a bf16
rounding edge, an element differs by one ulp and the difference travels
through the later ops.  The tolerance is derived from that: flipping 1% of
every stored activation of the oracle by one ulp moves its outputs by up to
2.4 times the single-op bound 2e-2 + 1e-2 |x| (measured in
tests/test_oracle_layer.py, which also pins this), so each element must be
within 4 times that bound, and the mean error within a quarter of the
bound's mean (1% flips give 0.15 - 0.2).  Clean rows must equal the same layer without adapters (every B = 0)
bit for bit: causal attention keeps MASK rows out of clean rows ("Lossless
R-ISD").
"""
import math

import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from oracle import isd
from speculative_verify_accept_step_b300 import workloads as wl
from _layer_cases import small_case

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2       # the single-op bf16 bound
LAYER_FACTOR = 4.0              # chained bf16 activations (see the module docstring)


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


def assert_close(got, ref, factor=LAYER_FACTOR):
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    worst = float((err / bound).max())
    assert np.all(err <= factor * bound), f"worst err/bound {worst:.3f}"
    assert err.mean() <= 0.25 * bound.mean(), f"mean err {err.mean():.4g}"
    return worst


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
