"""GPU parity of idlm_isd_attention against the oracle (marked gpu)."""
import math

import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from _gpu import assert_attention_close, gpu_attention, oracle_attention
from speculative_verify_accept_step_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _custom(C, N, lens, Hq=32, Hkv=8, D=128, P=16, dtype=torch.bfloat16, seed=0, fresh=()):
    """Small attention case with chosen context lengths (ragged tails)."""
    g = torch.Generator().manual_seed(seed)
    rows = [N if c in fresh else 2 * N - 1 for c in range(C)]
    qo = torch.zeros(C + 1, dtype=torch.int32)
    qo[1:] = torch.cumsum(torch.tensor(rows), 0).to(torch.int32)
    T = int(qo[-1])
    need = [(L + N + P - 1) // P for L in lens]
    pool = sum(need) + 5
    perm = torch.randperm(pool, generator=g)
    table = torch.full((C, max(need)), -1, dtype=torch.int32)
    at = 0
    for c, n in enumerate(need):
        table[c, :n] = perm[at:at + n].to(torch.int32)
        at += n
    return dict(q=torch.randn(T, Hq, D, generator=g).to(dtype),
                k_new=torch.randn(T, Hkv, D, generator=g).to(dtype),
                v_new=torch.randn(T, Hkv, D, generator=g).to(dtype),
                k_cache=torch.randn(pool, Hkv, P, D, generator=g).to(dtype),
                v_cache=torch.randn(pool, Hkv, P, D, generator=g).to(dtype),
                page_table=table, seq_lens=torch.tensor(lens, dtype=torch.int32), qo_indptr=qo,
                num_pages=pool, sm_scale=1.0 / math.sqrt(D)), max(rows)


def test_tiny_fp32_workload(cuda_device):
    w = wl.WORKLOADS["isd_tiny_c1_n2_f32"]
    a = wl.attention_inputs(w)
    out, st = gpu_attention(a, w.rows_full)
    assert st == 0
    assert_attention_close(out, oracle_attention(a), bf16=False)


def test_small_bf16_workload(cuda_device):
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    a = wl.attention_inputs(w)
    out, st = gpu_attention(a, w.rows_full)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


@pytest.mark.parametrize("N", [2, 4, 6, 8])
def test_ragged_tails_and_row_packings(cuda_device, N):
    # G * (2N-1) = 12, 28, 44, 60 packed rows: one to four m-tiles
    lens = [0, 1, 15, 16, 17, 100, 257, 33]
    a, R = _custom(len(lens), N, lens, seed=N)
    out, st = gpu_attention(a, R)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


@pytest.mark.parametrize("Hq,N", [(8, 9), (8, 16), (8, 20), (16, 9), (16, 16), (24, 11)])
def test_more_than_16_rows_per_request(cuda_device, Hq, N):
    # G = Hq / 8 query heads per kv head; R = 2N - 1 = 17 .. 39 rows per
    # request, so a unit's new keys span two or three 16-row blocks
    lens = [0, 1, 15, 16, 40, 257]
    a, R = _custom(len(lens), N, lens, Hq=Hq, Hkv=8, seed=20 + N, fresh=(2,))
    assert (Hq // 8) * R <= 64 and R > 16
    out, st = gpu_attention(a, R)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


@pytest.mark.parametrize("N", [2, 4, 8])
def test_many_short_units_per_cta(cuda_device, N):
    """300 requests with contexts of 0-160 tokens: every CTA of the grid walks
    several short units, so the consumers' pairs of blocks meet unit
    boundaries at both parities (a pair never spans two units: the block
    before a boundary goes alone) and segments start on odd blocks; one to
    four m-tiles (G (2N - 1) = 12, 28, 60 rows).  Every output is compared."""
    rng = np.random.default_rng(N)
    lens = [int(v) for v in rng.integers(0, 161, 300)]
    a, R = _custom(len(lens), N, lens, seed=40 + N, fresh=tuple(range(0, 300, 7)))
    out, st = gpu_attention(a, R)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


def test_mixed_fresh_and_full_rows(cuda_device):
    lens = [40, 0, 300, 16]
    a, R = _custom(4, 4, lens, seed=11, fresh=(1, 2))
    out, st = gpu_attention(a, R)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


def test_general_path_bf16_other_page_size(cuda_device):
    a, R = _custom(3, 3, [5, 40, 0], Hq=8, Hkv=2, D=64, P=8, seed=3)
    out, st = gpu_attention(a, R)
    assert st == 0
    assert_attention_close(out, oracle_attention(a))


def test_headline_workload_full_size(cuda_device):
    w = wl.WORKLOADS["isd_c64_n4_ctx4096"]
    a = wl.attention_inputs(w)
    out, st = gpu_attention(a, w.rows_full)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    # every request: at this size every unit is cut by the balanced split, so
    # this also checks the merge of partial results everywhere
    assert_attention_close(out, oracle_attention(a))


def test_ragged_workload_sampled_requests(cuda_device):
    w = wl.WORKLOADS["isd_c64_n4_ctx1k_32k"]
    a = wl.attention_inputs(w)
    out, st = gpu_attention(a, w.rows_full)
    assert st == 0
    assert torch.isfinite(out.float()).all()
    L = a["seq_lens"].numpy()
    pick = sorted({int(np.argmin(L)), int(np.argmax(L))} | set(range(0, 64, 5)))
    assert_attention_close(out, oracle_attention(a, requests=pick))


def test_page_permutation_gives_identical_output(cuda_device):
    a, R = _custom(4, 4, [64, 200, 31, 500], seed=5)
    out1, _ = gpu_attention(a, R)
    perm = torch.randperm(a["k_cache"].shape[0], generator=torch.Generator().manual_seed(1))
    kc = torch.empty_like(a["k_cache"])
    vc = torch.empty_like(a["v_cache"])
    kc[perm] = a["k_cache"]
    vc[perm] = a["v_cache"]
    t = a["page_table"].long()
    table = torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32)
    out2, _ = gpu_attention(dict(a, k_cache=kc, v_cache=vc, page_table=table), R)
    assert torch.equal(out1, out2)


def test_bad_page_id_sets_status(cuda_device):
    a, R = _custom(2, 4, [40, 40], seed=7)
    a["page_table"][1, 1] = 10_000
    _, st = gpu_attention(a, R)
    assert st == 1


def test_graph_replays_merge_split_units(cuda_device):
    """A CUDA graph replays the call's two launches (the pass over the pages
    and the programmatic-dependent merge of units the balanced split cut)
    with their parameters frozen: every replay must write the eager call's
    output bit for bit, the cut units' rows (which only the merge writes)
    included."""
    w = wl.WORKLOADS["isd_c64_n4_ctx4096"]
    a = wl.attention_inputs(w)
    eager, st = gpu_attention(a, w.rows_full)
    assert st == 0
    dev = "cuda"
    q = a["q"].to(dev)
    T, Hq, D = q.shape
    num_pages, Hkv, P, _ = a["k_cache"].shape
    C = a["page_table"].shape[0]
    dv = {k: a[k].to(dev) for k in ("k_new", "v_new", "k_cache", "v_cache", "page_table",
                                    "seq_lens", "qo_indptr")}
    ws = torch.empty(lib.idlm_isd_attention_workspace_size(C, Hq, Hkv, D, P, w.rows_full,
                                                           lib.IDLM_BF16),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            lib.idlm_isd_attention(q, dv["k_new"], dv["v_new"], dv["k_cache"], dv["v_cache"],
                                   dv["page_table"], dv["seq_lens"], dv["qo_indptr"], out, ws,
                                   st, max_rows=w.rows_full, sm_scale=a["sm_scale"])
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out, eager)
