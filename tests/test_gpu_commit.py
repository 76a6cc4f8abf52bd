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
