"""idlm_isd_accept_noalloc against idlm_isd_accept (marked gpu).

Some callers of this library cannot allocate device memory: a plugin whose
host process owns all GPU memory and hands out no scratch space, or a decode
loop that runs under a fixed memory budget and may not call the allocator.
idlm_isd_accept_noalloc serves them: it takes no workspace and uses a 4 MiB
scratch array compiled into the library instead.  This file checks that it
returns the same results as the workspace entry point on two calls in a row
(a FRESH step, then the FULL step that verifies its proposals), and that it
refuses a batch whose scratch would not fit.  It is named to run last.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_verify_accept_step_b300 as lib
from speculative_verify_accept_step_b300 import _lib

pytestmark = pytest.mark.gpu

RTOL = 1e-5   # the probability tolerance of the parity tests


def _outputs(C, N, T, dev):
    M = N - 1
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(n_accepted=torch.full((C,), -7, **i32), out_tokens=torch.full((C, N), -7, **i32),
                n_out=torch.full((C,), -7, **i32), n_commit=torch.full((C,), -7, **i32),
                next_drafts=torch.full((C, M), -7, **i32),
                next_q_stats=torch.zeros((C, M, 2), dtype=torch.float32, device=dev),
                next_mode=torch.zeros((C,), dtype=torch.uint8, device=dev),
                next_mask_row0=torch.full((C,), -7, **i32),
                row_stats=torch.zeros((T, 2), dtype=torch.float32, device=dev),
                dbg=torch.zeros((C, M, 4), dtype=torch.float32, device=dev))


def _call(noalloc, logits, qo, mode, drafts, dq, prev, prow, N, step, dev):
    T, V = logits.shape
    C = mode.shape[0]
    o = _outputs(C, N, T, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    common = (logits, qo, mode, drafts, dq, prev, prow, N, 1.0, lib.PROPOSE_ARGMAX, 7, step,
              o["n_accepted"], o["out_tokens"], o["n_out"], o["n_commit"], o["next_drafts"],
              o["next_q_stats"], o["next_mode"], o["next_mask_row0"])
    if noalloc:
        lib.idlm_isd_accept_noalloc(*common, st, row_stats=o["row_stats"], dbg=o["dbg"])
    else:
        ws = torch.empty(lib.idlm_isd_accept_workspace_size(C, T, N, V), dtype=torch.uint8,
                         device=dev)
        lib.idlm_isd_accept(*common, ws, st, row_stats=o["row_stats"], dbg=o["dbg"])
    torch.cuda.synchronize()
    o["status"] = int(st.item())
    return o


def _two_steps(noalloc, b, N, dev):
    C = b["mode0"].shape[0]
    M = N - 1
    l0, l1 = b["logits0"], b["logits1"]
    s0 = _call(noalloc, l0, b["qo0"], b["mode0"], torch.full((C, M), -1, dtype=torch.int32, device=dev),
               torch.zeros((C, M, 2), dtype=torch.float32, device=dev), l0,
               torch.zeros(C, dtype=torch.int32, device=dev), N, 1, dev)
    s1 = _call(noalloc, l1, b["qo1"], s0["next_mode"], s0["next_drafts"], s0["next_q_stats"], l0,
               s0["next_mask_row0"], N, 2, dev)
    return s0, s1


def _batch(C, N, V, dev, seed=0):
    g = torch.Generator().manual_seed(seed)
    l1 = torch.randn(C * (2 * N - 1), V, generator=g) * 3
    l0 = torch.empty(C * N, V)
    for c in range(C):
        l0[c * N] = torch.randn(V, generator=g) * 3
        for k in range(1, N):
            l0[c * N + k] = l1[c * (2 * N - 1) + k - 1] + 0.3 * torch.randn(V, generator=g)
    return dict(logits0=l0.bfloat16().to(dev), logits1=l1.bfloat16().to(dev),
                qo0=torch.arange(0, C * N + 1, N, dtype=torch.int32, device=dev),
                qo1=torch.arange(0, C * (2 * N - 1) + 1, 2 * N - 1, dtype=torch.int32, device=dev),
                mode0=torch.zeros(C, dtype=torch.uint8, device=dev))


def _same(a, b):
    assert a["status"] == 0 and b["status"] == 0
    for k in ("n_accepted", "out_tokens", "n_out", "n_commit", "next_drafts", "next_mode",
              "next_mask_row0"):
        assert torch.equal(a[k], b[k]), k
    for k in ("next_q_stats", "row_stats", "dbg"):
        np.testing.assert_allclose(a[k].cpu().numpy(), b[k].cpu().numpy(), rtol=RTOL, atol=0)


@pytest.mark.parametrize("C,N,V", [(64, 4, 151936), (16, 3, 8192)])
def test_noalloc_matches_workspace_entry_point(cuda_device, C, N, V):
    b = _batch(C, N, V, cuda_device)
    w0, w1 = _two_steps(False, b, N, cuda_device)
    n0, n1 = _two_steps(True, b, N, cuda_device)
    _same(w0, n0)
    _same(w1, n1)
    # and once more: the shared scratch keeps the previous call's contents
    m0, m1 = _two_steps(True, b, N, cuda_device)
    _same(w0, m0)
    _same(w1, m1)


def test_noalloc_refuses_scratch_beyond_its_array(cuda_device):
    dummy = ctypes.c_void_p(256)      # never dereferenced: the size check comes first
    C, T, N, V = 4096, 4096 * 7, 4, 151936
    assert lib.idlm_isd_accept_workspace_size(C, T, N, V) > (4 << 20)
    args = ([dummy, lib.IDLM_BF16, V] + [dummy] * 5 + [T, dummy] +
            [C, T, N, 1.0, 0, 0, 0] + [dummy] * 10 + [dummy, None])
    assert _lib.lib().idlm_isd_accept_noalloc(*args) == 3   # IDLM_ERR_WORKSPACE
