"""Pins of the oracle's paged strict-causal GQA attention (CPU only).

Independent checks: torch's scaled_dot_product_attention in float64 on the
contiguous sequence (a library routine), closed forms (one visible key; all
keys equal), and the invariants of paging and strict causality.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle.isd import isd_attention


def _case(C=3, Hq=8, Hkv=2, D=32, P=4, lens=(0, 5, 13), rows=(3, 2, 4), seed=0):
    rng = np.random.default_rng(seed)
    qo = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    T = int(qo[-1])
    need = [(L + P - 1) // P + 1 for L in lens]
    pool = sum(need) + 3
    perm = rng.permutation(pool)
    table = np.full((C, max(need)), -1, dtype=np.int64)
    at = 0
    for c, n in enumerate(need):
        table[c, :n] = perm[at:at + n]
        at += n
    return dict(
        q=rng.standard_normal((T, Hq, D)), k_new=rng.standard_normal((T, Hkv, D)),
        v_new=rng.standard_normal((T, Hkv, D)),
        k_cache=rng.standard_normal((pool, Hkv, P, D)),
        v_cache=rng.standard_normal((pool, Hkv, P, D)),
        page_table=table, seq_lens=np.array(lens), qo_indptr=qo, page_size=P,
        sm_scale=1.0 / np.sqrt(D))


def _run(case):
    return isd_attention(case["q"], case["k_new"], case["v_new"], case["k_cache"],
                         case["v_cache"], case["page_table"], case["seq_lens"],
                         case["qo_indptr"], case["page_size"], case["sm_scale"])


def _contiguous(cache, table_row, L, P):
    # written out slot by slot, independently of the oracle's gather
    out = np.zeros((L,) + cache.shape[1:2] + cache.shape[3:])
    for s in range(L):
        out[s] = cache[table_row[s // P], :, s % P, :]
    return out


def test_matches_torch_sdpa_float64():
    case = _case()
    got = _run(case)
    Hq, Hkv = case["q"].shape[1], case["k_new"].shape[1]
    for c in range(len(case["seq_lens"])):
        L = int(case["seq_lens"][c])
        t0, t1 = case["qo_indptr"][c], case["qo_indptr"][c + 1]
        R = t1 - t0
        k = np.concatenate([_contiguous(case["k_cache"], case["page_table"][c], L, case["page_size"]),
                            case["k_new"][t0:t1]])
        v = np.concatenate([_contiguous(case["v_cache"], case["page_table"][c], L, case["page_size"]),
                            case["v_new"][t0:t1]])
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        qt = torch.from_numpy(case["q"][t0:t1]).permute(1, 0, 2)
        mask = torch.tensor([[s <= L + r for s in range(L + R)] for r in range(R)])
        ref = F.scaled_dot_product_attention(qt[None], kt[None], vt[None],
                                             attn_mask=mask, scale=case["sm_scale"])[0]
        np.testing.assert_allclose(got[t0:t1], ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


def test_page_shuffle_invariance():
    case = _case(seed=1)
    base = _run(case)
    rng = np.random.default_rng(7)
    pool = case["k_cache"].shape[0]
    perm = rng.permutation(pool)          # physical page p moves to perm[p]
    kc = np.empty_like(case["k_cache"])
    vc = np.empty_like(case["v_cache"])
    kc[perm] = case["k_cache"]
    vc[perm] = case["v_cache"]
    table = np.where(case["page_table"] >= 0, perm[case["page_table"]], -1)
    moved = dict(case, k_cache=kc, v_cache=vc, page_table=table)
    assert np.array_equal(_run(moved), base)


def test_strict_causality_perturbation():
    case = _case(seed=2, lens=(6, 9, 1), rows=(4, 4, 4))
    base = _run(case)
    P = case["page_size"]
    pert = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in case.items()}
    for c in range(3):
        L = int(case["seq_lens"][c])
        # cache slots >= L in the last partial page and the next page
        for s in range(L, L + P):
            page = case["page_table"][c][s // P]
            pert["k_cache"][page, :, s % P, :] += 100.0
            pert["v_cache"][page, :, s % P, :] -= 50.0
    got = _run(pert)
    assert np.array_equal(got, base)
    # a later new row does not reach an earlier one
    for r_changed in range(1, 4):
        p2 = dict(case, k_new=case["k_new"].copy(), v_new=case["v_new"].copy())
        t = case["qo_indptr"][1] + r_changed
        p2["k_new"][t] += 3.0
        p2["v_new"][t] += 3.0
        out = _run(p2)
        t0 = case["qo_indptr"][1]
        assert np.array_equal(out[t0:t], base[t0:t])
        assert not np.allclose(out[t], base[t])
    # and a committed slot does change the outputs
    p3 = dict(case, v_cache=case["v_cache"].copy())
    p3["v_cache"][case["page_table"][0][0], :, 0, :] += 1.0
    assert not np.allclose(_run(p3)[0:4], base[0:4])


def test_single_visible_key_returns_its_value():
    case = _case(seed=3, lens=(0, 0, 0), rows=(1, 1, 1))
    out = _run(case)
    group = case["q"].shape[1] // case["k_new"].shape[1]
    for t in range(3):
        for h in range(case["q"].shape[1]):
            assert np.array_equal(out[t, h], case["v_new"][t, h // group])


def test_identical_keys_average_the_values():
    case = _case(seed=4, lens=(7, 3, 10), rows=(2, 3, 1))
    case["k_cache"][:] = 0.5
    case["k_new"][:] = 0.5
    out = _run(case)
    Hkv = case["k_new"].shape[1]
    group = case["q"].shape[1] // Hkv
    for c in range(3):
        L = int(case["seq_lens"][c])
        t0 = case["qo_indptr"][c]
        vc = _contiguous(case["v_cache"], case["page_table"][c], L, case["page_size"])
        for r in range(case["qo_indptr"][c + 1] - t0):
            vals = np.concatenate([vc, case["v_new"][t0:t0 + r + 1]])
            for h in range(case["q"].shape[1]):
                np.testing.assert_allclose(out[t0 + r, h], vals[:, h // group].mean(0), rtol=1e-12, atol=1e-13)
