"""Pins of the oracle's KV commit / rollback (CPU only): brute force on small
paged caches, written slot by slot in the test."""
import numpy as np
import pytest

from oracle.isd import kv_commit


def _case(seed=0, lens=(0, 3, 16, 30), rows=(7, 4, 7, 7), P=16, Hkv=2, D=8, slack=4):
    rng = np.random.default_rng(seed)
    C = len(lens)
    need = [(L + slack + P - 1) // P for L in lens]
    pool = sum(need) + 2
    perm = rng.permutation(pool)
    table = np.full((C, max(need)), -1, dtype=np.int64)
    at = 0
    for c, n in enumerate(need):
        table[c, :n] = perm[at:at + n]
        at += n
    qo = np.concatenate([[0], np.cumsum(rows)])
    T = int(qo[-1])
    return dict(k_cache=rng.standard_normal((pool, Hkv, P, D)),
                v_cache=rng.standard_normal((pool, Hkv, P, D)),
                page_table=table, seq_lens=np.array(lens),
                k_new=rng.standard_normal((T, Hkv, D)), v_new=rng.standard_normal((T, Hkv, D)),
                qo_indptr=qo, page_size=P)


def _seq(cache, table_row, L, P):
    return np.stack([cache[table_row[s // P], :, s % P, :] for s in range(L)]) if L else None


def test_commit_appends_rows_and_nothing_else():
    case = _case()
    n_commit = np.array([1, 4, 2, 3])
    kc, vc, seq, rel = kv_commit(case["k_cache"], case["v_cache"], case["page_table"],
                                 case["seq_lens"], case["k_new"], case["v_new"],
                                 case["qo_indptr"], n_commit, case["page_size"])
    P = case["page_size"]
    touched = set()
    for c, L in enumerate(case["seq_lens"]):
        n = n_commit[c]
        assert seq[c] == L + n
        # releasable_from: one past the last page-table entry that holds a
        # committed slot, counted slot by slot (no page holds one: 0)
        holding = {s // P for s in range(L + n)}
        assert rel[c] == (max(holding) + 1 if holding else 0)
        assert all(j in holding for j in range(rel[c]))
        t0 = case["qo_indptr"][c]
        if L:
            assert np.array_equal(_seq(kc, case["page_table"][c], L, P),
                                  _seq(case["k_cache"], case["page_table"][c], L, P))
        for j in range(n):
            s = L + j
            page = case["page_table"][c][s // P]
            touched.add((page, s % P))
            assert np.array_equal(kc[page, :, s % P], case["k_new"][t0 + j])
            assert np.array_equal(vc[page, :, s % P], case["v_new"][t0 + j])
    # every other slot of the pool is bit-unchanged
    for page in range(kc.shape[0]):
        for off in range(P):
            if (page, off) not in touched:
                assert np.array_equal(kc[page, :, off], case["k_cache"][page, :, off])
                assert np.array_equal(vc[page, :, off], case["v_cache"][page, :, off])


@pytest.mark.parametrize("lens", [(0, 15, 16, 17), (31, 32, 33, 1)])
def test_releasable_pages_counted_slot_by_slot(lens):
    """Every page-table entry before releasable_from holds a committed slot,
    none from it on: checked against the slots' own page indices."""
    case = _case(seed=3, lens=lens)
    P = case["page_size"]
    for n_commit in ([0, 0, 0, 0], [1, 1, 1, 1], [4, 4, 7, 7]):
        n_commit = np.minimum(np.array(n_commit), np.diff(case["qo_indptr"]))
        _, _, seq, rel = kv_commit(case["k_cache"], case["v_cache"], case["page_table"],
                                   case["seq_lens"], case["k_new"], case["v_new"],
                                   case["qo_indptr"], n_commit, P)
        for c in range(len(lens)):
            used = np.zeros(case["page_table"].shape[1], dtype=bool)
            for s in range(int(seq[c])):
                used[s // P] = True
            free = np.nonzero(~used)[0]
            first_free = int(free[0]) if free.size else used.size
            assert rel[c] == first_free
            assert not used[first_free:].any()


def test_zero_commit_keeps_everything():
    case = _case(seed=1)
    kc, vc, seq, rel = kv_commit(case["k_cache"], case["v_cache"], case["page_table"],
                                 case["seq_lens"], case["k_new"], case["v_new"],
                                 case["qo_indptr"], np.zeros(4, dtype=int), case["page_size"])
    assert np.array_equal(kc, case["k_cache"]) and np.array_equal(vc, case["v_cache"])
    assert np.array_equal(seq, case["seq_lens"])


@pytest.mark.parametrize("bad", ["page", "slot", "rows"])
def test_invalid_commit_raises(bad):
    case = _case(seed=2)
    n = np.array([1, 1, 1, 1])
    table = case["page_table"].copy()
    if bad == "page":
        table[1, 0] = 10_000
    elif bad == "slot":
        n = np.array([1, 1, 1, 7])
        table = table[:, :2]          # request 3 needs a third page
    else:
        n = np.array([8, 1, 1, 1])    # more than its 7 rows
    with pytest.raises(ValueError):
        kv_commit(case["k_cache"], case["v_cache"], table, case["seq_lens"],
                  case["k_new"], case["v_new"], case["qo_indptr"], n, case["page_size"])
