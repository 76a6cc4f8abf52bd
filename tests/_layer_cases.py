"""A small decoder-layer case (torch CPU tensors) shared by the GPU layer
parity test and the CPU pin of its tolerance."""
import torch


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
