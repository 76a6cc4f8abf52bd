"""The seeded input generators: shapes, page tables and determinism (CPU)."""
import numpy as np
import torch

from oracle.isd import softmax_t
from speculative_verify_accept_step_b300 import workloads as wl


def test_tiny_shapes_and_pages():
    w = wl.WORKLOADS["isd_tiny_c1_n2_f32"]
    a = wl.attention_inputs(w)
    assert a["q"].shape == (3, 4, 64) and a["q"].dtype == torch.float32
    assert a["k_cache"].shape[1:] == (1, 16, 64)
    assert int(a["seq_lens"][0]) == 256
    used = a["page_table"][a["page_table"] >= 0]
    assert used.unique().numel() == used.numel()
    assert int(used.max()) < a["num_pages"]
    assert (256 + 2 + 15) // 16 == (a["page_table"][0] >= 0).sum()


def test_generators_are_deterministic():
    w = wl.WORKLOADS["isd_c4_n4_ctx512_2048"]
    a1, a2 = wl.attention_inputs(w, seed=3), wl.attention_inputs(w, seed=3)
    for k in ("q", "k_cache", "page_table", "seq_lens"):
        assert torch.equal(a1[k], a2[k])
    b1, b2 = wl.accept_inputs(w, seed=3), wl.accept_inputs(w, seed=3)
    assert torch.equal(b1["logits1"], b2["logits1"])
    assert b1["logits1"].shape == (4 * 7, 151936) and b1["logits1"].dtype == torch.bfloat16
    assert b1["logits0"].shape == (4 * 4, 151936)
    L = a1["seq_lens"]
    assert int(L.min()) >= 512 and int(L.max()) <= 2048


def test_fragmented_pool_has_holes():
    w = wl.WORKLOADS["isd_c64_n4_ctx1k_32k"]
    g = torch.Generator().manual_seed(0)
    L = wl.context_lengths(w, g)
    assert int(L.min()) >= 1024 and int(L.max()) <= 32768
    table, pool = wl.page_tables(w, L, g)
    used = table[table >= 0]
    assert used.numel() < pool and used.unique().numel() == used.numel()


def test_noise_table_meets_its_targets():
    # the stored sigma gives the target mean overlap sum(min(p, q)) on fresh rows
    table = wl.noise_table()
    g = torch.Generator().manual_seed(99)
    z = (torch.randn(4, 151936, generator=g) * 3.0).bfloat16().double().numpy()
    eps = torch.randn(4, 151936, generator=g).double().numpy()
    p = softmax_t(z, 1.0)
    for target, sigma in table.items():
        y = torch.from_numpy(z + sigma * eps).bfloat16().double().numpy()
        overlap = np.minimum(p, softmax_t(y, 1.0)).sum(-1).mean()
        assert abs(overlap - target) < 0.03


def test_fused_projections_are_exact():
    """fuse_projections (q|k|v, gate|up as one call): stacked weights give the
    separate base projections, and the block-diagonal adapter gives each block
    exactly its own adapter term (float64 on a few rows)."""
    w = wl.WORKLOADS["lora_layer_m448"]
    inp = wl.lora_inputs(w)
    x = inp["x"][:6].double()
    for names in (("q", "k", "v"), ("gate", "up")):
        f = wl.fuse_projections(inp["proj"], names)
        assert f["a"].shape[0] == sum(inp["proj"][n]["a"].shape[0] for n in names)
        fused = x @ f["w"].double().T + (x @ f["a"].double().T) @ f["b"].double().T
        sep = torch.cat([x @ inp["proj"][n]["w"].double().T
                         + (x @ inp["proj"][n]["a"].double().T) @ inp["proj"][n]["b"].double().T
                         for n in names], 1)
        assert torch.equal(fused, sep) or float((fused - sep).abs().max()) < 1e-12


# ------------------------------------------------- synthetic model for loops

def test_philox4x32_known_answers():
    """Philox4x32-10 against the generator authors' published known-answer
    vectors (Random123 distribution, kat_vectors: philox4x32 with 10 rounds)."""
    cases = [((0, 0, 0, 0), (0, 0), (0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8)),
             ((0xffffffff,) * 4, (0xffffffff,) * 2,
              (0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd)),
             ((0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344), (0xa4093822, 0x299f31d0),
              (0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1))]
    for ctr, key, want in cases:
        got = wl.philox4x32_10(ctr, key)
        assert tuple(int(x) for x in got) == want


def test_synth_rows_moments_and_slot_consistency():
    import numpy as np
    V = 8192
    sz = wl.synth_scale(3.0)
    se = np.array([wl.synth_scale(0.5)], dtype=np.float32)
    clean = wl.bf16_bits_to_f32(wl.synth_rows([0] * 4, [10, 11, 12, 13], [False] * 4, V, sz, se,
                                              3, 0)).astype(np.float64)
    assert abs(clean.mean()) < 0.05 and abs(clean.std() - 3.0) < 0.05
    # the same slot at another step: clean rows identical, MASK rows differ by
    # noise of the requested scale
    again = wl.bf16_bits_to_f32(wl.synth_rows([0], [11], [False], V, sz, se, 3, 7))
    assert np.array_equal(again[0], clean[1].astype(np.float32))
    m5 = wl.bf16_bits_to_f32(wl.synth_rows([0], [11], [True], V, sz, se, 3, 5)).astype(np.float64)
    m6 = wl.bf16_bits_to_f32(wl.synth_rows([0], [11], [True], V, sz, se, 3, 6)).astype(np.float64)
    d5, d6 = m5[0] - clean[1], m6[0] - clean[1]
    assert abs(d5.std() - 0.5) < 0.03 and abs(d6.std() - 0.5) < 0.03
    assert abs(np.corrcoef(d5, d6)[0, 1]) < 0.05
    # another request, same slot: independent values
    other = wl.bf16_bits_to_f32(wl.synth_rows([1], [11], [False], V, sz, se, 3, 0))
    assert abs(np.corrcoef(other[0], clean[1])[0, 1]) < 0.05
