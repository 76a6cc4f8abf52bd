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
