"""Seeded synthetic inputs for the ISD step: the only code the CUDA path and the
CPU oracle's tests share.

This module draws random numbers and lays them out in the shapes the step
takes.  It holds none of the step's arithmetic (no softmax, no acceptance, no
attention).  Every tensor comes from a CPU ``torch.Generator`` with a fixed
seed, so a test can hand the same inputs to the library and to the oracle.

Workloads (the pages measure on public benchmarks that are not used here; these
synthetic batches stand in for them with the pages' stride N=4 and batch C=64):

=========================  ====================================================
``isd_tiny_c1_n2_f32``     C=1, N=2 (3 rows), 4 q / 1 kv heads, D=64, fp32,
                           256-token context in 16-token shuffled pages,
                           V=1024, clean logits N(0, 2^2), MASK logits = clean
                           + N(0, 0.5^2).
``isd_c4_n4_ctx512_2048``  C=4, N=4 (7 rows), 32/8 heads, D=128, bf16 KV,
                           context U[512, 2048], shuffled page pool,
                           V=151936, logits N(0, 3^2), MASK logits = clean +
                           sigma * N(0, 1), sigma set for mean
                           sum(min(p, q)) ~ 0.9.
``isd_c64_n4_ctx4096``     C=64, N=4, every context 4096, otherwise as above:
                           the headline batch.
``isd_c64_n4_ctx1k_32k``   C=64, N=4, context log-uniform in [1024, 32768],
                           per-request acceptance target from {0.5, 0.9,
                           0.99}, fragmented page pool (holes).
``lora_layer_m448``        one decoder layer's projections, hidden 4096, FFN
                           12288, 32/8 heads, rank-16 LoRA on q/k/v/o/gate/up/
                           down, weights N(0, 0.02^2), 448 rows (64 x 7) with
                           the gate on at MASK rows, plus attention over 4096
                           cached tokens.
=========================  ====================================================

The noise scale sigma per acceptance target is read from ``noise_table.json``
beside this module (input-generation parameters only), written by
``tests/golden/make_noise_table.py`` (a bisection that calls the oracle's
softmax only; the script is test infrastructure, the table is data).
"""

import json
import math
import os
from dataclasses import dataclass, field

import torch

FULL = 1
FRESH = 0

_HERE = os.path.dirname(os.path.abspath(__file__))
NOISE_TABLE = os.path.join(_HERE, "noise_table.json")


@dataclass(frozen=True)
class Workload:
    name: str
    C: int
    N: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    V: int
    dtype: str                 # "f32" or "bf16": KV, Q and logits storage
    ctx: str                   # "fixed", "uniform" or "loguniform"
    ctx_lo: int
    ctx_hi: int
    logit_std: float
    mask_noise: float = -1.0   # fixed sigma, or -1: from the noise table
    targets: tuple = (0.9,)    # acceptance targets drawn per request
    page_layout: str = "shuffled"   # or "fragmented"
    temperature: float = 1.0
    # gated-LoRA layer (lora_layer_m448 only)
    hidden: int = 0
    ffn: int = 0
    lora_rank: int = 0
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def rows_full(self):
        return 2 * self.N - 1

    @property
    def T(self):
        return self.C * self.rows_full

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "isd_tiny_c1_n2_f32": Workload(
        "isd_tiny_c1_n2_f32", C=1, N=2, Hq=4, Hkv=1, D=64, page_size=16, V=1024,
        dtype="f32", ctx="fixed", ctx_lo=256, ctx_hi=256, logit_std=2.0,
        mask_noise=0.5),
    "isd_c4_n4_ctx512_2048": Workload(
        "isd_c4_n4_ctx512_2048", C=4, N=4, Hq=32, Hkv=8, D=128, page_size=16,
        V=151936, dtype="bf16", ctx="uniform", ctx_lo=512, ctx_hi=2048,
        logit_std=3.0),
    "isd_c64_n4_ctx4096": Workload(
        "isd_c64_n4_ctx4096", C=64, N=4, Hq=32, Hkv=8, D=128, page_size=16,
        V=151936, dtype="bf16", ctx="fixed", ctx_lo=4096, ctx_hi=4096,
        logit_std=3.0),
    "isd_c64_n4_ctx1k_32k": Workload(
        "isd_c64_n4_ctx1k_32k", C=64, N=4, Hq=32, Hkv=8, D=128, page_size=16,
        V=151936, dtype="bf16", ctx="loguniform", ctx_lo=1024, ctx_hi=32768,
        logit_std=3.0, targets=(0.5, 0.9, 0.99), page_layout="fragmented"),
    "lora_layer_m448": Workload(
        "lora_layer_m448", C=64, N=4, Hq=32, Hkv=8, D=128, page_size=16,
        V=151936, dtype="bf16", ctx="fixed", ctx_lo=4096, ctx_hi=4096,
        logit_std=3.0, hidden=4096, ffn=12288, lora_rank=16),
}

HEADLINE = "isd_c64_n4_ctx4096"


def noise_table():
    with open(NOISE_TABLE) as f:
        return {float(k): float(v) for k, v in json.load(f)["sigma"].items()}


def _gen(seed):
    return torch.Generator().manual_seed(int(seed))


def context_lengths(w, g):
    if w.ctx == "fixed":
        return torch.full((w.C,), w.ctx_lo, dtype=torch.int64)
    if w.ctx == "uniform":
        return torch.randint(w.ctx_lo, w.ctx_hi + 1, (w.C,), generator=g)
    lo, hi = math.log(w.ctx_lo), math.log(w.ctx_hi)
    u = torch.rand(w.C, generator=g, dtype=torch.float64)
    return torch.exp(lo + u * (hi - lo)).round().to(torch.int64).clamp(w.ctx_lo, w.ctx_hi)


def page_tables(w, seq_lens, g, slack_rows=None):
    """Per-request page lists covering L_c + slack_rows slots.

    slack_rows defaults to N: room to commit up to N rows after the step.
    Unused table entries hold -1.  "shuffled": the pool is exactly the pages in
    use, handed out in a random order.  "fragmented": the pool is 25% larger
    and the pages in use are a random subset of it (holes), in random order.
    Returns (page_table int32 [C, max_pages], num_pages).
    """
    slack = w.N if slack_rows is None else slack_rows
    need = [(int(L) + slack + w.page_size - 1) // w.page_size for L in seq_lens]
    total = sum(need)
    pool = total if w.page_layout == "shuffled" else (total * 5 + 3) // 4
    perm = torch.randperm(pool, generator=g)[:total]
    max_pages = max(need)
    table = torch.full((w.C, max_pages), -1, dtype=torch.int32)
    at = 0
    for c, n in enumerate(need):
        table[c, :n] = perm[at:at + n].to(torch.int32)
        at += n
    return table, pool


def attention_inputs(w, seed=0, mode=None):
    """Q / new K, V rows and the paged cache of one step.

    mode: [C] FULL/FRESH per request (default: all FULL), which fixes the
    number of rows per request (2N-1 or N).
    """
    g = _gen(seed)
    dt = w.torch_dtype
    if mode is None:
        mode = torch.full((w.C,), FULL, dtype=torch.int64)
    rows = torch.where(mode == FULL, 2 * w.N - 1, w.N)
    qo_indptr = torch.zeros(w.C + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.cumsum(rows, 0).to(torch.int32)
    T = int(qo_indptr[-1])
    seq_lens = context_lengths(w, g)
    page_table, num_pages = page_tables(w, seq_lens, g)
    q = torch.randn(T, w.Hq, w.D, generator=g).to(dt)
    k_new = torch.randn(T, w.Hkv, w.D, generator=g).to(dt)
    v_new = torch.randn(T, w.Hkv, w.D, generator=g).to(dt)
    k_cache = torch.randn(num_pages, w.Hkv, w.page_size, w.D, generator=g).to(dt)
    v_cache = torch.randn(num_pages, w.Hkv, w.page_size, w.D, generator=g).to(dt)
    return dict(q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                page_table=page_table, seq_lens=seq_lens.to(torch.int32),
                qo_indptr=qo_indptr, num_pages=num_pages,
                sm_scale=1.0 / math.sqrt(w.D))


def acceptance_targets(w, g):
    idx = torch.randint(0, len(w.targets), (w.C,), generator=g)
    return [w.targets[int(i)] for i in idx]


def accept_inputs(w, seed=0):
    """Logits of a two-step sequence: a FRESH step, then a FULL step.

    Step 0 (every request FRESH): rows [clean, MASK x (N-1)].  Its MASK row k
    is the q-logit row of draft k for step 1: the clean logits of step 1's row
    k-1 plus sigma_c * N(0, 1), with sigma_c set from the request's
    acceptance target (or fixed by the workload).
    Step 1 (every request FULL): rows [N clean, N-1 MASK] with clean and MASK
    logits N(0, logit_std^2).
    Logits are drawn in float32 and stored in the workload dtype.
    """
    g = _gen(seed + 1)
    dt = w.torch_dtype
    C, N, V = w.C, w.N, w.V
    M = N - 1
    targets = acceptance_targets(w, g)
    if w.mask_noise >= 0:
        sig = [w.mask_noise] * C
    else:
        table = noise_table()
        sig = [table[t] for t in targets]
    logits1 = torch.randn(C * (2 * N - 1), V, generator=g) * w.logit_std
    logits0 = torch.empty(C * N, V)
    for c in range(C):
        r1 = c * (2 * N - 1)
        r0 = c * N
        logits0[r0] = torch.randn(V, generator=g) * w.logit_std
        for k in range(1, M + 1):
            noise = torch.randn(V, generator=g)
            logits0[r0 + k] = logits1[r1 + k - 1] + sig[c] * noise
    qo0 = torch.arange(0, C * N + 1, N, dtype=torch.int32)
    qo1 = torch.arange(0, C * (2 * N - 1) + 1, 2 * N - 1, dtype=torch.int32)
    return dict(
        logits0=logits0.to(dt), qo0=qo0, mode0=torch.full((C,), FRESH, dtype=torch.uint8),
        logits1=logits1.to(dt), qo1=qo1, mode1=torch.full((C,), FULL, dtype=torch.uint8),
        targets=targets, sigma=sig, temperature=w.temperature)


def lora_inputs(w, seed=0, rank=None):
    """Weights and activations of one decoder layer's seven projections.

    Projections (K -> N): q 4096->4096, k 4096->1024, v 4096->1024,
    o 4096->4096, gate 4096->12288, up 4096->12288, down 12288->4096, each
    with a rank-r LoRA pair (A: [r, K], B: [N, r]); all weights N(0, 0.02^2).
    x: [M, hidden] N(0, 1).  row_gate: 1 at MASK rows (rows N..2N-2 of each
    request's 2N-1 rows), 0 elsewhere.
    """
    g = _gen(seed + 2)
    H, F = w.hidden, w.ffn
    r = w.lora_rank if rank is None else rank
    kvd = w.Hkv * w.D
    shapes = dict(q=(H, H), k=(kvd, H), v=(kvd, H), o=(H, H), gate=(F, H),
                  up=(F, H), down=(H, F))
    M = w.T
    x = torch.randn(M, H, generator=g).bfloat16()
    proj = {}
    for name, (n, k) in shapes.items():
        proj[name] = dict(
            w=(torch.randn(n, k, generator=g) * 0.02).bfloat16(),
            a=(torch.randn(r, k, generator=g) * 0.02).bfloat16(),
            b=(torch.randn(n, r, generator=g) * 0.02).bfloat16())
    pos = torch.arange(M) % (2 * w.N - 1)
    row_gate = (pos >= w.N).to(torch.uint8)
    return dict(x=x, proj=proj, row_gate=row_gate, lora_scale=1.0, rank=r)


def fuse_projections(proj, names):
    """One projection equal to several that share their input (q|k|v, gate|up):
    weights stacked along N, adapters stacked along the rank (A) with B block
    diagonal, so row block i of the output is projection i's output (the
    other blocks' adapter columns meet zeros in B).  Data layout only."""
    ws = [proj[n]["w"] for n in names]
    As = [proj[n]["a"] for n in names]
    Bs = [proj[n]["b"] for n in names]
    W = torch.cat(ws, 0)
    A = torch.cat(As, 0)
    B = torch.zeros(W.shape[0], sum(a.shape[0] for a in As), dtype=Bs[0].dtype)
    n0 = r0 = 0
    for b in Bs:
        B[n0:n0 + b.shape[0], r0:r0 + b.shape[1]] = b
        n0 += b.shape[0]
        r0 += b.shape[1]
    return dict(w=W, a=A, b=B)



# ---------------------------------------------------------------------------
# Synthetic model for multi-step loops: logit rows as a function of
# (request, slot, step).  The same definition runs on the GPU in
# idlm_synth_logits; this is its CPU twin (bit-identical by construction).
# ---------------------------------------------------------------------------

PHILOX32_M = (0xD2511F53, 0xCD9E8D57)
PHILOX32_W = (0x9E3779B9, 0xBB67AE85)
SYNTH_KEY1 = 0x1D1A7E5D
IH8_CENTRE = 4 * 65535


def philox4x32_10(ctr, key):
    """Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) on numpy arrays.

    ctr: four counter words (ints or uint32-valued arrays, broadcast
    together); key: two key words.  Returns four uint64 arrays holding the
    32-bit output words."""
    import numpy as np
    m32 = np.uint64(0xFFFFFFFF)
    c0, c1, c2, c3 = np.broadcast_arrays(*[np.asarray(x, dtype=np.uint64) & m32 for x in ctr])
    k0, k1 = (np.uint64(int(k) & 0xFFFFFFFF) for k in key)
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(PHILOX32_W[0])) & m32
            k1 = (k1 + np.uint64(PHILOX32_W[1])) & m32
        p0 = c0 * np.uint64(PHILOX32_M[0])
        p1 = c2 * np.uint64(PHILOX32_M[1])
        c0, c1, c2, c3 = (((p1 >> np.uint64(32)) ^ c1 ^ k0) & m32, p1 & m32,
                          ((p0 >> np.uint64(32)) ^ c3 ^ k1) & m32, p0 & m32)
    return c0, c1, c2, c3


def ih8(words):
    """Centred sum of the eight 16-bit halves of four 32-bit words (int64)."""
    import numpy as np
    s = np.zeros(np.shape(words[0]), dtype=np.int64)
    for w in words:
        w = w.astype(np.int64)
        s += (w & 0xFFFF) + (w >> 16)
    return s - IH8_CENTRE


def synth_scale(std):
    """fp32 factor that turns a centred IH8 sum into a value of standard
    deviation `std` (the sum's variance is (2/3) 65536^2)."""
    import numpy as np
    return float(np.float32(std * math.sqrt(1.5) / 65536.0))


def f32_to_bf16_bits(x):
    """Round float32 values to bfloat16, nearest-even (finite values)."""
    import numpy as np
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def bf16_bits_to_f32(b):
    import numpy as np
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def synth_rows(req, pos, is_mask, V, scale_z, scale_e, seed, step):
    """Logit rows of the synthetic model (bf16 bits, uint16 [rows, V]).

    Row i of request req[i] at position pos[i] predicts slot pos[i] + 1; a
    clean row holds z(c, s) = fp32(IH8(c, s, 0)) * scale_z, a MASK row
    z(c, s) + fp32(IH8(c, s, 1 + step)) * scale_e[c], where IH8(c, s, d) is
    the centred sum of the halves of Philox4x32-10(counter = (v, s, c, d),
    key = (seed, 0x1D1A7E5D)).  Products and the sum are rounded to nearest
    in fp32, the result to nearest-even in bf16."""
    import numpy as np
    req = np.asarray(req, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    v = np.arange(V, dtype=np.uint64)[None, :]
    slot = (pos + 1).astype(np.uint64)[:, None]
    c = req.astype(np.uint64)[:, None]
    key = (seed, SYNTH_KEY1)
    sz = ih8(philox4x32_10((v, slot, c, 0), key))
    x = sz.astype(np.float32) * np.float32(scale_z)
    mask = np.asarray(is_mask, dtype=bool)
    if mask.any():
        rows = np.nonzero(mask)[0]
        sn = ih8(philox4x32_10((v, slot[rows], c[rows], 1 + int(step)), key))
        se = np.asarray(scale_e, dtype=np.float32)[req[rows]][:, None]
        x[rows] = x[rows] + sn.astype(np.float32) * se
    return f32_to_bf16_bits(x)



def layer_inputs(w, rank=None, seed=0, requests=None):
    """A whole decoder layer of the gated-LoRA workload, stacked the way
    idlm_risd_layer takes it: w_qkv = [Wq; Wk; Wv], a_qkv = [Aq; Ak; Av],
    b_qkv = [Bq; Bk; Bv], w_gu = [Wgate; Wup], a_gu, b_gu; plus the step's
    rows (x, MASK gate) and the attention's paged KV (the workload's contexts).
    rank overrides the adapters' rank (0: no adapters).  requests: keep only
    these requests' rows and KV (a smaller batch of the same layer)."""
    inp = lora_inputs(w, seed=seed, rank=rank if rank else (w.lora_rank if rank is None else 8))
    P = inp["proj"]
    cat = lambda names, key: torch.cat([P[n][key] for n in names])
    W = dict(w_qkv=cat("qkv", "w"), a_qkv=cat("qkv", "a"), b_qkv=cat("qkv", "b"),
             w_o=P["o"]["w"], a_o=P["o"]["a"], b_o=P["o"]["b"],
             w_gu=cat(("gate", "up"), "w"), a_gu=cat(("gate", "up"), "a"),
             b_gu=cat(("gate", "up"), "b"),
             w_down=P["down"]["w"], a_down=P["down"]["a"], b_down=P["down"]["b"])
    if rank == 0:
        for k in [k for k in W if k[0] in "ab"]:
            del W[k]
    a = attention_inputs(w, seed=seed)
    x, gate = inp["x"], inp["row_gate"]
    if requests is not None:
        qo = a["qo_indptr"]
        rows = torch.cat([torch.arange(int(qo[c]), int(qo[c + 1])) for c in requests])
        sub_qo = torch.zeros(len(requests) + 1, dtype=torch.int32)
        sub_qo[1:] = torch.cumsum(torch.tensor([int(qo[c + 1] - qo[c]) for c in requests]), 0)
        a = dict(a, page_table=a["page_table"][list(requests)], seq_lens=a["seq_lens"][list(requests)],
                 qo_indptr=sub_qo)
        x, gate = x[rows], gate[rows]
    return dict(W=W, x=x, row_gate=gate, rank=0 if rank == 0 else inp["rank"],
                k_cache=a["k_cache"], v_cache=a["v_cache"], page_table=a["page_table"],
                seq_lens=a["seq_lens"], qo_indptr=a["qo_indptr"], lora_scale=1.0)
