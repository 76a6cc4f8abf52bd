"""Plain float64 CPU oracle of the ISD verify/accept step.

Test infrastructure (see ``oracle/__init__``): not for the product path.

Page references (full titles in ``oracle/__init__``):
  [IDLM] "Introspective Diffusion Language Models" (project page)
  [GN]   "I-DLM - Icgozlemsel Difuzyon Dil Modelleri" (GeekNews summary)
  [OJ]   ojeo.com news note

What one ISD step computes, as read from the pages
---------------------------------------------------
[IDLM] "Inference & ISD" (and [GN] "I-DLM Yontemi", "Inference & ISD"): one
forward pass both proposes new tokens at MASK positions (distribution q) and
verifies earlier proposals at clean positions (anchor distribution p); a draft x
is kept with probability min(1, p(x)/q(x)), which keeps the output on the
autoregressive distribution.  [IDLM] "How do DLMs perform ..." fixes the query
count at 2N-1 per forward, and the speedup panel fixes the memory-bound tokens
per forward at TPF = (2 + p + ... + p^(N-2)) / (2 - p^(N-1)).

The row layout that gives exactly 2N-1 rows AND exactly that TPF (the reading
used throughout; the pages do not spell the layout out):

* FULL request (previous step accepted everything): rows
  [a, d_1 .. d_{N-1}, MASK x (N-1)] at positions L .. L+2N-2, where L is the
  committed length, a the token emitted last step (not yet in the KV cache)
  and d_i the drafts proposed last step.  With the logit shift of
  [IDLM] "Training" / [ABS], the output row at position t predicts position
  t+1, so clean row i-1 gives p_i, the anchor distribution for draft d_i, and
  clean row N-1 gives p_N for the slot after the last draft (the bonus slot).
  MASK row k gives q for the slot after it: the k-th draft of the next step.
* FRESH request (previous step ended in a rejection): rows
  [a, MASK x (N-1)]; row 0 gives p for one new token, the MASK rows give the
  next drafts.

Verification (FULL only): u_i < min(1, p_i(d_i) / q_i(d_i)) for i = 1, 2, ...
until the first failure.  q_i is softmax of the previous step's MASK row that
proposed d_i.  At the first rejection j the token is resampled from
normalize(max(0, p_j - q_j)) (the standard speculative-sampling residual; the
pages name only the min(1, p/q) rule).  If all N-1 drafts pass, one more token
is drawn from p_N.  A FRESH request draws its one token from p of row 0.

Commit: the anchor and the accepted drafts (rows 0 .. n_acc) enter the KV
cache; MASK rows and rejected drafts never do ("rollback").

Renewal count: a FULL step emits sum_{i<=N-1} p^i + 1 tokens on average and
stays FULL with probability p^(N-1); a FRESH step emits one token.  The
stationary tokens per forward is (2 + p + ... + p^(N-2)) / (2 - p^(N-1)),
the speedup panel's formula (pinned by simulation in the tests).

Sampling (bonus, fresh, residual and SAMPLE-mode proposals) is inverse-CDF
over the vocabulary in index order: the first v with sum_{t<=v} w_t > u * W.
The pages are silent on the sampler; this is the textbook definition.
"""

import numpy as np

from . import philox

FULL = 1
FRESH = 0
PROPOSE_ARGMAX = 0
PROPOSE_SAMPLE = 1

# Kinds of the token that ends a request's step (diagnostic output).
END_FRESH = 0
END_BONUS = 1
END_RESIDUAL = 2
END_RESIDUAL_FALLBACK = 3   # residual mass exactly zero: sample from p_j


# ---------------------------------------------------------------------------
# Row layout
# ---------------------------------------------------------------------------

def rows_per_request(mode, N):
    """2N-1 rows for a FULL request, N rows for a FRESH one.

    [IDLM] "How do DLMs perform ...": I-DLM processes 2N-1 queries per forward.
    """
    mode = np.asarray(mode)
    return np.where(mode == FULL, 2 * N - 1, N).astype(np.int64)


def clean_rows(mode, N):
    """Clean (non-MASK) rows at the head of each request's block."""
    return np.where(np.asarray(mode) == FULL, N, 1).astype(np.int64)


# ---------------------------------------------------------------------------
# Distributions
# ---------------------------------------------------------------------------

def softmax_t(logits, temperature):
    """softmax(x / T) along the last axis in float64.

    T == 0 means greedy: the one-hot vector of the first (lowest-index)
    maximum.  The pages' quick start samples at temperature 1.0
    ([IDLM] "Quick Start").
    """
    x = np.asarray(logits, dtype=np.float64)
    if temperature == 0:
        out = np.zeros_like(x)
        idx = np.argmax(x, axis=-1)
        np.put_along_axis(out, idx[..., None], 1.0, axis=-1)
        return out
    z = x / temperature
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


def row_stats(logits, temperature):
    """(max_v x_v/T, sum_v exp(x_v/T - max)) per row: the softmax normaliser.

    For T == 0 the stats of the one-hot distribution are reported as
    (max_v x_v, 1).
    """
    x = np.asarray(logits, dtype=np.float64)
    if temperature == 0:
        return x.max(axis=-1), np.ones(x.shape[:-1])
    z = x / temperature
    m = z.max(axis=-1)
    return m, np.exp(z - m[..., None]).sum(axis=-1)


def sample_icdf(weights, u):
    """Inverse-CDF draw from unnormalised weights, one draw per row.

    weights: [K, V] non-negative, each row with positive total.  u: [K] in
    [0, 1).  Returns (tokens [K], margins [K]) where the token is the first v
    whose running sum (index order) exceeds u times the row total, and the
    margin is the distance of u*total to the nearer edge of that token's CDF
    interval, divided by the total (a small margin means a tie a different
    summation order could break differently).
    """
    w = np.asarray(weights, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    cum = np.cumsum(w, axis=-1)
    total = cum[:, -1]
    target = u * total
    tok = np.argmax(cum > target[:, None], axis=-1)
    rows = np.arange(w.shape[0])
    upper = cum[rows, tok] - target
    lower = target - np.where(tok > 0, cum[rows, np.maximum(tok - 1, 0)], 0.0)
    return tok.astype(np.int64), np.minimum(upper, lower) / total


# ---------------------------------------------------------------------------
# a2: paged strict-causal GQA attention of the step's rows
# ---------------------------------------------------------------------------

def gather_cache(cache, page_table_row, length, page_size):
    """Logical slots 0..length-1 of one request from a paged cache.

    cache: [num_pages, Hkv, page_size, D]; slot s lives in page
    page_table_row[s // page_size] at offset s % page_size.
    Returns [length, Hkv, D].
    """
    slots = np.arange(length)
    pages = np.asarray(page_table_row)[slots // page_size]
    return cache[pages, :, slots % page_size, :]


def isd_attention(q, k_new, v_new, k_cache, v_cache, page_table, seq_lens,
                  qo_indptr, page_size, sm_scale):
    """Strict-causal attention of every step row against its request's context.

    Row r of request c sits at absolute position L_c + r and attends to the
    committed slots 0..L_c-1 (read through the page table) and to this step's
    own new keys/values of rows 0..r ([IDLM] "Training": strict causal masking
    across all positions; "Serving (SGLang)": paged KV cache).  Query head h
    reads KV head h // (Hq / Hkv) (grouped-query attention; the pages name the
    Qwen3 base models, which use contiguous groups).  Scores are scaled by
    sm_scale (1/sqrt(D) in every workload).  Q and K are taken as given: no
    positional rotation is applied here (the pages are silent on it).

    q: [T, Hq, D]; k_new, v_new: [T, Hkv, D]; caches: [P, Hkv, page_size, D];
    page_table: [C, max_pages]; seq_lens: [C]; qo_indptr: [C+1].
    Returns float64 [T, Hq, D].
    """
    q = np.asarray(q, dtype=np.float64)
    k_new = np.asarray(k_new, dtype=np.float64)
    v_new = np.asarray(v_new, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = k_new.shape[1]
    group = Hq // Hkv
    out = np.zeros((T, Hq, D))
    for c in range(len(seq_lens)):
        L = int(seq_lens[c])
        t0, t1 = int(qo_indptr[c]), int(qo_indptr[c + 1])
        kc = gather_cache(k_cache, page_table[c], L, page_size).astype(np.float64)
        vc = gather_cache(v_cache, page_table[c], L, page_size).astype(np.float64)
        for r in range(t1 - t0):
            keys = np.concatenate([kc, k_new[t0:t0 + r + 1]], axis=0)
            vals = np.concatenate([vc, v_new[t0:t0 + r + 1]], axis=0)
            for h in range(Hq):
                g = h // group
                s = keys[:, g, :] @ q[t0 + r, h] * sm_scale
                p = np.exp(s - s.max())
                p /= p.sum()
                out[t0 + r, h] = p @ vals[:, g, :]
    return out


# ---------------------------------------------------------------------------
# a4-a7: vocab pass, accept scan, residual resample, proposals, next state
# ---------------------------------------------------------------------------

def isd_accept(logits, qo_indptr, mode, drafts, prev_logits, prev_mask_row0,
               N, temperature, proposal_mode, seed, step, request_ids=None):
    """One ISD accept step for a batch of requests.

    logits: [T, V] this step's output rows, laid out per request as the module
        docstring says (FULL: N clean + N-1 MASK; FRESH: 1 clean + N-1 MASK).
    qo_indptr: [C+1] first row of each request.
    mode: [C] FULL (1) or FRESH (0).
    drafts: [C, N-1] tokens proposed last step (read for FULL requests only).
    prev_logits, prev_mask_row0: the previous step's logits and, per request,
        the row that proposed draft 1 (draft i came from row
        prev_mask_row0 + i - 1).  Only FULL requests read them.
    proposal_mode: PROPOSE_ARGMAX (the pages' serving default, [IDLM]
        "Serving (SGLang)": argmax proposals) or PROPOSE_SAMPLE.
    seed, step, request_ids: select the Philox draws (see oracle.philox).

    Returns a dict of arrays (see the keys at the end).
    """
    x = np.asarray(logits, dtype=np.float64)
    mode = np.asarray(mode).astype(np.int64)
    qo_indptr = np.asarray(qo_indptr).astype(np.int64)
    C = mode.shape[0]
    M = N - 1
    req = np.arange(C) if request_ids is None else np.asarray(request_ids)
    full = mode == FULL
    n_clean = clean_rows(mode, N)
    row0 = qo_indptr[:-1]
    if not np.array_equal(qo_indptr[1:] - row0, n_clean + M):
        raise ValueError("qo_indptr does not match the FULL/FRESH row layout")

    P = softmax_t(x, temperature)                        # p or q of every row
    rmax, rsum = row_stats(x, temperature)

    # -- verification: u_i < min(1, p_i(d_i) / q_i(d_i)), FULL requests only
    u = philox.accept_uniforms(seed, step, req, M)        # [C, M]
    p_d = np.zeros((C, M))
    q_d = np.zeros((C, M))
    ratio = np.zeros((C, M))
    ok = np.zeros((C, M), dtype=bool)
    fr = np.nonzero(full)[0]
    if fr.size:
        d = np.asarray(drafts)[fr].astype(np.int64)
        prev = np.asarray(prev_logits, dtype=np.float64)
        pm0 = np.asarray(prev_mask_row0).astype(np.int64)[fr]
        for i in range(1, M + 1):
            p_row = P[row0[fr] + i - 1]                   # p_i: clean row i-1
            q_row = softmax_t(prev[pm0 + i - 1], temperature)   # q_i
            pv = p_row[np.arange(fr.size), d[:, i - 1]]
            qv = q_row[np.arange(fr.size), d[:, i - 1]]
            with np.errstate(divide="ignore", invalid="ignore"):
                rt = np.where(qv > 0, pv / np.where(qv > 0, qv, 1.0), np.inf)
            p_d[fr, i - 1] = pv
            q_d[fr, i - 1] = qv
            ratio[fr, i - 1] = rt
            ok[fr, i - 1] = u[fr, i - 1] < np.minimum(1.0, rt)
    # accepted drafts = length of the leading run of passes
    n_acc = np.zeros(C, dtype=np.int64)
    alive = full.copy()
    for i in range(M):
        alive = alive & ok[:, i]
        n_acc += alive
    all_acc = full & (n_acc == M)
    rejected = full & (n_acc < M)

    # -- the token that ends the step
    final = np.full(C, -1, dtype=np.int64)
    margin = np.full(C, np.inf)
    kind = np.full(C, -1, dtype=np.int64)
    u_s = philox.sample_uniform(seed, step, req)
    u_r = philox.residual_uniform(seed, step, req)
    draw_p = np.nonzero(~rejected)[0]           # bonus (FULL) or fresh token
    if draw_p.size:
        srow = row0[draw_p] + n_clean[draw_p] - 1
        tok, mg = sample_icdf(P[srow], u_s[draw_p])
        final[draw_p] = tok
        margin[draw_p] = mg
        kind[draw_p] = np.where(full[draw_p], END_BONUS, END_FRESH)
    rj = np.nonzero(rejected)[0]
    if rj.size:
        j = n_acc[rj] + 1                              # first rejected draft
        p_j = P[row0[rj] + j - 1]
        prev = np.asarray(prev_logits, dtype=np.float64)
        q_j = softmax_t(prev[np.asarray(prev_mask_row0)[rj] + j - 1], temperature)
        w = np.maximum(p_j - q_j, 0.0)
        empty = w.sum(axis=1) == 0
        w[empty] = p_j[empty]
        tok, mg = sample_icdf(w, u_r[rj])
        final[rj] = tok
        margin[rj] = mg
        kind[rj] = np.where(empty, END_RESIDUAL_FALLBACK, END_RESIDUAL)

    # -- proposals of the next step's drafts from the MASK rows
    mrows = row0[:, None] + n_clean[:, None] + np.arange(M)[None, :]   # [C, M]
    prop_margin = np.full((C, M), np.inf)
    if proposal_mode == PROPOSE_ARGMAX:
        proposals = np.argmax(x[mrows.reshape(-1)], axis=-1).reshape(C, M)
    else:
        up = philox.propose_uniforms(seed, step, req, M)
        tok, mg = sample_icdf(P[mrows.reshape(-1)], up.reshape(-1))
        proposals = tok.reshape(C, M)
        prop_margin = mg.reshape(C, M)
    next_mode = np.where(rejected, FRESH, FULL).astype(np.int64)
    next_drafts = np.where(next_mode[:, None] == FULL, proposals, -1)

    # -- emitted tokens: accepted drafts, then the final token
    out_tokens = np.full((C, N), -1, dtype=np.int64)
    for i in range(M):
        keep = n_acc > i                       # draft i+1 was accepted
        out_tokens[keep, i] = np.asarray(drafts)[keep, i]
    out_tokens[np.arange(C), n_acc] = final
    n_out = n_acc + 1
    n_commit = np.where(full, 1 + n_acc, 1)

    return dict(
        n_accepted=n_acc, out_tokens=out_tokens, n_out=n_out, n_commit=n_commit,
        next_drafts=next_drafts, next_mode=next_mode,
        next_mask_row0=row0 + n_clean,
        u=u, p_draft=p_d, q_draft=q_d, ratio=ratio,
        final_token=final, final_margin=margin, final_kind=kind,
        proposals=proposals, propose_margin=prop_margin,
        row_max=rmax, row_sum=rsum,
    )


# ---------------------------------------------------------------------------
# a8: KV commit / rollback
# ---------------------------------------------------------------------------

def kv_commit(k_cache, v_cache, page_table, seq_lens, k_new, v_new, qo_indptr,
              n_commit, page_size):
    """Append the committed rows' K/V to the paged cache.

    Rows 0 .. n_commit[c]-1 of request c (the anchor and its accepted drafts,
    or the one clean row of a FRESH request) go to logical slots
    L_c .. L_c + n_commit[c] - 1.  The other rows (rejected drafts, MASK rows)
    are never written, which is the rollback ([IDLM] "Serving (SGLang)":
    paged KV cache).  Pages wholly past the new length are returned as
    releasable: releasable_from[c] = ceil(new_len / page_size).

    Raises ValueError on a page id outside the pool, a slot outside the page
    table row, or n_commit larger than the request's rows.
    Returns (k_cache', v_cache', seq_lens', releasable_from).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    num_pages = kc.shape[0]
    max_pages = page_table.shape[1]
    seq_out = np.asarray(seq_lens).astype(np.int64).copy()
    for c in range(len(seq_lens)):
        L = int(seq_lens[c])
        t0, t1 = int(qo_indptr[c]), int(qo_indptr[c + 1])
        n = int(n_commit[c])
        if n < 0 or n > t1 - t0:
            raise ValueError(f"request {c}: n_commit {n} outside its {t1 - t0} rows")
        for j in range(n):
            slot = L + j
            if slot // page_size >= max_pages:
                raise ValueError(f"request {c}: slot {slot} beyond its page table")
            page = int(page_table[c, slot // page_size])
            if not 0 <= page < num_pages:
                raise ValueError(f"request {c}: page id {page} outside the pool")
            kc[page, :, slot % page_size, :] = k_new[t0 + j]
            vc[page, :, slot % page_size, :] = v_new[t0 + j]
        seq_out[c] = L + n
    releasable_from = -(-seq_out // page_size)
    return kc, vc, seq_out, releasable_from


# ---------------------------------------------------------------------------
# a3: gated LoRA (R-ISD)
# ---------------------------------------------------------------------------

def gated_lora(x, w, lora_a, lora_b, row_gate, lora_scale, store=None):
    """Y = X W^T + g * s * (X A^T) B^T with g = 1 only at MASK rows.

    [IDLM] "Lossless R-ISD" / [GN] "Speedup Factor Explorer": the LoRA adapter
    is active only at MASK positions; verify positions use the base weights
    alone, so their outputs equal the base model's bit for bit.
    x: [M, K], w: [N, K], lora_a: [r, K], lora_b: [N, r], row_gate: [M].
    store: the rounding applied to the rank-r intermediate T = g s X A^T
    where an implementation stores it (None: exact float64).
    """
    x = np.asarray(x, dtype=np.float64)
    base = x @ np.asarray(w, dtype=np.float64).T
    t = x @ np.asarray(lora_a, dtype=np.float64).T
    t = t * (np.asarray(row_gate, dtype=np.float64)[:, None] * lora_scale)
    if store is not None:
        t = store(t)
    return base + t @ np.asarray(lora_b, dtype=np.float64).T


def gated_lora_grouped(x, w, lora_a, lora_b, row_gate, lora_scale, group_rows, store=None):
    """Several gated-LoRA projections of one input with stacked weights.

    Group g owns weight rows [sum(group_rows[:g]), sum(group_rows[:g+1]));
    lora_a stacks the groups' A matrices ([ngroups * r, K]) and lora_b holds
    each weight row's B row ([N, r]).  Each group is gated_lora with its own
    A and B; the outputs sit side by side along N.
    """
    ng = len(group_rows)
    r = np.asarray(lora_a).shape[0] // ng
    outs, n0 = [], 0
    for g, n in enumerate(group_rows):
        outs.append(gated_lora(x, np.asarray(w)[n0:n0 + n], np.asarray(lora_a)[g * r:(g + 1) * r],
                               np.asarray(lora_b)[n0:n0 + n], row_gate, lora_scale, store))
        n0 += n
    return np.concatenate(outs, axis=1)


# ---------------------------------------------------------------------------
# One R-ISD decoder layer ([IDLM] "Lossless R-ISD"; pre-norm layout of the
# Qwen3-style base models the pages convert -- the pages do not spell the
# layer out)
# ---------------------------------------------------------------------------

def round_bf16(x):
    """Nearest bfloat16 of each value (through float32, ties to even)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def rmsnorm(x, eps, weight=None):
    """x / sqrt(mean(x^2) + eps) * weight along the last axis (weight 1 if None)."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if weight is None else y * np.asarray(weight, dtype=np.float64)


def silu(x):
    """x * sigmoid(x) = x / (1 + exp(-x))."""
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def risd_layer(x, W, row_gate, lora_scale, eps, n_heads, n_kv_heads, head_dim,
               k_cache, v_cache, page_table, seq_lens, qo_indptr, page_size, store=None):
    """One decoder layer over the step's rows, gated LoRA at MASK rows.

    W: dict with w_qkv [(Hq+2Hkv)D, H], a_qkv [3r, H], b_qkv [(Hq+2Hkv)D, r],
    w_o [H, Hq D], a_o, b_o, w_gu [2F, H] (gate rows, then up rows), a_gu
    [2r, H], b_gu, w_down [H, F], a_down, b_down, norm1, norm2 ([H] or None);
    rank 0 means no adapters (a_* of zero rows).  store: the rounding applied
    where an implementation stores an activation, the adapters' rank-r
    intermediates included (None: exact float64).

        n1 = RMSNorm(x)               h  = x + a Wo^T (+ LoRA)
        [q|k|v] = n1 Wqkv^T (+ LoRA)  n2 = RMSNorm(h)
        a = isd_attention(q, k, v)    [g|u] = n2 Wgu^T (+ LoRA)
                                      out = h + (silu(g) * u) Wd^T (+ LoRA)
    Returns (out, k_new, v_new).
    """
    st = store or (lambda a: a)
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    nq, nkv = n_heads * head_dim, n_kv_heads * head_dim
    F = np.asarray(W["w_gu"]).shape[0] // 2

    def proj(inp, w, a, b, rows):
        if np.asarray(a).shape[0] == 0:
            return np.asarray(inp, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T
        return gated_lora_grouped(inp, w, a, b, row_gate, lora_scale, rows, store)

    n1 = st(rmsnorm(x, eps, W.get("norm1")))
    qkv = st(proj(n1, W["w_qkv"], W["a_qkv"], W["b_qkv"], [nq, nkv, nkv]))
    q = qkv[:, :nq].reshape(T, n_heads, head_dim)
    k_new = qkv[:, nq:nq + nkv].reshape(T, n_kv_heads, head_dim)
    v_new = qkv[:, nq + nkv:].reshape(T, n_kv_heads, head_dim)
    a = st(isd_attention(q, k_new, v_new, k_cache, v_cache, page_table, seq_lens, qo_indptr,
                         page_size, 1.0 / np.sqrt(head_dim)).reshape(T, nq))
    o = st(proj(a, W["w_o"], W["a_o"], W["b_o"], [H]))
    h = st(x + o)
    n2 = st(rmsnorm(h, eps, W.get("norm2")))
    gu = st(proj(n2, W["w_gu"], W["a_gu"], W["b_gu"], [F, F]))
    act = st(silu(gu[:, :F]) * gu[:, F:])
    d = st(proj(act, W["w_down"], W["a_down"], W["b_down"], [H]))
    return st(h + d), k_new, v_new


# ---------------------------------------------------------------------------
# Closed forms of the pages
# ---------------------------------------------------------------------------

def tpf_closed_form(p, N):
    """Tokens per forward in the memory-bound regime.

    [IDLM] speedup panel / [GN] "Speedup Factor Explorer":
    TPF = (2 + p + ... + p^(N-2)) / (2 - p^(N-1)).
    """
    num = 2.0 + sum(p ** k for k in range(1, N - 1))
    return num / (2.0 - p ** (N - 1))


def compute_efficiency(tpf, N):
    """TPF^2 / query_size with 2N-1 queries per forward.

    [IDLM] "How do DLMs perform as they approach compute-bound?".
    """
    return tpf * tpf / (2 * N - 1)


# ---------------------------------------------------------------------------
# Multi-step decode loop (used by the pins of the closed form and of the
# output distribution)
# ---------------------------------------------------------------------------

MASK_TOKEN = -1


def isd_decode(model, first_token, N, n_steps, temperature, proposal_mode,
               seed, step0=0, start_len=None, with_positions=False):
    """Run n_steps ISD steps for a batch of requests from FRESH.

    model(row_tok, row_req, row_mask_k, row_last_clean) -> logits [T, V]:
        row_tok is the input token of each row (MASK_TOKEN at MASK rows),
        row_req its request, row_mask_k the MASK offset k = 1..N-1 (0 at
        clean rows) and row_last_clean the input token of the request's last
        clean row in this step.  With with_positions=True the model also
        receives row_pos, the absolute position of each row: the request's
        committed length L plus the row's offset in its block (the rows sit
        at L .. L + rows - 1; the module docstring's layout).
    first_token: [C] the token each request starts from (the end of its
        prompt, not yet in the cache).
    start_len: [C] committed lengths at the start (default 0); every step
        adds its n_commit.
    Returns (emitted [C, N*n_steps] padded with -1, n_emitted [C],
    per_step [n_steps, C] tokens emitted by each step).
    """
    first_token = np.asarray(first_token).astype(np.int64)
    C = first_token.shape[0]
    M = N - 1
    mode = np.full(C, FRESH, dtype=np.int64)
    pending = first_token.copy()
    drafts = np.full((C, M), -1, dtype=np.int64)
    prev_logits = None
    prev_mask_row0 = np.zeros(C, dtype=np.int64)
    emitted = np.full((C, N * n_steps), -1, dtype=np.int64)
    n_emitted = np.zeros(C, dtype=np.int64)
    per_step = np.zeros((n_steps, C), dtype=np.int64)
    length = (np.zeros(C, dtype=np.int64) if start_len is None
              else np.asarray(start_len).astype(np.int64).copy())
    for s in range(n_steps):
        n_rows = rows_per_request(mode, N)
        qo = np.concatenate([[0], np.cumsum(n_rows)])
        Ttot = int(qo[-1])
        row_req = np.repeat(np.arange(C), n_rows)
        pos = np.arange(Ttot) - qo[row_req]
        ncl = clean_rows(mode, N)[row_req]
        is_mask = pos >= ncl
        row_tok = np.full(Ttot, MASK_TOKEN, dtype=np.int64)
        row_tok[pos == 0] = pending
        dpos = (~is_mask) & (pos > 0)
        row_tok[dpos] = drafts[row_req[dpos], pos[dpos] - 1]
        row_mask_k = np.where(is_mask, pos - ncl + 1, 0)
        last_clean = np.where(mode == FULL, drafts[:, M - 1], pending)
        row_last_clean = last_clean[row_req]
        if with_positions:
            logits = model(row_tok, row_req, row_mask_k, row_last_clean, length[row_req] + pos)
        else:
            logits = model(row_tok, row_req, row_mask_k, row_last_clean)
        if prev_logits is None:
            prev_logits = np.zeros((1, logits.shape[1]))
        out = isd_accept(logits, qo, mode, drafts, prev_logits, prev_mask_row0,
                         N, temperature, proposal_mode, seed, step0 + s)
        for k in range(N):
            sel = np.nonzero(out["n_out"] > k)[0]
            emitted[sel, n_emitted[sel] + k] = out["out_tokens"][sel, k]
        n_emitted += out["n_out"]
        per_step[s] = out["n_out"]
        pending = out["out_tokens"][np.arange(C), out["n_out"] - 1]
        drafts = out["next_drafts"]
        mode = out["next_mode"]
        prev_logits = logits
        prev_mask_row0 = out["next_mask_row0"]
        length += out["n_commit"]
    return emitted, n_emitted, per_step
