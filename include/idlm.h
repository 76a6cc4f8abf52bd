/*
 * idlm.h -- C ABI of the Introspective Strided Decoding (ISD) step on B300.
 *
 * One ISD step of an Introspective Diffusion Language Model proposes new
 * tokens at MASK positions (distribution q) and verifies the previous step's
 * proposals at clean positions (anchor distribution p) in one forward pass,
 * keeping a draft x with probability min(1, p(x)/q(x)).  Sources, cited by
 * title and section:
 *   [IDLM] "Introspective Diffusion Language Models" (project page):
 *          "Inference & ISD", "Serving (SGLang)", "Lossless R-ISD",
 *          "Training", "How do DLMs perform as they approach compute-bound?".
 *   [GN]   "I-DLM - Icgozlemsel Difuzyon Dil Modelleri" (GeekNews summary):
 *          "I-DLM Yontemi", "Inference & ISD", "Speedup Factor Explorer".
 *
 * Row layout of a request inside a step (rows are consecutive, the request's
 * first row is qo_indptr[c]):
 *   FULL  (mode 1): N clean rows [anchor, d_1 .. d_{N-1}] then N-1 MASK rows
 *                   (2N-1 rows; [IDLM] "How do DLMs perform ...": 2N-1
 *                   queries per forward).  Clean row i-1 verifies draft d_i;
 *                   clean row N-1 gives the bonus slot; MASK row k proposes
 *                   the next step's draft k.
 *   FRESH (mode 0): 1 clean row [anchor] then N-1 MASK rows (N rows), used
 *                   after a rejection.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, unless the
 *     comment says otherwise.  The library allocates nothing and keeps no
 *     state between calls.
 *   - Tensors are dense row-major ("C order") with the shapes given.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream).  They launch kernels and nothing else.
 *   - The return value reports what the host can check before launching
 *     (argument ranges, workspace size, unsupported shapes) and launch
 *     errors.  On a non-OK return nothing was launched, except for
 *     IDLM_ERR_CUDA, which reports a failed launch.
 *   - Errors that depend on device data (a page id outside the pool, a token
 *     id outside the vocabulary, a row layout that disagrees with `mode`, a
 *     wait that ran out) are written to the caller's device word `status`
 *     (int32, one per call, set to 0 by the caller beforehand): the first
 *     error code wins (atomicCAS).  Kernels never trap.  Outputs of a call
 *     that set `status` are unspecified, but no memory outside the buffers
 *     passed in is written.
 *   - `workspace` is caller-owned device scratch of at least the size the
 *     matching *_workspace_size() query returns, 256-byte aligned.  Its
 *     contents need no initialisation.  A workspace must not be shared by
 *     calls that may run concurrently.
 */
#ifndef IDLM_H
#define IDLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IDLM_OK = 0,
  IDLM_ERR_INVALID_ARG = 1,   /* a pointer, size or enum out of range */
  IDLM_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype, D, group) */
  IDLM_ERR_WORKSPACE = 3,     /* workspace missing or too small */
  IDLM_ERR_CUDA = 4           /* a CUDA runtime call or launch failed */
} idlm_status;

/* Codes written to the device `status` word. */
#define IDLM_DEV_OK 0
#define IDLM_DEV_BAD_PAGE 1     /* page id outside [0, num_pages) */
#define IDLM_DEV_BAD_TOKEN 2    /* draft token outside [0, V) */
#define IDLM_DEV_BAD_LAYOUT 3   /* rows of a request disagree with its mode */
#define IDLM_DEV_SLOT_OVERFLOW 4 /* a slot beyond the request's page table */
#define IDLM_DEV_TIMEOUT 5      /* a bounded wait inside a kernel ran out */

/* Element types. */
#define IDLM_F32 0
#define IDLM_BF16 1

/* Request modes and proposal modes. */
#define IDLM_MODE_FRESH 0
#define IDLM_MODE_FULL 1
#define IDLM_PROPOSE_ARGMAX 0
#define IDLM_PROPOSE_SAMPLE 1

/* Library version (major * 10000 + minor * 100 + patch). */
int idlm_version(void);

/* Static text for a status code. */
const char* idlm_status_string(int status);

/* ------------------------------------------------------------------------
 * a2. Paged strict-causal GQA attention of the step rows.
 *
 * [IDLM] "Training" (strict causal masking across all positions) and
 * "Serving (SGLang)" (paged KV cache, paged-only attention kernel).
 * Row r of request c sits at position L_c + r (L_c = seq_lens[c]) and
 * attends to the committed slots 0 .. L_c-1, read through
 * page_table[c][slot / page_size] at offset slot % page_size, and to this
 * step's new K/V rows 0 .. r of the same request.  Query head h reads KV head
 * h / (Hq / Hkv).  out = softmax(q k^T * sm_scale) v, accumulated in fp32.
 *
 *   q          [T, Hq, D]              this step's query rows
 *   k_new      [T, Hkv, D]             this step's keys (not yet cached)
 *   v_new      [T, Hkv, D]
 *   k_cache    [num_pages, Hkv, page_size, D]
 *   v_cache    [num_pages, Hkv, page_size, D]
 *   page_table [C, max_pages] int32   physical page of each logical page
 *   seq_lens   [C] int32               committed length L_c (read only)
 *   qo_indptr  [C+1] int32             first row of each request; qo_indptr[C] = T
 *   out        [T, Hq, D]              written for every row
 *   dtype      IDLM_BF16 or IDLM_F32 for q, k_*, v_*, caches and out
 *   max_rows   upper bound on qo_indptr[c+1]-qo_indptr[c] (e.g. 2N-1)
 * Fast path: dtype BF16, D = 128, page_size = 16, (Hq/Hkv) * max_rows <= 64
 * (a TMA-fed tensor-core kernel, then a small kernel that merges the KV
 * ranges of a (request, KV head) split between CTAs, launched as its
 * programmatic dependent); other shapes run a simple CUDA-core kernel
 * (any page_size, D a multiple of 32 up to 256).  Device errors: BAD_PAGE,
 * BAD_LAYOUT (a request with more than max_rows rows), TIMEOUT.
 * Workspace: idlm_isd_attention_workspace_size(); it depends on the current
 * device's SM count.
 * ---------------------------------------------------------------------- */
size_t idlm_isd_attention_workspace_size(int C, int Hq, int Hkv, int D,
                                         int page_size, int max_rows, int dtype);

idlm_status idlm_isd_attention(
    const void* q, const void* k_new, const void* v_new,
    const void* k_cache, const void* v_cache,
    const int32_t* page_table, int max_pages,
    const int32_t* seq_lens, const int32_t* qo_indptr,
    int C, int T, int Hq, int Hkv, int D, int page_size, int num_pages,
    int max_rows, float sm_scale, int dtype, void* out,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * a3. Gated-LoRA projection (R-ISD).
 *
 * [IDLM] "Lossless R-ISD": a LoRA adapter is applied only at MASK positions;
 * verify (clean) positions use the base weights alone, so their outputs equal
 * the base model's bit for bit; the pages' adapter has rank 128.  [IDLM]
 * speedup panel: R-ISD overhead 1.12.
 *
 *   Y = X W^T + g_row * lora_scale * (X A^T) B^T,   g_row = row_gate[m] != 0
 *
 *   x          [M, K]  bf16   token rows of the step
 *   w          [N, K]  bf16   base weight (row n gives output column n)
 *   lora_a     [r, K]  bf16
 *   lora_b     [N, r]  bf16
 *   row_gate   [M]     uint8  1 at MASK rows, 0 at clean rows
 *   y          [M, N]  bf16   written for every row
 * fp32 accumulation on the tensor cores (tcgen05); the adapter enters the
 * same accumulation as one (r <= 64) or two (r <= 128) more K steps, so rows
 * with row_gate = 0 come out bit-identical to the projection with
 * lora_b = 0.  Requirements: K % 8 == 0, r % 8 == 0, 0 <= r <= 128 (r = 0:
 * no adapter; lora_a, lora_b and row_gate may then be NULL), 16-byte aligned
 * x, w, lora_a, lora_b; any M (token rows run in slices of 448).
 * Workspace: idlm_gated_lora_workspace_size() bytes, 256-byte aligned (the
 * adapter operands T = g s X A^T and, where r % 64 != 0, B padded to 64
 * columns; fp32 partial tiles, two slots per SM); its contents need no
 * initialisation, and one workspace must not be used by two calls at once.
 * The size depends on the current device.
 * The call launches per slice of 448 token rows: the adapter kernel
 * (T = g s X A^T), the GEMM (a persistent grid of at most one CTA per SM
 * holding whole weight-row tiles and an even share of the K steps of the
 * tiles left over) and, when a tile's K sum was split, a fix-up kernel that
 * adds its fp32 partial tiles in a fixed order.  No CTA waits for another,
 * and results are reproducible on a given device.
 * The environment variable IDLM_LORA_GRID, if set, fixes the grid size
 * (capped at the SMs).  Device errors: TIMEOUT.  Failure-detection test
 * switch: with IDLM_TEST_STALL=1 in the environment, every GEMM CTA first
 * waits (for 20 ms) on a barrier that nothing arrives on, so the call ends
 * with TIMEOUT in `status` and Y unspecified; it still returns normally and
 * the CUDA context stays usable.
 * ---------------------------------------------------------------------- */
size_t idlm_gated_lora_workspace_size(int M, int K, int N, int r);

idlm_status idlm_gated_lora(
    const void* x, const void* w, const void* lora_a, const void* lora_b,
    const uint8_t* row_gate, float lora_scale, int M, int K, int N, int r, void* y,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* Several gated-LoRA projections that share the input X (q|k|v, gate|up) as
 * one call: the weights are stacked along N, group g owning weight rows
 * [sum_{h<g} group_rows[h], sum_{h<=g} group_rows[h]) (group_rows is a HOST
 * array of ngroups entries, each a multiple of 128 except the last, summing
 * to N); lora_a stacks the groups' adapters, [ngroups * r, K]; lora_b is
 * [N, r], row n holding the B row of n's group.  Y = X W^T plus, for the
 * rows of group g, g_row * lora_scale * (X A_g^T) B_g^T.  1 <= ngroups <= 4;
 * otherwise as idlm_gated_lora, with its own workspace query. */
size_t idlm_gated_lora_grouped_workspace_size(int M, int K, int N, int r, int ngroups);

idlm_status idlm_gated_lora_grouped(
    const void* x, const void* w, const void* lora_a, const void* lora_b,
    const uint8_t* row_gate, float lora_scale, int M, int K, int N, int r,
    int ngroups, const int* group_rows, void* y,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * a4-a7. Accept: vocab pass, p/q acceptance, residual resample, bonus or
 * fresh draw, proposals and next state.
 *
 * [IDLM] "Inference & ISD" / [GN] "Inference & ISD": MASK positions propose
 * (q), clean positions verify (anchor p), a draft x passes with probability
 * min(1, p(x)/q(x)).  p and q are softmax(logits / temperature)
 * (temperature 0 = greedy one-hot argmax).  For a FULL request, draft i
 * (i = 1..N-1) passes when u_i < min(1, p_i(d_i)/q_i(d_i)), where p_i comes
 * from clean row i-1 and q_i from the previous step's MASK row that proposed
 * it; the first failure j ends the scan and its token is drawn from
 * normalize(max(0, p_j - q_j)) (p_j if that is all zero).  If all N-1 pass,
 * a bonus token is drawn from p of clean row N-1.  A FRESH request draws one
 * token from p of its row 0.  Draws are inverse-CDF in vocabulary order with
 * Philox4x64-10 uniforms (Salmon et al., SC'11): counter (step, c, purpose,
 * index/4), key (seed, 0), word index%4, u = top 24 bits * 2^-24; purpose 0:
 * u_i; purpose 1: word 0 bonus/fresh draw, word 1 residual draw; purpose 2:
 * SAMPLE-mode proposal of MASK row k (index k-1).  Proposals: argmax of each
 * MASK row (lowest index on ties) or a draw from its q (SAMPLE).
 *
 *   logits         [T, V] (dtype)          this step's output rows; T is the
 *                                          buffer's capacity: rows from
 *                                          qo_indptr[C] on are not read, so a
 *                                          fixed-shape loop may pass its
 *                                          largest row count every step
 *   qo_indptr      [C+1] int32
 *   mode           [C] uint8               IDLM_MODE_FULL / IDLM_MODE_FRESH
 *   drafts         [C, N-1] int32          read for FULL requests
 *   draft_q_stats  [C, N-1, 2] float       (m, S) of each draft's proposing
 *                                          row, as written to next_q_stats by
 *                                          the previous call
 *   prev_logits    [prev_rows, V] (dtype)  the previous step's logits
 *   prev_mask_row0 [C] int32               row of prev_logits that proposed
 *                                          draft 1 (draft i: row + i - 1), as
 *                                          written to next_mask_row0 before
 *   outputs (all [C] unless noted):
 *   n_accepted     int32    accepted drafts (0 for FRESH)
 *   out_tokens     [C, N] int32  emitted tokens: accepted drafts, then the
 *                           resampled / bonus / fresh token; -1 after them
 *   n_out          int32    n_accepted + 1
 *   n_commit       int32    rows to commit to the KV cache: 1 + n_accepted
 *                           (FULL) or 1 (FRESH)
 *   next_drafts    [C, N-1] int32  proposals if next_mode is FULL, else -1
 *   next_q_stats   [C, N-1, 2] float (m, S) = (max_v x_v/T,
 *                           sum_v exp(x_v/T - m)) of each MASK row
 *   next_mode      uint8    FULL if nothing was rejected, else FRESH
 *   next_mask_row0 int32    qo_indptr[c] + (number of clean rows)
 *   row_stats      [T, 2] float or NULL: (m, S) of every row in use
 *   dbg            [C, N-1, 4] float or NULL: (u_i, p_i(d_i), q_i(d_i),
 *                           ratio) per draft of FULL requests
 * Requirements: V % 8 == 0, 2 <= N <= 16, temperature >= 0.
 * Device errors: BAD_TOKEN, BAD_LAYOUT (rows of a request disagree with its
 * mode, qo_indptr leaves [0, T], or a draft's proposing row leaves
 * [0, prev_rows)).  The call launches three kernels and nothing else: a
 * streaming pass over the logits, a per-request decision kernel and a
 * residual kernel, the last two as programmatic dependents of the kernel
 * before them (plain stream order where the stream does not take that
 * attribute).  Workspace contents need no initialisation.
 * ---------------------------------------------------------------------- */
size_t idlm_isd_accept_workspace_size(int C, int T, int N, int V);

idlm_status idlm_isd_accept(
    const void* logits, int dtype, int V, const int32_t* qo_indptr,
    const uint8_t* mode, const int32_t* drafts, const float* draft_q_stats,
    const void* prev_logits, int prev_rows, const int32_t* prev_mask_row0,
    int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step,
    int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out, int32_t* n_commit,
    int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Accept + KV commit in one call ([IDLM] "Inference & ISD" and "Serving
 * (SGLang)": the kept rows of a step go to the paged KV cache).
 *
 * The same outputs as idlm_isd_accept followed by idlm_kv_commit with
 * n_commit from the accept (the cache, seq_lens_out and releasable_from as
 * idlm_kv_commit writes them).  The accept's decision kernel appends each
 * request's commit to its residual kernel's work list, so the copies run
 * beside the residual and draw work and the call launches the accept's three
 * kernels and nothing else.
 *   logits .. dbg    as for idlm_isd_accept
 *   k_cache .. releasable_from, Hkv, D, page_size, num_pages, kv_dtype
 *                    as for idlm_kv_commit (k_new / v_new: the step's new
 *                    keys and values, rows as qo_indptr lays them out)
 *   workspace        idlm_isd_accept_workspace_size(C, T, N, V) bytes
 * Device errors: those of both calls.
 * ---------------------------------------------------------------------- */
idlm_status idlm_isd_accept_commit(
    const void* logits, int dtype, int V, const int32_t* qo_indptr,
    const uint8_t* mode, const int32_t* drafts, const float* draft_q_stats,
    const void* prev_logits, int prev_rows, const int32_t* prev_mask_row0,
    int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step,
    int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out, int32_t* n_commit,
    int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg,
    void* k_cache, void* v_cache, const int32_t* page_table, int max_pages,
    const int32_t* seq_lens_in, int32_t* seq_lens_out, const void* k_new,
    const void* v_new, int Hkv, int D, int page_size, int num_pages, int kv_dtype,
    int32_t* releasable_from, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Fused LM head + accept ([IDLM] "Inference & ISD": p and q both come from
 * the one forward pass, whose last product is the LM head).
 *
 * logits = hidden W^T, then the accept step of idlm_isd_accept on them, in
 * one call.  The GEMM (tcgen05, the gated-LoRA GEMM without an adapter)
 * writes the logits once and, in the same epilogue, the softmax statistics
 * of every logits row per 128-entry tile of the vocabulary, taken from the
 * bf16 values it stores; a merge kernel turns them into the accept's
 * per-chunk records and the accept runs without its own pass over the
 * logits.  The draws (one chunk per inverse-CDF search, the two rows of a
 * rejected draft's residual) read the logits written here.
 *
 *   hidden   [T, H] bf16, 16-byte aligned: the step's rows (the final hidden
 *            states after the model's last norm)
 *   w_vocab  [V, H] bf16, 16-byte aligned: the LM head's weights
 *   logits   [T, V] bf16 out (16-byte aligned), the same logits that
 *            idlm_isd_accept would take
 *   the remaining arguments as for idlm_isd_accept with dtype = IDLM_BF16;
 *   prev_logits is the previous step's `logits` buffer.
 * Requirements: H % 8 == 0, V % 8 == 0, 2 <= N <= 16, temperature >= 0.
 * Launches: the GEMM and (where its plan splits tiles) its fix-up, the merge
 * kernel, then the accept's three kernels.  Workspace contents need no
 * initialisation.
 * ---------------------------------------------------------------------- */
size_t idlm_lm_head_accept_workspace_size(int C, int T, int N, int H, int V);

idlm_status idlm_lm_head_accept(
    const void* hidden, const void* w_vocab, int H, void* logits, int V,
    const int32_t* qo_indptr, const uint8_t* mode, const int32_t* drafts,
    const float* draft_q_stats, const void* prev_logits, int prev_rows,
    const int32_t* prev_mask_row0, int C, int T, int N, float temperature,
    int proposal_mode, uint64_t seed, uint64_t step,
    int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out, int32_t* n_commit,
    int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg,
    void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free accept.  The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory -- a plugin whose
 * host owns all GPU memory and offers no scratch, or a decode loop held to a
 * fixed memory budget that may not call the allocator while it runs.
 *
 * Same arguments and results as idlm_isd_accept without the workspace pair.
 * The scratch is one 4 MiB array compiled into the library (a static
 * __device__ array), which every GPU that loads the library keeps until the
 * process exits.  The call allocates nothing and frees nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is cached per CUDA context
 *     (keyed on the context's unique id): after cudaDeviceReset, or under
 *     another context on the same device, the next call looks it up again,
 *     so make that call, too, outside a stream capture.
 *   - Returns IDLM_ERR_WORKSPACE, launching nothing, when the call needs more
 *     than 4 MiB, i.e. when idlm_isd_accept_workspace_size(C, T, N, V)
 *     exceeds 4194304 bytes.
 *   - Every call uses the same array and it keeps the last call's contents;
 *     each call clears the counters it relies on before its kernels run.
 *     Calls that can overlap on the GPU (two streams, two host threads) race
 *     on the array and corrupt each other's results: serialise them.
 * ---------------------------------------------------------------------- */
idlm_status idlm_isd_accept_noalloc(
    const void* logits, int dtype, int V, const int32_t* qo_indptr,
    const uint8_t* mode, const int32_t* drafts, const float* draft_q_stats,
    const void* prev_logits, int prev_rows, const int32_t* prev_mask_row0,
    int C, int T, int N, float temperature, int proposal_mode,
    uint64_t seed, uint64_t step,
    int32_t* n_accepted, int32_t* out_tokens, int32_t* n_out, int32_t* n_commit,
    int32_t* next_drafts, float* next_q_stats, uint8_t* next_mode,
    int32_t* next_mask_row0, float* row_stats, float* dbg,
    int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * a8. KV commit / rollback.
 *
 * [IDLM] "Serving (SGLang)": paged KV cache.  Rows 0 .. n_commit[c]-1 of
 * request c (the anchor and its accepted drafts, or a FRESH request's one
 * clean row) are copied from k_new / v_new to logical slots
 * L_c .. L_c + n_commit[c] - 1 of the cache.  Rejected drafts and MASK rows
 * are never written (rollback).  seq_lens_out[c] = L_c + n_commit[c];
 * releasable_from[c] = ceil(seq_lens_out[c] / page_size): page-table entries
 * from that index on hold no committed slot and may return to the caller's
 * pool.  The caller allocates pages for the slots before the call.
 *
 *   k_cache, v_cache [num_pages, Hkv, page_size, D]   (dtype) in/out
 *   page_table      [C, max_pages] int32
 *   seq_lens_in     [C] int32; seq_lens_out [C] int32 (may be the same buffer)
 *   k_new, v_new    [T, Hkv, D] (dtype); qo_indptr [C+1] int32 (within [0, T])
 *   n_commit        [C] int32 (as written by idlm_isd_accept)
 *   releasable_from [C] int32 or NULL
 * A request whose commit would touch a page id outside the pool, a slot
 * beyond its page-table row, or more rows than it has, sets status
 * (BAD_PAGE, SLOT_OVERFLOW, BAD_LAYOUT) and writes nothing, its length
 * included.  Requirements: D * element size a multiple of 16 bytes.
 * ---------------------------------------------------------------------- */
idlm_status idlm_kv_commit(
    void* k_cache, void* v_cache, const int32_t* page_table, int max_pages,
    const int32_t* seq_lens_in, int32_t* seq_lens_out,
    const void* k_new, const void* v_new, const int32_t* qo_indptr,
    const int32_t* n_commit, int C, int T, int Hkv, int D, int page_size,
    int num_pages, int dtype, int32_t* releasable_from, int32_t* status,
    void* stream);

/* ------------------------------------------------------------------------
 * One R-ISD decoder layer over the step's rows.
 *
 * [IDLM] "Lossless R-ISD": LoRA adapters (rank 128 on the pages) act only at
 * MASK positions, so clean positions reproduce the base model; "Training":
 * strict causal attention.  The pages do not spell the layer out; this is
 * the pre-norm layout of the Qwen3-style base models they convert (no rotary
 * embedding or QK-norm inside the step, as for idlm_isd_attention):
 *   n1 = RMSNorm(x); [q|k|v] = n1 Wqkv^T (+ gated LoRA per group);
 *   a = attention(q, k, v) over the paged cache (idlm_isd_attention);
 *   h = x + a Wo^T (+ gated LoRA); n2 = RMSNorm(h);
 *   [g|u] = n2 Wgu^T (+ gated LoRA per group);
 *   out = h + (silu(g) * u) Wd^T (+ gated LoRA)
 * with RMSNorm(v) = v / sqrt(mean(v^2) + rms_eps) * weight.  Activations
 * are stored in bf16 between the kernels (fp32 accumulation and elementwise
 * arithmetic).  Because the step's rows are laid out [clean..., MASK...] per
 * request and attention is causal, clean rows never see a MASK row, so with
 * any adapters their outputs equal those of the layer with rank 0 bit for
 * bit.
 * ---------------------------------------------------------------------- */
typedef struct {
  int hidden, ffn, n_heads, n_kv_heads, head_dim;
  int rank;                /* adapter rank, 0 (no adapters) or 8 .. 128, % 8 */
  float lora_scale, rms_eps;
  const void* w_qkv;       /* [(Hq + 2 Hkv) D, hidden] bf16: q rows, k rows, v rows */
  const void* a_qkv;       /* [3 rank, hidden]: the q, k, v adapters' A stacked */
  const void* b_qkv;       /* [(Hq + 2 Hkv) D, rank] */
  const void* w_o;         /* [hidden, Hq D] */
  const void* a_o;         /* [rank, Hq D] */
  const void* b_o;         /* [hidden, rank] */
  const void* w_gu;        /* [2 ffn, hidden]: gate rows, then up rows */
  const void* a_gu;        /* [2 rank, hidden] */
  const void* b_gu;        /* [2 ffn, rank] */
  const void* w_down;      /* [hidden, ffn] */
  const void* a_down;      /* [rank, ffn] */
  const void* b_down;      /* [hidden, rank] */
  const void* norm1;       /* [hidden] bf16, or NULL for weight 1 */
  const void* norm2;       /* [hidden] bf16, or NULL */
} idlm_layer_weights;

/* Workspace of idlm_risd_layer (the activations, one gated-LoRA workspace
 * and one attention workspace); 0 for an unsupported shape.  Shapes:
 * hidden % 8 == 0, ffn % 128 == 0, Hq D and Hkv D multiples of 128. */
size_t idlm_risd_layer_workspace_size(const idlm_layer_weights* weights, int M, int C,
                                      int page_size, int max_rows);

/*   x, out        [M, hidden] bf16 (16-byte aligned), M = qo_indptr[C]
 *   row_gate      [M] uint8  1 at MASK rows
 *   k_cache .. max_rows   the paged cache and layout, as for
 *                 idlm_isd_attention (the layer does not write the cache)
 *   k_new_out, v_new_out  [M, Hkv, D] bf16 or NULL: the step's keys and
 *                 values, for idlm_kv_commit afterwards
 * Launches the kernels of the layer in stream order (about 14 launches);
 * device errors as for idlm_isd_attention and idlm_gated_lora. */
idlm_status idlm_risd_layer(
    const idlm_layer_weights* weights, const void* x, void* out, int M,
    const uint8_t* row_gate, const void* k_cache, const void* v_cache,
    const int32_t* page_table, int max_pages, const int32_t* seq_lens,
    const int32_t* qo_indptr, int C, int page_size, int num_pages, int max_rows,
    void* k_new_out, void* v_new_out, void* workspace, size_t workspace_bytes,
    int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Stationary-batch decode loop: the hand-off between two steps.
 *
 * [IDLM] "Serving (SGLang)": the batch keeps its shape from step to step
 * (stationary-batch decode loop) and the step is replayed from a CUDA graph;
 * the abstract names a stationary-batch scheduler.  From this step's accept
 * and commit results, writes the next step's row layout and row inputs:
 *   FULL  (next_mode 1): rows [anchor, d_1 .. d_{N-1}, MASK x (N-1)]
 *   FRESH (next_mode 0): rows [anchor, MASK x (N-1)]
 * at positions L .. L + rows - 1, where L = seq_lens[c] (after the commit),
 * the anchor is the last token the step emitted (out_tokens[c][n_out-1], not
 * yet in the cache) and d_k = next_drafts[c][k-1].
 *
 *   mode          [C] uint8 or NULL   this step's modes (counters only)
 *   next_mode, out_tokens [C, N], n_out, n_accepted (or NULL), next_drafts
 *                 [C, N-1]            as written by idlm_isd_accept
 *   seq_lens      [C] int32           committed lengths after idlm_kv_commit
 *   qo_indptr     [C+1] int32         out: the next step's row layout
 *   row_req, row_pos, row_token [T] int32   out: request, absolute position
 *                 and input token of each row (-1 at MASK rows); rows from
 *                 qo_indptr[C] to T get request 0, position 0, token -2
 *   counters      [4, C] int32 or NULL   in/out, when count != 0: tokens
 *                 emitted, forwards, accepted drafts, drafts tested
 *   history       [C, hist_cap] int32 or NULL   in/out, when count != 0:
 *                 emitted tokens appended at hist_len[c] (dropped past
 *                 hist_cap); hist_len [C] int32 in/out
 *   count         0 for a loop's first layout (nothing to count), else 1
 * Requirements: 2 <= N <= 16, T >= C (2N - 1).  Device errors: BAD_LAYOUT
 * (n_out outside [1, N], a negative length).  One kernel launch.
 * ---------------------------------------------------------------------- */
idlm_status idlm_isd_advance(
    int C, int N, int T, const uint8_t* mode, const uint8_t* next_mode,
    const int32_t* out_tokens, const int32_t* n_out, const int32_t* n_accepted,
    const int32_t* next_drafts, const int32_t* seq_lens, int32_t* qo_indptr,
    int32_t* row_req, int32_t* row_pos, int32_t* row_token, int32_t* counters,
    int32_t* history, int hist_cap, int32_t* hist_len, int count,
    int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Synthetic logit rows: the seeded workloads' stand-in for the model's
 * forward pass in a decode loop (not part of the ISD step).
 *
 * Row i (i < qo_indptr[C]) of request c = row_req[i] at position
 * row_pos[i] predicts slot s = row_pos[i] + 1 ([IDLM] "Training": logit
 * shift).  A clean row (row_token[i] >= 0) holds z(c, s); a MASK row holds
 * z(c, s) + e(c, s, step) scaled per request, so a draft proposed at one step
 * is verified against z(c, s) at the next.  Each value is an Irwin-Hall sum
 * of the eight 16-bit halves of one Philox4x32-10 output (Salmon et al.,
 * SC'11; counter (v, s, c, d), key (seed, 0x1D1A7E5D), d = 0 for z and
 * 1 + step for e), centred (minus 4 * 65535), converted exactly to fp32 and
 * multiplied by scale_z (z) or scale_e[c] (e), the sum rounded to nearest in
 * fp32 and then to nearest-even in bf16.  A CPU implementation of this
 * definition reproduces every bit.
 *
 *   logits    [T, V] bf16, 16-byte aligned, V % 8 == 0 (rows in use written)
 *   qo_indptr [C+1], row_req, row_pos, row_token [T] int32 (as
 *             idlm_isd_advance writes them)
 *   scale_e   [C] float
 *   step      < 2^32 - 1
 * One kernel launch.
 * ---------------------------------------------------------------------- */
idlm_status idlm_synth_logits(
    void* logits, int C, int T, int V, const int32_t* qo_indptr,
    const int32_t* row_req, const int32_t* row_pos, const int32_t* row_token,
    float scale_z, const float* scale_e, uint32_t seed, uint32_t step,
    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* IDLM_H */
