"""ctypes binding of libidlm.so: argument marshalling only.

Each function has the name of the C entry point it calls, takes torch tensors
(device memory) and plain numbers, reads the sizes off the tensors, and passes
raw pointers and the current CUDA stream to the library.  No arithmetic of the
ISD step happens here.  A non-OK return raises ``IDLMError``; device-side
errors land in the caller's ``status`` tensor.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libidlm.so")

IDLM_F32 = 0
IDLM_BF16 = 1
MODE_FRESH = 0
MODE_FULL = 1
PROPOSE_ARGMAX = 0
PROPOSE_SAMPLE = 1

DEV_STATUS = {0: "ok", 1: "bad page", 2: "bad token", 3: "bad layout", 4: "slot overflow",
              5: "timeout"}

_lib = None


class IDLMError(RuntimeError):
    pass


class LayerWeights(ctypes.Structure):
    """idlm_layer_weights (include/idlm.h)."""
    _fields_ = [("hidden", ctypes.c_int), ("ffn", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("rank", ctypes.c_int),
                ("lora_scale", ctypes.c_float), ("rms_eps", ctypes.c_float)] + [
        (n, ctypes.c_void_p) for n in ("w_qkv", "a_qkv", "b_qkv", "w_o", "a_o", "b_o", "w_gu",
                                       "a_gu", "b_gu", "w_down", "a_down", "b_down", "norm1",
                                       "norm2")]


def lib():
    """Load libidlm.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise IDLMError(f"{LIB_PATH} is missing: run python -m "
                            "speculative_verify_accept_step_b300.build")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, u64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                 ctypes.c_float, ctypes.c_size_t)
        L.idlm_version.restype = i32
        L.idlm_status_string.restype = ctypes.c_char_p
        L.idlm_status_string.argtypes = [i32]
        L.idlm_isd_attention_workspace_size.restype = sz
        L.idlm_isd_attention_workspace_size.argtypes = [i32] * 7
        L.idlm_isd_attention.restype = i32
        L.idlm_isd_attention.argtypes = (
            [vp] * 6 + [i32] + [vp, vp] + [i32] * 8 + [f32, i32, vp, vp, sz, vp, vp])
        L.idlm_isd_accept_workspace_size.restype = sz
        L.idlm_isd_accept_workspace_size.argtypes = [i32] * 4
        L.idlm_isd_accept.restype = i32
        L.idlm_isd_accept.argtypes = (
            [vp, i32, i32] + [vp] * 5 + [i32, vp] + [i32, i32, i32, f32, i32, u64, u64]
            + [vp] * 10
            + [vp, sz, vp, vp])
        L.idlm_lm_head_accept_workspace_size.restype = sz
        L.idlm_lm_head_accept_workspace_size.argtypes = [i32, i32, i32, i32, i32]
        L.idlm_lm_head_accept.restype = i32
        L.idlm_lm_head_accept.argtypes = (
            [vp, vp, i32, vp, i32] + [vp] * 4 + [vp, i32, vp] + [i32, i32, i32, f32, i32, u64, u64]
            + [vp] * 10
            + [vp, sz, vp, vp])
        L.idlm_isd_accept_noalloc.restype = i32
        L.idlm_isd_accept_noalloc.argtypes = (
            [vp, i32, i32] + [vp] * 5 + [i32, vp] + [i32, i32, i32, f32, i32, u64, u64]
            + [vp] * 10 + [vp, vp])
        L.idlm_gated_lora_workspace_size.restype = sz
        L.idlm_gated_lora_workspace_size.argtypes = [i32] * 4
        L.idlm_gated_lora.restype = i32
        L.idlm_gated_lora.argtypes = [vp] * 5 + [f32] + [i32] * 4 + [vp, vp, sz, vp, vp]
        L.idlm_gated_lora_grouped_workspace_size.restype = sz
        L.idlm_gated_lora_grouped_workspace_size.argtypes = [i32] * 5
        L.idlm_gated_lora_grouped.restype = i32
        L.idlm_gated_lora_grouped.argtypes = ([vp] * 5 + [f32] + [i32] * 5
                                              + [ctypes.POINTER(ctypes.c_int), vp, vp, sz, vp, vp])
        L.idlm_synth_logits.restype = i32
        L.idlm_synth_logits.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, f32, vp,
                                        ctypes.c_uint32, ctypes.c_uint32, vp]
        L.idlm_isd_advance.restype = i32
        L.idlm_isd_advance.argtypes = ([i32, i32, i32] + [vp] * 11 + [vp, vp, i32, vp, i32, vp,
                                                                      vp])
        L.idlm_risd_layer_workspace_size.restype = sz
        L.idlm_risd_layer_workspace_size.argtypes = [ctypes.POINTER(LayerWeights)] + [i32] * 4
        L.idlm_risd_layer.restype = i32
        L.idlm_risd_layer.argtypes = ([ctypes.POINTER(LayerWeights), vp, vp, i32, vp, vp, vp, vp,
                                       i32, vp, vp] + [i32] * 4 + [vp, vp, vp, sz, vp, vp])
        L.idlm_kv_commit.restype = i32
        L.idlm_kv_commit.argtypes = ([vp, vp, vp, i32, vp, vp, vp, vp, vp, vp] + [i32] * 7
                                     + [vp, vp, vp])
        L.idlm_isd_accept_commit.restype = i32
        L.idlm_isd_accept_commit.argtypes = (
            [vp, i32, i32] + [vp] * 5 + [i32, vp] + [i32, i32, i32, f32, i32, u64, u64]
            + [vp] * 10
            + [vp, vp, vp, i32, vp, vp, vp, vp] + [i32] * 5 + [vp]
            + [vp, sz, vp, vp])
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return IDLM_BF16
    if t.dtype == torch.float32:
        return IDLM_F32
    raise IDLMError(f"unsupported dtype {t.dtype}")


def _check(rc, what):
    if rc != 0:
        raise IDLMError(f"{what}: {lib().idlm_status_string(rc).decode()} ({rc})")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise IDLMError("tensors passed to libidlm must be contiguous")


def version():
    return lib().idlm_version()


# ------------------------------------------------------------------ attention

def idlm_isd_attention_workspace_size(C, Hq, Hkv, D, page_size, max_rows, dtype):
    return int(lib().idlm_isd_attention_workspace_size(C, Hq, Hkv, D, page_size, max_rows, dtype))


def idlm_isd_attention(q, k_new, v_new, k_cache, v_cache, page_table, seq_lens, qo_indptr,
                       out, workspace, status, max_rows, sm_scale, stream=None):
    _contig(q, k_new, v_new, k_cache, v_cache, page_table, seq_lens, qo_indptr, out, workspace)
    T, Hq, D = q.shape
    num_pages, Hkv, page_size, _ = k_cache.shape
    C, max_pages = page_table.shape
    rc = lib().idlm_isd_attention(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(page_table),
        max_pages, _ptr(seq_lens), _ptr(qo_indptr), C, T, Hq, Hkv, D, page_size, num_pages,
        max_rows, float(sm_scale), _dtype(q), _ptr(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_isd_attention")


# --------------------------------------------------------------------- accept

def idlm_isd_accept_workspace_size(C, T, N, V):
    return int(lib().idlm_isd_accept_workspace_size(C, T, N, V))


def idlm_isd_accept(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
                    prev_mask_row0, N, temperature, proposal_mode, seed, step,
                    n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats,
                    next_mode, next_mask_row0, workspace, status, row_stats=None, dbg=None,
                    stream=None):
    _contig(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits, prev_mask_row0,
            n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats, next_mode,
            next_mask_row0, workspace, row_stats, dbg)
    T, V = logits.shape
    C = mode.shape[0]
    rc = lib().idlm_isd_accept(
        _ptr(logits), _dtype(logits), V, _ptr(qo_indptr), _ptr(mode), _ptr(drafts),
        _ptr(draft_q_stats), _ptr(prev_logits), prev_logits.shape[0], _ptr(prev_mask_row0),
        C, T, N,
        float(temperature), int(proposal_mode), int(seed), int(step), _ptr(n_accepted),
        _ptr(out_tokens), _ptr(n_out), _ptr(n_commit), _ptr(next_drafts), _ptr(next_q_stats),
        _ptr(next_mode), _ptr(next_mask_row0), _ptr(row_stats), _ptr(dbg), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    _check(rc, "idlm_isd_accept")


def idlm_lm_head_accept_workspace_size(C, T, N, H, V):
    return lib().idlm_lm_head_accept_workspace_size(C, T, N, H, V)


def idlm_lm_head_accept(hidden, w_vocab, logits, qo_indptr, mode, drafts, draft_q_stats,
                        prev_logits, prev_mask_row0, N, temperature, proposal_mode, seed, step,
                        n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats,
                        next_mode, next_mask_row0, workspace, status, row_stats=None, dbg=None,
                        stream=None):
    """logits = hidden @ w_vocab^T (written to `logits`, bf16 [T, V]), then the
    accept step on them, with the vocabulary statistics taken in the GEMM's
    epilogue instead of a separate pass over the logits."""
    _contig(hidden, w_vocab, logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
            prev_mask_row0, n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats,
            next_mode, next_mask_row0, workspace, row_stats, dbg)
    T, H = hidden.shape
    V = w_vocab.shape[0]
    C = mode.shape[0]
    rc = lib().idlm_lm_head_accept(
        _ptr(hidden), _ptr(w_vocab), H, _ptr(logits), V, _ptr(qo_indptr), _ptr(mode),
        _ptr(drafts), _ptr(draft_q_stats), _ptr(prev_logits), prev_logits.shape[0],
        _ptr(prev_mask_row0), C, T, N, float(temperature), int(proposal_mode), int(seed),
        int(step), _ptr(n_accepted), _ptr(out_tokens), _ptr(n_out), _ptr(n_commit),
        _ptr(next_drafts), _ptr(next_q_stats), _ptr(next_mode), _ptr(next_mask_row0),
        _ptr(row_stats), _ptr(dbg), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_lm_head_accept")


def idlm_isd_accept_noalloc(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
                            prev_mask_row0, N, temperature, proposal_mode, seed, step,
                            n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats,
                            next_mode, next_mask_row0, status, row_stats=None, dbg=None,
                            stream=None):
    """idlm_isd_accept without a workspace: the library's fixed 4 MiB scratch
    array is used instead, so the call allocates nothing.  Calls that may
    overlap on the GPU share that array and must be serialised."""
    _contig(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits, prev_mask_row0,
            n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats, next_mode,
            next_mask_row0, row_stats, dbg)
    T, V = logits.shape
    C = mode.shape[0]
    rc = lib().idlm_isd_accept_noalloc(
        _ptr(logits), _dtype(logits), V, _ptr(qo_indptr), _ptr(mode), _ptr(drafts),
        _ptr(draft_q_stats), _ptr(prev_logits), prev_logits.shape[0], _ptr(prev_mask_row0),
        C, T, N, float(temperature), int(proposal_mode), int(seed), int(step),
        _ptr(n_accepted), _ptr(out_tokens), _ptr(n_out), _ptr(n_commit), _ptr(next_drafts),
        _ptr(next_q_stats), _ptr(next_mode), _ptr(next_mask_row0), _ptr(row_stats), _ptr(dbg),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_isd_accept_noalloc")


# ----------------------------------------------------------------- gated LoRA

def idlm_gated_lora_workspace_size(M, K, N, r):
    return int(lib().idlm_gated_lora_workspace_size(M, K, N, r))


def idlm_gated_lora(x, w, lora_a, lora_b, row_gate, lora_scale, y, workspace, status,
                    stream=None):
    _contig(x, w, lora_a, lora_b, row_gate, y, workspace)
    M, K = x.shape
    N = w.shape[0]
    r = lora_a.shape[0]
    rc = lib().idlm_gated_lora(
        _ptr(x), _ptr(w), _ptr(lora_a), _ptr(lora_b), _ptr(row_gate), float(lora_scale), M, K,
        N, r, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_gated_lora")


def idlm_gated_lora_grouped_workspace_size(M, K, N, r, ngroups):
    return int(lib().idlm_gated_lora_grouped_workspace_size(M, K, N, r, ngroups))


def idlm_gated_lora_grouped(x, w, lora_a, lora_b, row_gate, lora_scale, group_rows, y, workspace,
                            status, stream=None):
    """group_rows: the weight rows of each group (a host list of ints)."""
    _contig(x, w, lora_a, lora_b, row_gate, y, workspace)
    M, K = x.shape
    N = w.shape[0]
    ng = len(group_rows)
    r = lora_a.shape[0] // ng
    rows = (ctypes.c_int * ng)(*[int(v) for v in group_rows])
    rc = lib().idlm_gated_lora_grouped(
        _ptr(x), _ptr(w), _ptr(lora_a), _ptr(lora_b), _ptr(row_gate), float(lora_scale), M, K,
        N, r, ng, rows, _ptr(y), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_gated_lora_grouped")


# --------------------------------------------------------------------- commit

def idlm_kv_commit(k_cache, v_cache, page_table, seq_lens_in, seq_lens_out, k_new, v_new,
                   qo_indptr, n_commit, status, releasable_from=None, stream=None):
    _contig(k_cache, v_cache, page_table, seq_lens_in, seq_lens_out, k_new, v_new, qo_indptr,
            n_commit, releasable_from)
    num_pages, Hkv, page_size, D = k_cache.shape
    C, max_pages = page_table.shape
    rc = lib().idlm_kv_commit(
        _ptr(k_cache), _ptr(v_cache), _ptr(page_table), max_pages, _ptr(seq_lens_in),
        _ptr(seq_lens_out), _ptr(k_new), _ptr(v_new), _ptr(qo_indptr), _ptr(n_commit), C,
        k_new.shape[0], Hkv,
        D, page_size, num_pages, _dtype(k_cache), _ptr(releasable_from), _ptr(status),
        _stream(stream))
    _check(rc, "idlm_kv_commit")


def idlm_isd_accept_commit(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits,
                           prev_mask_row0, N, temperature, proposal_mode, seed, step,
                           n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats,
                           next_mode, next_mask_row0, k_cache, v_cache, page_table, seq_lens_in,
                           seq_lens_out, k_new, v_new, workspace, status, row_stats=None,
                           dbg=None, releasable_from=None, stream=None):
    """idlm_isd_accept, then the KV commit of the kept rows, in one call (the
    commits run as work items of the accept's residual kernel)."""
    _contig(logits, qo_indptr, mode, drafts, draft_q_stats, prev_logits, prev_mask_row0,
            n_accepted, out_tokens, n_out, n_commit, next_drafts, next_q_stats, next_mode,
            next_mask_row0, workspace, row_stats, dbg, k_cache, v_cache, page_table,
            seq_lens_in, seq_lens_out, k_new, v_new, releasable_from)
    T, V = logits.shape
    C = mode.shape[0]
    num_pages, Hkv, page_size, D = k_cache.shape
    max_pages = page_table.shape[1]
    rc = lib().idlm_isd_accept_commit(
        _ptr(logits), _dtype(logits), V, _ptr(qo_indptr), _ptr(mode), _ptr(drafts),
        _ptr(draft_q_stats), _ptr(prev_logits), prev_logits.shape[0], _ptr(prev_mask_row0),
        C, T, N, float(temperature), int(proposal_mode), int(seed), int(step), _ptr(n_accepted),
        _ptr(out_tokens), _ptr(n_out), _ptr(n_commit), _ptr(next_drafts), _ptr(next_q_stats),
        _ptr(next_mode), _ptr(next_mask_row0), _ptr(row_stats), _ptr(dbg), _ptr(k_cache),
        _ptr(v_cache), _ptr(page_table), max_pages, _ptr(seq_lens_in), _ptr(seq_lens_out),
        _ptr(k_new), _ptr(v_new), Hkv, D, page_size, num_pages, _dtype(k_cache),
        _ptr(releasable_from), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream))
    _check(rc, "idlm_isd_accept_commit")


# ------------------------------------------------------- multi-step loop pieces

def idlm_synth_logits(logits, qo_indptr, row_req, row_pos, row_token, scale_z, scale_e, seed,
                      step, stream=None):
    """Synthetic model rows (the seeded workload's stand-in for the forward
    pass) into logits [T, V] bf16 for the rows in use."""
    _contig(logits, qo_indptr, row_req, row_pos, row_token, scale_e)
    T, V = logits.shape
    C = scale_e.shape[0]
    rc = lib().idlm_synth_logits(_ptr(logits), C, T, V, _ptr(qo_indptr), _ptr(row_req),
                                 _ptr(row_pos), _ptr(row_token), float(scale_z), _ptr(scale_e),
                                 int(seed) & 0xFFFFFFFF, int(step), _stream(stream))
    _check(rc, "idlm_synth_logits")


def idlm_isd_advance(N, mode, next_mode, out_tokens, n_out, n_accepted, next_drafts, seq_lens,
                     qo_indptr, row_req, row_pos, row_token, status, counters=None,
                     history=None, hist_len=None, count=True, stream=None):
    _contig(mode, next_mode, out_tokens, n_out, n_accepted, next_drafts, seq_lens, qo_indptr,
            row_req, row_pos, row_token, counters, history, hist_len)
    C = next_mode.shape[0]
    T = row_req.shape[0]
    cap = 0 if history is None else history.shape[1]
    rc = lib().idlm_isd_advance(C, N, T, _ptr(mode), _ptr(next_mode), _ptr(out_tokens),
                                _ptr(n_out), _ptr(n_accepted), _ptr(next_drafts), _ptr(seq_lens),
                                _ptr(qo_indptr), _ptr(row_req), _ptr(row_pos), _ptr(row_token),
                                _ptr(counters), _ptr(history), cap, _ptr(hist_len),
                                1 if count else 0, _ptr(status), _stream(stream))
    _check(rc, "idlm_isd_advance")


# ------------------------------------------------------------- decoder layer

def layer_weights(W, hidden, ffn, n_heads, n_kv_heads, head_dim, rank, lora_scale=1.0,
                  rms_eps=1e-6):
    """idlm_layer_weights over a dict of device tensors (keys as in the
    struct; a_* / b_* / norm* may be missing).  The dict must outlive the
    struct."""
    lw = LayerWeights(hidden, ffn, n_heads, n_kv_heads, head_dim, rank, lora_scale, rms_eps)
    for name, _ in LayerWeights._fields_[8:]:
        t = W.get(name)
        if t is not None:
            _contig(t)
            setattr(lw, name, t.data_ptr())
    return lw


def idlm_risd_layer_workspace_size(lw, M, C, page_size, max_rows):
    return int(lib().idlm_risd_layer_workspace_size(ctypes.byref(lw), M, C, page_size, max_rows))


def idlm_risd_layer(lw, x, out, row_gate, k_cache, v_cache, page_table, seq_lens, qo_indptr,
                    max_rows, workspace, status, k_new_out=None, v_new_out=None, stream=None):
    _contig(x, out, row_gate, k_cache, v_cache, page_table, seq_lens, qo_indptr, workspace,
            k_new_out, v_new_out)
    M = x.shape[0]
    num_pages, _, page_size, _ = k_cache.shape
    C, max_pages = page_table.shape
    rc = lib().idlm_risd_layer(
        ctypes.byref(lw), _ptr(x), _ptr(out), M, _ptr(row_gate), _ptr(k_cache), _ptr(v_cache),
        _ptr(page_table), max_pages, _ptr(seq_lens), _ptr(qo_indptr), C, page_size, num_pages,
        max_rows, _ptr(k_new_out), _ptr(v_new_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    _check(rc, "idlm_risd_layer")
