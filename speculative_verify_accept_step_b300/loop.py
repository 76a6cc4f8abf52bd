"""Stationary-batch ISD decode loop on one GPU: K consecutive steps for a
fixed batch of C requests, with every FULL/FRESH transition decided and
handed on by the device ("Introspective Diffusion Language Models", section
"Serving (SGLang)": stationary-batch decode loop, CUDA-graph capture).

This module only wires C-ABI calls together and owns their device buffers
(PyTorch tensors); every step of the path runs in the library's kernels:

    per step k (one stream):
      idlm_synth_logits   the seeded stand-in for the model's forward pass
                          (logit rows of this step's layout)
      idlm_isd_attention  the step rows against the paged KV cache (optional)
      idlm_isd_accept_commit  p/q test, residual / bonus / fresh draw,
                          proposals, and the anchor + accepted drafts into the
                          cache (the commits as work items of the accept)
      idlm_isd_advance    the next step's row layout, counters, history

Accept state is double-buffered: step k reads the outputs of step k-1 and
writes its own; the logits alternate between two buffers so that step k's
MASK rows are step k+1's q rows.  The buffers have the largest shape
(C (2N-1) rows), and every kernel reads the row count in use from the device
layout, so the launches are identical from step to step and K steps capture
into one CUDA graph.
"""
import torch

from . import _lib as L


class StationaryLoop:
    """K ISD steps for a fixed batch.

    first_token [C]: the token each request starts from (end of its prompt,
    not yet in the cache); start_len [C]: committed lengths.  sigma [C]: the
    synthetic model's MASK-row noise scale per request (acceptance target);
    logit_std: scale of its clean rows.  attention: None (no attention call)
    or dict(Hq, Hkv, D) for a bf16 paged cache with random keys and values
    and random step rows; the cache always exists (the commit writes it),
    with 16-token pages and room for every slot the loop can commit.
    """

    def __init__(self, C, N, V, first_token, start_len, sigma, steps, logit_std=3.0, seed=0,
                 temperature=1.0, proposal_mode=L.PROPOSE_ARGMAX, attention=None,
                 hist_cap=None, dev="cuda", data_seed=0):
        self.C, self.N, self.V, self.K = C, N, V, steps
        self.seed, self.temperature, self.proposal_mode = seed, temperature, proposal_mode
        self.dev = dev
        M = N - 1
        T = C * (2 * N - 1)
        self.T = T
        i32 = dict(dtype=torch.int32, device=dev)
        from . import workloads as wl
        self.scale_z = wl.synth_scale(logit_std)
        self.scale_e = torch.tensor([wl.synth_scale(s) for s in sigma], dtype=torch.float32,
                                    device=dev)
        self.logits = [torch.zeros((T, V), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.qo = torch.zeros(C + 1, **i32)
        self.row_req = torch.zeros(T, **i32)
        self.row_pos = torch.zeros(T, **i32)
        self.row_token = torch.zeros(T, **i32)

        def outs():
            return dict(n_accepted=torch.zeros(C, **i32), out_tokens=torch.full((C, N), -1, **i32),
                        n_out=torch.ones(C, **i32), n_commit=torch.zeros(C, **i32),
                        next_drafts=torch.full((C, M), -1, **i32),
                        next_q_stats=torch.zeros((C, M, 2), dtype=torch.float32, device=dev),
                        next_mode=torch.zeros(C, dtype=torch.uint8, device=dev),
                        next_mask_row0=torch.zeros(C, **i32))
        self.o = [outs(), outs()]
        # "step -1": every request FRESH with its first token pending
        self.o[1]["out_tokens"][:, 0] = first_token.to(dev).to(torch.int32)
        self.o[1]["next_mode"].fill_(L.MODE_FRESH)
        self.seq_lens = start_len.to(dev).to(torch.int32).clone()
        self.counters = torch.zeros((4, C), **i32)
        cap = hist_cap if hist_cap is not None else N * steps
        self.history = torch.full((C, cap), -1, **i32)
        self.hist_len = torch.zeros(C, **i32)
        self.status = torch.zeros(1, **i32)

        # paged KV cache with room for every slot the loop can commit (drawn
        # on the device: nothing downstream compares attention outputs here)
        g = torch.Generator(device=dev).manual_seed(data_seed)
        P = 16
        a = attention or dict(Hq=4, Hkv=1, D=64)
        self.att = attention is not None
        self.Hq, self.Hkv, self.D = a["Hq"], a["Hkv"], a["D"]
        start_max = int(start_len.max())
        per_req = (start_max + N * (steps + 1) + P - 1) // P
        self.page_table = torch.randperm(C * per_req, generator=g, device=dev).to(
            torch.int32).reshape(C, per_req)
        num_pages = C * per_req
        kv_dt = torch.bfloat16
        shape = (num_pages, self.Hkv, P, self.D)
        if self.att:
            self.k_cache = torch.randn(shape, generator=g, device=dev).to(kv_dt)
            self.v_cache = torch.randn(shape, generator=g, device=dev).to(kv_dt)
        else:
            self.k_cache = torch.zeros(shape, dtype=kv_dt, device=dev)
            self.v_cache = torch.zeros(shape, dtype=kv_dt, device=dev)
        self.q = torch.randn(T, self.Hq, self.D, generator=g, device=dev).to(kv_dt)
        self.k_new = torch.randn(T, self.Hkv, self.D, generator=g, device=dev).to(kv_dt)
        self.v_new = torch.randn(T, self.Hkv, self.D, generator=g, device=dev).to(kv_dt)
        self.att_out = torch.empty_like(self.q)
        ws = L.idlm_isd_attention_workspace_size(C, self.Hq, self.Hkv, self.D, P, 2 * N - 1,
                                                 L.IDLM_BF16)
        self.att_ws = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
        self.acc_ws = torch.empty(L.idlm_isd_accept_workspace_size(C, T, N, V),
                                  dtype=torch.uint8, device=dev)
        self.releasable = torch.zeros(C, **i32)
        self.sm_scale = self.D ** -0.5
        # the first step's layout
        o = self.o[1]
        L.idlm_isd_advance(N, o["next_mode"], o["next_mode"], o["out_tokens"], o["n_out"],
                           o["n_accepted"], o["next_drafts"], self.seq_lens, self.qo,
                           self.row_req, self.row_pos, self.row_token, self.status,
                           counters=self.counters, history=self.history,
                           hist_len=self.hist_len, count=False)

    def step(self, k, step0=0, model=True):
        """Launch step k (no host synchronisation).  model=False skips the
        synthetic model (the logits of buffer k % 2 are used as they are)."""
        N = self.N
        cur, prev = self.o[k % 2], self.o[(k + 1) % 2]
        logits, prev_logits = self.logits[k % 2], self.logits[(k + 1) % 2]
        if model:
            L.idlm_synth_logits(logits, self.qo, self.row_req, self.row_pos, self.row_token,
                                self.scale_z, self.scale_e, self.seed, step0 + k)
        if self.att:
            L.idlm_isd_attention(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                 self.page_table, self.seq_lens, self.qo, self.att_out,
                                 self.att_ws, self.status, max_rows=2 * N - 1,
                                 sm_scale=self.sm_scale)
        # accept, then the kept rows into the cache (lengths advanced in place),
        # in one call
        L.idlm_isd_accept_commit(logits, self.qo, prev["next_mode"], prev["next_drafts"],
                                 prev["next_q_stats"], prev_logits, prev["next_mask_row0"], N,
                                 self.temperature, self.proposal_mode, self.seed, step0 + k,
                                 cur["n_accepted"], cur["out_tokens"], cur["n_out"],
                                 cur["n_commit"], cur["next_drafts"], cur["next_q_stats"],
                                 cur["next_mode"], cur["next_mask_row0"], self.k_cache,
                                 self.v_cache, self.page_table, self.seq_lens, self.seq_lens,
                                 self.k_new, self.v_new, self.acc_ws, self.status,
                                 releasable_from=self.releasable)
        L.idlm_isd_advance(N, prev["next_mode"], cur["next_mode"], cur["out_tokens"],
                           cur["n_out"], cur["n_accepted"], cur["next_drafts"], self.seq_lens,
                           self.qo, self.row_req, self.row_pos, self.row_token, self.status,
                           counters=self.counters, history=self.history,
                           hist_len=self.hist_len, count=True)

    def capture(self, steps, step0=0, model=True):
        """One CUDA graph of `steps` consecutive steps (replay() runs them)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for k in range(steps):
                    self.step(k, step0, model)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def run(self, steps=None, step0=0, graph=False):
        steps = self.K if steps is None else steps
        if graph:
            self.capture(steps, step0).replay()
        else:
            for k in range(steps):
                self.step(k, step0)

    def results(self):
        torch.cuda.synchronize()
        c = self.counters.cpu()
        return dict(status=int(self.status.item()), tokens=c[0], forwards=c[1],
                    accepted=c[2], tested=c[3], history=self.history.cpu(),
                    hist_len=self.hist_len.cpu(), seq_lens=self.seq_lens.cpu())
