"""Benchmark of the ISD verify/accept step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload isd_c64_n4_ctx4096]

One step = the whole hot path over one batch: paged strict-causal attention of
the 2N-1 rows of every request against its KV cache, the accept pass (softmax
statistics, p/q test, residual / bonus draw, proposals, next state) and the KV
commit of the accepted rows.  The default workload is C=64 requests, N=4,
4096-token contexts, 32/8 heads of 128, V=151936: synthetic, seeded inputs of
those shapes.  Every step reads ~1.08 GB of KV and 136 MB of logits, more than
the 126 MB L2, so no explicit flush is needed between steps.

The metric is emitted tokens per second (accepted drafts plus the resampled,
bonus or fresh token of each request, the numerator of the pages' tokens per
forward).  Under torchrun each rank runs its own batch (replicas, weak
scaling); the reported value is all ranks' tokens over the slowest rank's
time.  Prints one JSON line (rank 0).
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "ISD accepted tokens/s at C=64,N=4; attention+accept HBM GB/s vs B300 peak"
# library kernel launches per timed step: attention 2 (the pass and the merge
# of units cut between CTAs), accept 3 (the KV commit runs as work items of
# the accept's residual kernel); 6 with --separate-commit
LAUNCHES_PER_STEP = 5


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="isd_c64_n4_ctx4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-lora", action="store_true", help="skip the gated-LoRA leg")
    ap.add_argument("--no-loop", action="store_true", help="skip the decode-loop leg")
    ap.add_argument("--no-ragged", action="store_true",
                    help="skip the ragged 1k-32k workload leg")
    ap.add_argument("--no-lmhead", action="store_true", help="skip the fused LM-head leg")
    ap.add_argument("--separate-commit", action="store_true",
                    help="time the step as idlm_isd_accept then idlm_kv_commit (6 launches) "
                         "instead of idlm_isd_accept_commit (5)")
    ap.add_argument("--leg", default="step", choices=["step", "lora", "layer", "loop", "lmhead"],
                    help="lora: only the gated-LoRA projections (prints their JSON)")
    ap.add_argument("--lora-reps", type=int, default=20)
    ap.add_argument("--lora-rank", type=int, default=None)
    ap.add_argument("--profile-run", action="store_true",
                    help="few launches for a profiler: no clock sampling, e2e or CPU leg")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


def sustained_bf16():
    """The bf16 GEMM rate held for seconds under the power cap (measured), or
    the fallback's settled figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured"
    return 1400.0, "fallback"


LORA_LAYER = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")),
              ("down", ("down",))]


def lora_leg(dev, reps=20, fused=True, rank=None):
    """The gated-LoRA projections of one decoder layer (workload lora_layer_m448:
    hidden 4096, FFN 12288, 448 token rows, rank 16, gate on at MASK rows),
    timed alone with CUDA events.  fused=True is the layer's path: the
    projections that share an input run as one idlm_gated_lora_grouped call
    each (q|k|v: N = 6144, three adapter groups; gate|up: N = 24576, two),
    four calls in all; fused=False times the seven projections one call
    each.  rank overrides the adapters' rank (r = 128 is the pages').
    Returns per-call and whole-layer TFLOP/s (algorithmic 2 M K N per
    projection; the adapter's own work is not counted)."""
    import speculative_verify_accept_step_b300 as L
    from speculative_verify_accept_step_b300 import workloads as wl
    w = wl.WORKLOADS["lora_layer_m448"]
    inp = wl.lora_inputs(w, rank=rank)
    x = inp["x"].to(dev)
    xf = torch.randn(w.T, w.ffn, generator=torch.Generator().manual_seed(3)).bfloat16().to(dev)
    gate = inp["row_gate"].to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    groups = LORA_LAYER if fused else [(n, (n,)) for n in ("q", "k", "v", "o", "gate", "up", "down")]
    out, tot_flop, tot_ms = {}, 0.0, 0.0
    for name, members in groups:
        pj = {k: torch.cat([inp["proj"][m][k] for m in members]).to(dev) for k in ("w", "a", "b")}
        rows = [inp["proj"][m]["w"].shape[0] for m in members]
        xi = xf if name == "down" else x
        M, K = xi.shape
        N, r = pj["w"].shape[0], pj["a"].shape[0] // len(members)
        ws = torch.empty(L.idlm_gated_lora_grouped_workspace_size(M, K, N, r, len(members)),
                         dtype=torch.uint8, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)

        def call():
            L.idlm_gated_lora_grouped(xi, pj["w"], pj["a"], pj["b"], gate, inp["lora_scale"],
                                      rows, y, ws, st)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        fl = 2.0 * M * K * N
        tot_flop += fl
        tot_ms += ms
        out[name] = {"M": M, "K": K, "N": N, "r": r, "groups": len(members), "us": ms * 1e3,
                     "TFLOP/s": fl / ms / 1e9}
        del ws, y
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return {"workload": w.name, "rank": inp["rank"], "calls": out, "layer_us": tot_ms * 1e3,
            "TFLOP/s": tot_flop / tot_ms / 1e9, "layer_GFLOP": tot_flop / 1e9}


def layer_leg(dev, reps=10):
    """The whole decoder layer of the gated-LoRA workload through
    idlm_risd_layer (RMSNorm, q|k|v, attention over the 4096-token paged KV,
    o, residual, RMSNorm, gate|up, SwiGLU, down, residual; 448 rows), timed
    with CUDA events at adapter rank 0, 16 (the workload) and 128 (the
    pages'); alpha = time with adapters / time without.  The KV cache and
    page table are the headline attention batch's."""
    import speculative_verify_accept_step_b300 as L
    from speculative_verify_accept_step_b300 import workloads as wl
    w = wl.WORKLOADS["lora_layer_m448"]
    res = {"workload": w.name, "rows": w.T}
    base = None
    for rank in (0, 16, 128):
        inp = wl.layer_inputs(w, rank=rank)
        W = {k: v.to(dev) for k, v in inp["W"].items()}
        lw = L.layer_weights(W, w.hidden, w.ffn, w.Hq, w.Hkv, w.D, rank, inp["lora_scale"])
        x = inp["x"].to(dev)
        M, C = x.shape[0], inp["page_table"].shape[0]
        ws = torch.empty(L.idlm_risd_layer_workspace_size(lw, M, C, w.page_size, w.rows_full),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(x)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        dv = {k: inp[k].to(dev) for k in ("k_cache", "v_cache", "page_table", "seq_lens",
                                         "qo_indptr", "row_gate")}

        def call():
            L.idlm_risd_layer(lw, x, out, dv["row_gate"], dv["k_cache"], dv["v_cache"],
                              dv["page_table"], dv["seq_lens"], dv["qo_indptr"], w.rows_full,
                              ws, st)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"device status {int(st.item())}"
        us = e0.elapsed_time(e1) / reps * 1e3
        res[f"r{rank}_us"] = us
        if rank == 0:
            base = us
        else:
            res[f"alpha_r{rank}"] = us / base
        del W, ws, dv, inp
        torch.cuda.empty_cache()
    res["alpha_pages"] = 1.12
    return res


def lmhead_leg(dev, reps=20):
    """The LM head fused with the accept step (idlm_lm_head_accept) against
    the two calls it replaces: the same tcgen05 GEMM writing the logits
    (idlm_gated_lora without an adapter), then idlm_isd_accept with its own
    pass over them.  The headline batch: 64 requests, N = 4 (448 rows of a
    FULL step), hidden 4096, V = 151936; random bf16 hidden states and LM-head
    weights (synthetic), the drafts those weights propose at a FRESH step
    before.  Both sides are timed with CUDA events over `reps` calls each."""
    import speculative_verify_accept_step_b300 as L
    C, N, H, V = 64, 4, 4096, 151936
    M = N - 1
    g = torch.Generator(device=dev).manual_seed(5)
    h0 = torch.randn(C * N, H, device=dev, generator=g).bfloat16()
    h1 = torch.randn(C * (2 * N - 1), H, device=dev, generator=g)
    for k in range(1, N):   # clean row k - 1 close to the FRESH step's MASK row k
        h1[k - 1::2 * N - 1] = h0[k::N].float() + 0.35 * torch.randn(C, H, device=dev, generator=g)
    h1 = h1.bfloat16()
    w = (torch.randn(V, H, device=dev, generator=g) * (2.0 / H ** 0.5)).bfloat16()
    i32 = dict(dtype=torch.int32, device=dev)
    qo0 = torch.arange(0, C * N + 1, N, **i32)
    qo1 = torch.arange(0, C * (2 * N - 1) + 1, 2 * N - 1, **i32)
    l0 = torch.empty(C * N, V, dtype=torch.bfloat16, device=dev)
    l1 = torch.empty(C * (2 * N - 1), V, dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, **i32)

    def outs():
        return dict(n_accepted=torch.empty(C, **i32), out_tokens=torch.empty((C, N), **i32),
                    n_out=torch.empty(C, **i32), n_commit=torch.empty(C, **i32),
                    next_drafts=torch.empty((C, M), **i32),
                    next_q_stats=torch.empty((C, M, 2), dtype=torch.float32, device=dev),
                    next_mode=torch.empty(C, dtype=torch.uint8, device=dev),
                    next_mask_row0=torch.empty(C, **i32))
    ws = torch.empty(L.idlm_lm_head_accept_workspace_size(C, C * (2 * N - 1), N, H, V),
                     dtype=torch.uint8, device=dev)
    o0, o1 = outs(), outs()
    L.idlm_lm_head_accept(h0, w, l0, qo0, torch.zeros(C, dtype=torch.uint8, device=dev),
                          torch.full((C, M), -1, **i32),
                          torch.zeros((C, M, 2), dtype=torch.float32, device=dev), l0,
                          torch.zeros(C, **i32), N, 1.0, L.PROPOSE_ARGMAX, 0, 0,
                          o0["n_accepted"], o0["out_tokens"], o0["n_out"], o0["n_commit"],
                          o0["next_drafts"], o0["next_q_stats"], o0["next_mode"],
                          o0["next_mask_row0"], ws, st)

    def fused():
        L.idlm_lm_head_accept(h1, w, l1, qo1, o0["next_mode"], o0["next_drafts"],
                              o0["next_q_stats"], l0, o0["next_mask_row0"], N, 1.0,
                              L.PROPOSE_ARGMAX, 0, 1, o1["n_accepted"], o1["out_tokens"],
                              o1["n_out"], o1["n_commit"], o1["next_drafts"], o1["next_q_stats"],
                              o1["next_mode"], o1["next_mask_row0"], ws, st)
    T1 = C * (2 * N - 1)
    empty_a = torch.zeros((0, H), dtype=torch.bfloat16, device=dev)
    empty_b = torch.zeros((V, 0), dtype=torch.bfloat16, device=dev)
    gate = torch.zeros(T1, dtype=torch.uint8, device=dev)
    gws = torch.empty(L.idlm_gated_lora_workspace_size(T1, H, V, 0), dtype=torch.uint8,
                      device=dev)
    aws = torch.empty(L.idlm_isd_accept_workspace_size(C, T1, N, V), dtype=torch.uint8,
                      device=dev)

    def gemm():
        L.idlm_gated_lora(h1, w, empty_a, empty_b, gate, 1.0, l1, gws, st)

    def accept():
        L.idlm_isd_accept(l1, qo1, o0["next_mode"], o0["next_drafts"], o0["next_q_stats"], l0,
                          o0["next_mask_row0"], N, 1.0, L.PROPOSE_ARGMAX, 0, 1, o1["n_accepted"],
                          o1["out_tokens"], o1["n_out"], o1["n_commit"], o1["next_drafts"],
                          o1["next_q_stats"], o1["next_mode"], o1["next_mask_row0"], aws, st)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3
    t_fused = timed(fused)
    t_gemm = timed(gemm)
    t_acc = timed(accept)
    t_pair = timed(lambda: (gemm(), accept()))
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    flop = 2.0 * T1 * H * V
    return {"requests": C, "N": N, "rows": T1, "hidden": H, "V": V,
            "fused_us": t_fused, "gemm_us": t_gemm, "accept_us": t_acc,
            "gemm_then_accept_us": t_pair, "saved_us": t_pair - t_fused,
            "gemm_TFLOP/s": flop / (t_gemm * 1e-6) / 1e12,
            "fused_TFLOP/s": flop / (t_fused * 1e-6) / 1e12,
            "logits_bytes": T1 * V * 2,
            "note": "logits written once by the GEMM in both; the fused call takes the "
                    "accept's vocabulary statistics in the GEMM's epilogue instead of a "
                    "second pass over the logits"}


def loop_leg(dev, steps=200, warm=10, target=0.9):
    """The stationary-batch decode loop (f1) on the device: the headline batch
    (64 requests, N = 4, V = 151936, 4096-token contexts, 32/8 heads of 128)
    stepping through the synthetic model, attention, accept, commit and the
    hand-off to the next step, `steps` steps replayed from one CUDA graph.
    SAMPLE-mode proposals, so that the realised acceptance is the synthetic
    model's overlap (target 0.9).  tokens_per_forward is the pages' TPF,
    measured; the closed form is evaluated at the acceptance the loop
    realised.  The synthetic model's kernel (which writes the step's logits,
    standing in for the LM head) is inside the timed region."""
    import json as _json
    import speculative_verify_accept_step_b300 as L
    from speculative_verify_accept_step_b300.loop import StationaryLoop
    C, N, V = 64, 4, 151936

    def tpf_closed_form(p, n):
        # memory-bound tokens per forward of the speedup panel:
        # (2 + p + ... + p^(n-2)) / (2 - p^(n-1))
        return (2.0 + sum(p ** i for i in range(1, n - 1))) / (2.0 - p ** (n - 1))
    path = os.path.join(ROOT, "speculative_verify_accept_step_b300", "synth_noise_table.json")
    with open(path) as f:
        sigma = float(_json.load(f)["sigma"][str(target)])
    lp = StationaryLoop(C, N, V, torch.arange(C), torch.full((C,), 4096), [sigma] * C,
                        steps=warm + steps + 1, seed=11, proposal_mode=L.PROPOSE_SAMPLE,
                        attention=dict(Hq=32, Hkv=8, D=128), hist_cap=8, dev=dev)
    lp.capture(warm).replay()
    before = lp.results()
    g = lp.capture(steps, step0=warm)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    after = lp.results()
    assert after["status"] == 0, f"device status {after['status']}"
    ms = e0.elapsed_time(e1)
    # the synthetic model alone, on the last step's layout (it stands in for
    # the LM's forward pass and is not part of the ISD step)
    reps = 20
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record()
    for k in range(reps):
        L.idlm_synth_logits(lp.logits[k % 2], lp.qo, lp.row_req, lp.row_pos, lp.row_token,
                            lp.scale_z, lp.scale_e, 11, 10_000 + k)
    e3.record()
    torch.cuda.synchronize()
    model_ms = e2.elapsed_time(e3) / reps
    d = {k: int((after[k] - before[k]).sum()) for k in ("tokens", "forwards", "accepted",
                                                       "tested")}
    p_hat = d["accepted"] / max(d["tested"], 1)
    tpf = d["tokens"] / max(d["forwards"], 1)
    return {"requests": C, "N": N, "context": 4096, "steps": steps, "graph": True,
            "proposals": "sample", "target_acceptance": target,
            "realised_acceptance": p_hat, "tokens_per_forward": tpf,
            "tpf_closed_form_at_realised": tpf_closed_form(p_hat, N),
            "ms_per_step": ms / steps, "tokens_per_s": d["tokens"] / (ms * 1e-3),
            "model_ms_per_step": model_ms,
            "tokens_per_s_without_model": d["tokens"] / ((ms - model_ms * steps) * 1e-3),
            # synth, attention, accept + commit, advance; kernels: synth 1,
            # attention 2, accept 3 (the commit as its work items), advance 1
            "api_calls_per_step": 4, "kernel_launches_per_step": 7,
            "note": "ms_per_step includes the synthetic model kernel (the step's logits, one "
                    "Philox4x32-10 per logit); model_ms_per_step is that kernel timed alone"}


def source_hash(name):
    path = os.path.join(ROOT, "speculative_verify_accept_step_b300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_file, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_file, {}).get(workload)
    if not e or e.get("source_sha") != source_hash(kernel_file):
        return None
    return e.get("bytes_per_launch")


# --------------------------------------------------------------- dist helpers

def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce(x, ws, op):
    """x reduced over the ranks (a host float); the tensor lives where the
    process group's backend wants it (GPU for NCCL, host for gloo)."""
    if ws <= 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def aggregate(tokens_local, ms_local, ws):
    """Whole-job throughput of replicas: every rank's tokens over the slowest
    rank's time.  Returns (tokens, ms, tokens per second)."""
    ms = allreduce(float(ms_local), ws, _max_op())
    tokens = allreduce(float(tokens_local), ws, _sum_op())
    return tokens, ms, tokens / (ms * 1e-3)


# ------------------------------------------------------------- clock sampling

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"isd_clocks_{os.getpid()}.csv")
        self.idx = device_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm

class Step:
    """Device buffers of one ISD step and the three C-ABI calls that run it."""

    def __init__(self, w, dev, seed=0):
        import speculative_verify_accept_step_b300 as L
        from speculative_verify_accept_step_b300 import workloads as wl
        self.L, self.w, self.dev = L, w, dev
        a = wl.attention_inputs(w, seed=seed)
        b = wl.accept_inputs(w, seed=seed)
        self.host = dict(a=a, b=b)
        d = lambda t: t.to(dev)
        self.q, self.k_new, self.v_new = d(a["q"]), d(a["k_new"]), d(a["v_new"])
        self.k_cache, self.v_cache = d(a["k_cache"]), d(a["v_cache"])
        self.page_table, self.seq_lens, self.qo = d(a["page_table"]), d(a["seq_lens"]), d(a["qo_indptr"])
        self.sm_scale = a["sm_scale"]
        self.logits0, self.logits1 = d(b["logits0"]), d(b["logits1"])
        self.qo0, self.qo1 = d(b["qo0"]), d(b["qo1"])
        C, N, T = w.C, w.N, w.T
        M = N - 1
        i32 = dict(dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        self.att_ws = torch.empty(max(L.idlm_isd_attention_workspace_size(
            C, w.Hq, w.Hkv, w.D, w.page_size, w.rows_full, L.IDLM_BF16), 256),
            dtype=torch.uint8, device=dev)
        V = w.V
        self.acc_ws = torch.empty(L.idlm_isd_accept_workspace_size(C, max(T, C * N), N, V),
                                  dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, **i32)
        self.seq_out = torch.empty_like(self.seq_lens)
        self.releasable = torch.empty_like(self.seq_lens)

        def outs():
            return dict(n_accepted=torch.empty(C, **i32), out_tokens=torch.empty((C, N), **i32),
                        n_out=torch.empty(C, **i32), n_commit=torch.empty(C, **i32),
                        next_drafts=torch.empty((C, M), **i32),
                        next_q_stats=torch.empty((C, M, 2), dtype=torch.float32, device=dev),
                        next_mode=torch.empty(C, dtype=torch.uint8, device=dev),
                        next_mask_row0=torch.empty(C, **i32))
        self.outs = outs
        # step 0 (FRESH): the MASK rows of logits0 propose the drafts verified by every
        # timed FULL step
        s0 = outs()
        L.idlm_isd_accept(self.logits0, self.qo0, d(b["mode0"]),
                          torch.full((C, M), -1, **i32),
                          torch.zeros((C, M, 2), dtype=torch.float32, device=dev), self.logits0,
                          torch.zeros(C, **i32), N, w.temperature, L.PROPOSE_ARGMAX, 0, 0,
                          s0["n_accepted"], s0["out_tokens"], s0["n_out"], s0["n_commit"],
                          s0["next_drafts"], s0["next_q_stats"], s0["next_mode"],
                          s0["next_mask_row0"], self.acc_ws, self.status)
        self.mode1, self.drafts, self.dq, self.prow = (s0["next_mode"], s0["next_drafts"],
                                                       s0["next_q_stats"], s0["next_mask_row0"])
        torch.cuda.synchronize()

    def attention(self):
        self.L.idlm_isd_attention(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                  self.page_table, self.seq_lens, self.qo, self.out, self.att_ws,
                                  self.status, max_rows=self.w.rows_full, sm_scale=self.sm_scale)

    def accept(self, o, step, logits=None):
        L, w = self.L, self.w
        L.idlm_isd_accept(self.logits1 if logits is None else logits, self.qo1, self.mode1,
                          self.drafts, self.dq, self.logits0, self.prow, w.N, w.temperature,
                          L.PROPOSE_ARGMAX, 0, step, o["n_accepted"], o["out_tokens"],
                          o["n_out"], o["n_commit"], o["next_drafts"], o["next_q_stats"],
                          o["next_mode"], o["next_mask_row0"], self.acc_ws, self.status)

    def commit(self, o):
        self.L.idlm_kv_commit(self.k_cache, self.v_cache, self.page_table, self.seq_lens,
                              self.seq_out, self.k_new, self.v_new, self.qo, o["n_commit"],
                              self.status, releasable_from=self.releasable)

    def accept_commit(self, o, step):
        L, w = self.L, self.w
        L.idlm_isd_accept_commit(self.logits1, self.qo1, self.mode1, self.drafts, self.dq,
                                 self.logits0, self.prow, w.N, w.temperature, L.PROPOSE_ARGMAX,
                                 0, step, o["n_accepted"], o["out_tokens"], o["n_out"],
                                 o["n_commit"], o["next_drafts"], o["next_q_stats"],
                                 o["next_mode"], o["next_mask_row0"], self.k_cache, self.v_cache,
                                 self.page_table, self.seq_lens, self.seq_out, self.k_new,
                                 self.v_new, self.acc_ws, self.status,
                                 releasable_from=self.releasable)

    def tail(self, o, step, fused=True):
        """Accept and KV commit of the step: one call, or the two calls."""
        if fused:
            self.accept_commit(o, step)
        else:
            self.accept(o, step)
            self.commit(o)


def attention_bytes(w, seq_lens):
    """Algorithmic HBM bytes of one attention launch: every cached K/V byte
    read once, Q and the new K/V rows read once, the output written once, and
    the page-table entries read."""
    el = 2 if w.dtype == "bf16" else 4
    kv = int(seq_lens.sum()) * w.Hkv * w.D * el * 2
    q = w.T * w.Hq * w.D * el
    new = w.T * w.Hkv * w.D * el * 2
    out = w.T * w.Hq * w.D * el
    pages = sum((int(L) + w.page_size - 1) // w.page_size for L in seq_lens) * 4
    return kv + q + new + out + pages


def accept_bytes(w, n_rejected):
    """Algorithmic HBM bytes of one accept call: every logit row read once,
    plus the p_j and q_j rows re-read for each rejected request."""
    el = 2 if w.dtype == "bf16" else 4
    return w.T * w.V * el + n_rejected * 2 * w.V * el


def run_ours(args):
    from speculative_verify_accept_step_b300 import workloads as wl
    rank, ws, local = dist_init()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    st = Step(w, dev, seed=rank)
    K, Wm = args.steps, args.warmup
    outs = [st.outs() for _ in range(K)]
    wo = st.outs()
    fused = not args.separate_commit
    for i in range(Wm):
        st.attention()
        st.tail(wo, 10_000_000 + i, fused)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    if not args.profile_run:
        clocks.start()
    # keep the GPU loaded for ~0.6 s while the sampler starts, so its readings
    # before the timed region are taken under the same load
    t_load = time.time()
    i = 0
    while time.time() - t_load < 0.6 and not args.profile_run:
        for _ in range(50):
            st.attention()
            st.tail(wo, 20_000_000 + i, fused)
            i += 1
        torch.cuda.synchronize()
    # The K timed steps run back to back with events only at the two ends
    # (an event between calls costs time of its own); the per-call split comes
    # from a second pass with an event around every call.
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    e0.record()
    for k in range(K):
        st.attention()
        st.tail(outs[k], k + 1, fused)
    e1.record()
    torch.cuda.synchronize()
    ms_local = e0.elapsed_time(e1)
    # the split pass follows at once, still under load and under the clock
    # sampler (an idle gap first would let the clocks drop and inflate it)
    KB = min(K, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(KB)]
    for k in range(10):
        st.attention()
        st.tail(wo, 60_000_000 + k, fused)
    for k in range(KB):
        ev[k][0].record()
        st.attention()
        ev[k][1].record()
        if fused:
            st.accept_commit(wo, 50_000_000 + k)
            ev[k][2].record()
        else:
            st.accept(wo, 50_000_000 + k)
            ev[k][2].record()
            st.commit(wo)
        ev[k][3].record()
    separate = None
    if fused and not args.profile_run:
        # the two calls the fused one replaces, timed apart (not part of the value)
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(50)]
        for k in range(50):
            st.attention()
            sev[k][0].record()
            st.accept(wo, 30_000_000 + k)
            sev[k][1].record()
            st.commit(wo)
            sev[k][2].record()
        torch.cuda.synchronize()
        separate = {"accept_us": sum(e[0].elapsed_time(e[1]) for e in sev) / 50 * 1e3,
                    "commit_us": sum(e[1].elapsed_time(e[2]) for e in sev) / 50 * 1e3}
    torch.cuda.synchronize()
    barrier(ws)
    clk = clocks.stop()
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    n_out = torch.stack([o["n_out"] for o in outs]).sum().item()
    n_acc = torch.stack([o["n_accepted"] for o in outs]).sum().item()
    n_rej = torch.stack([(o["next_mode"] == 0).sum() for o in outs]).sum().item()
    tokens, ms, _ = aggregate(n_out, ms_local, ws)
    att_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / KB
    acc_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / KB
    com_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / KB
    hbm, bf16, peak_kind = peaks()
    a_bytes = attention_bytes(w, st.host["a"]["seq_lens"])
    c_bytes = accept_bytes(w, n_rej / K)
    att_gbs = a_bytes / (att_ms * 1e-3) / 1e9
    acc_gbs = c_bytes / (acc_ms * 1e-3) / 1e9
    both_gbs = (a_bytes + c_bytes) / ((att_ms + acc_ms) * 1e-3) / 1e9

    e2e = None if args.profile_run else run_e2e(st, args.e2e_steps, ws)
    ragged = None
    if not args.profile_run and not args.no_ragged and w.name != "isd_c64_n4_ctx1k_32k":
        ragged = workload_leg("isd_c64_n4_ctx1k_32k", dev)
    lora = None
    if not args.profile_run and not args.no_lora:
        lora = lora_leg(dev)
        sus, sus_kind = sustained_bf16()
        lora.update({"peak": bf16, "peak_kind": peak_kind, "frac": lora["TFLOP/s"] / bf16,
                     "sustained_peak": sus, "sustained_peak_kind": sus_kind,
                     "frac_of_sustained": lora["TFLOP/s"] / sus,
                     "bound": "tensor", "path": "4 grouped calls (q|k|v, o, gate|up, down)"})
        try:   # the seven projections one call each, for comparison
            ls = lora_leg(dev, fused=False)
            lora["separate"] = {"layer_us": ls["layer_us"], "TFLOP/s": ls["TFLOP/s"],
                                "frac": ls["TFLOP/s"] / bf16, "calls": ls["calls"]}
        except Exception as e:   # reported, never fatal to the step's line
            lora["separate"] = {"error": str(e)[:300]}
    layer = None
    if not args.profile_run and not args.no_lora:
        try:
            layer = layer_leg(dev)
        except Exception as e:   # reported, never fatal to the step's line
            layer = {"error": str(e)[:300]}
    lmhead = None
    if not args.profile_run and not args.no_lmhead:
        try:
            lmhead = lmhead_leg(dev)
        except Exception as e:   # reported, never fatal to the step's line
            lmhead = {"error": str(e)[:300]}
    loop = None
    if not args.profile_run and not args.no_loop:
        try:
            loop = loop_leg(dev)
        except Exception as e:   # reported, never fatal to the step's line
            loop = {"error": str(e)[:300]}
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not args.profile_run:
        cpu = cpu_baseline(w, st.host)
    if rank != 0:
        return
    traffic = ncu_traffic("attention.cu", w.name)
    line = {
        "metric": METRIC,
        "value": tokens / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": ws,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": ms / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the workload)",
        "config": {"workload": w.name, "C": w.C, "N": w.N, "context": w.ctx_lo if w.ctx == "fixed"
                   else f"{w.ctx} [{w.ctx_lo}, {w.ctx_hi}]", "heads": f"{w.Hq}/{w.Hkv}",
                   "head_dim": w.D, "page_size": w.page_size, "V": w.V,
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "l2": "inputs larger than L2 (KV %.2f GB + logits %.0f MB read per step)"
                         % (a_bytes / 1e9, w.T * w.V * 2 / 1e6)},
        "roofline": {"bound": "hbm",
                     "kernel": "idlm_isd_attention (paged_attn_kernel + attn_merge_kernel)",
                     "achieved": att_gbs, "peak": hbm, "unit": "GB/s", "frac": att_gbs / hbm,
                     "peak_kind": peak_kind, "traffic": traffic,
                     "algorithmic_bytes": a_bytes},
        "kernels": {
            "attention": {"us": att_ms * 1e3, "GB/s": att_gbs, "frac": att_gbs / hbm},
            "accept": {"us": acc_ms * 1e3, "GB/s": acc_gbs, "frac": acc_gbs / hbm,
                       "algorithmic_bytes": c_bytes, "includes_kv_commit": fused},
            "commit": ({"us": com_ms * 1e3} if not fused else
                       {"fused_into_accept": True, "separate_calls": separate}),
            "attention+accept": {"GB/s": both_gbs, "frac": both_gbs / hbm},
        },
        "tokens_per_step": n_out / K,
        "accepted_drafts_per_step": n_acc / K,
        "accepted_drafts_per_s": allreduce(float(n_acc), ws, _sum_op()) / (ms * 1e-3),
        # per step: paged_attn_kernel, attn_merge_kernel; vocab_stream_kernel,
        # decide_kernel, work_kernel (which also commits the KV rows);
        # commit_kernel only with --separate-commit (no memsets or copies)
        "gpu_launches": (LAUNCHES_PER_STEP + (0 if fused else 1)) * K,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "lora": lora,
        "layer": layer,
        "loop": loop,
        "lm_head": lmhead,
        "workloads": {"isd_c64_n4_ctx1k_32k": ragged} if ragged else None,
    }
    print(json.dumps(line))


def _max_op():
    import torch.distributed as dist
    return dist.ReduceOp.MAX


def _sum_op():
    import torch.distributed as dist
    return dist.ReduceOp.SUM


def run_e2e(st, K, ws):
    """Same metric through the C ABI with host buffers: every step copies its
    inputs (Q, new K/V rows, logits, layout and draft state) from pinned host
    memory and reads the emitted tokens back.  The copies of step k+1 run on
    a copy stream while step k computes (two input buffers), and each step's
    results go back on a third stream, so the PCIe transfers overlap the
    kernels; the timed region spans all of it."""
    L, w = st.L, st.w
    a, b = st.host["a"], st.host["b"]
    pin = lambda t: t.pin_memory()
    h = dict(q=pin(a["q"]), k_new=pin(a["k_new"]), v_new=pin(a["v_new"]),
             logits=pin(b["logits1"]), page_table=pin(a["page_table"]),
             seq_lens=pin(a["seq_lens"]), qo=pin(a["qo_indptr"]), qo1=pin(b["qo1"]),
             mode=pin(st.mode1.cpu()), drafts=pin(st.drafts.cpu()), dq=pin(st.dq.cpu()),
             prow=pin(st.prow.cpu()))
    h2d = sum(t.numel() * t.element_size() for t in h.values())
    bufs = [{k: torch.empty(t.shape, dtype=t.dtype, device=st.dev) for k, t in h.items()}
            for _ in range(2)]
    outs = [st.outs() for _ in range(K)]
    keys_back = ("out_tokens", "n_out", "next_drafts", "next_mode")
    back = [{k: torch.empty(outs[0][k].shape, dtype=outs[0][k].dtype).pin_memory()
             for k in keys_back} for _ in range(K)]
    d2h = sum(t.numel() * t.element_size() for t in back[0].values())
    seq_out = torch.empty_like(st.seq_lens)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def step(k, base):
        d, o = bufs[k % 2], outs[k]
        L.idlm_isd_attention(d["q"], d["k_new"], d["v_new"], st.k_cache, st.v_cache,
                             d["page_table"], d["seq_lens"], d["qo"], st.out, st.att_ws,
                             st.status, max_rows=w.rows_full, sm_scale=st.sm_scale)
        L.idlm_isd_accept_commit(d["logits"], d["qo1"], d["mode"], d["drafts"], d["dq"],
                                 st.logits0, d["prow"], w.N, w.temperature, L.PROPOSE_ARGMAX, 0,
                                 base + k, o["n_accepted"], o["out_tokens"], o["n_out"],
                                 o["n_commit"], o["next_drafts"], o["next_q_stats"],
                                 o["next_mode"], o["next_mask_row0"], st.k_cache, st.v_cache,
                                 d["page_table"], d["seq_lens"], seq_out, d["k_new"], d["v_new"],
                                 st.acc_ws, st.status, releasable_from=st.releasable)

    rate = None
    for rep in range(2):   # one untimed pass, then the timed one
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        s_in.wait_event(e0)
        ready, free = [ev(), ev()], [None, None]
        done = []
        for k in range(K):
            bi = k % 2
            with torch.cuda.stream(s_in):
                if free[bi] is not None:
                    s_in.wait_event(free[bi])
                for key, t in h.items():
                    bufs[bi][key].copy_(t, non_blocking=True)
                ready[bi].record(s_in)
            comp.wait_event(ready[bi])
            step(k, 30_000_000 + 1000 * rep)
            free[bi] = ev()
            free[bi].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(free[bi])
                for key in keys_back:
                    back[k][key].copy_(outs[k][key], non_blocking=True)
                fin = ev()
                fin.record(s_out)
                done.append(fin)
        comp.wait_event(done[-1])
        e1.record(comp)
        torch.cuda.synchronize()
        if rep:
            tokens = sum(int(bk["n_out"].sum()) for bk in back)
            tokens, ms, rate = aggregate(tokens, e0.elapsed_time(e1), ws)
    return {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K,
            "note": "inputs double-buffered: copy stream for step k+1 overlaps step k"}


def workload_leg(name, dev, steps=20):
    """Attention, accept and commit of another workload (here the ragged
    1k-32k batch), timed per kernel with CUDA events as in the main loop."""
    from speculative_verify_accept_step_b300 import workloads as wl
    w = wl.WORKLOADS[name]
    st = Step(w, dev, seed=0)
    outs = [st.outs() for _ in range(steps)]
    for i in range(3):
        st.attention()
        st.tail(outs[0], 40_000_000 + i)
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for k in range(steps):
        ev[k][0].record()
        st.attention()
        ev[k][1].record()
        st.accept_commit(outs[k], k + 1)
        ev[k][2].record()
        ev[k][3].record()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, f"device status {int(st.status.item())}"
    att = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
    acc = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    tot = sum(e[0].elapsed_time(e[3]) for e in ev) / steps
    n_out = torch.stack([o["n_out"] for o in outs]).sum().item()
    n_rej = torch.stack([(o["next_mode"] == 0).sum() for o in outs]).sum().item()
    hbm, _, _ = peaks()
    ab = attention_bytes(w, st.host["a"]["seq_lens"])
    cb = accept_bytes(w, n_rej / steps)
    L = st.host["a"]["seq_lens"]
    res = {"workload": name, "steps": steps, "tokens_per_step": n_out / steps,
           "tokens_per_s": n_out / (tot * steps * 1e-3),
           "context": {"min": int(L.min()), "max": int(L.max()), "mean": float(L.float().mean())},
           "attention": {"us": att * 1e3, "GB/s": ab / (att * 1e-3) / 1e9,
                         "frac": ab / (att * 1e-3) / 1e9 / hbm, "algorithmic_bytes": ab},
           "accept": {"us": acc * 1e3, "GB/s": cb / (acc * 1e-3) / 1e9,
                      "frac": cb / (acc * 1e-3) / 1e9 / hbm, "algorithmic_bytes": cb,
                      "includes_kv_commit": True}}
    del st, outs
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------- CPU baseline
#
# The oracle (numpy float64) as it stands, timed on the host's cores.  The
# step's host tensors are placed once in shared memory; each worker process
# (spawned, one BLAS thread each) attaches to it and runs the oracle's full
# step (attention, accept, commit) for whole requests.

def _bf16_to_f64(a):
    """bf16 bits (int16 array) or float32 array -> float64."""
    import numpy as np
    if a.dtype == np.int16:
        return (a.astype(np.int32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


class SharedBatch:
    """The host tensors of one step in one shared-memory block (numpy views)."""
    KEYS = ("q", "k_new", "v_new", "k_cache", "v_cache", "page_table", "seq_lens", "qo_indptr",
            "logits0", "logits1", "qo0", "qo1")

    def __init__(self, host):
        import numpy as np
        from multiprocessing import shared_memory
        a, b = host["a"], host["b"]
        src = {k: (a if k in a else b)[k] for k in self.KEYS}
        arrs = {k: (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy()
                for k, t in src.items()}
        self.meta, off = {}, 0
        for k, x in arrs.items():
            self.meta[k] = (off, x.shape, x.dtype.str)
            off += (x.nbytes + 63) // 64 * 64
        self.shm = shared_memory.SharedMemory(create=True, size=max(off, 64))
        for k, x in arrs.items():
            o, shp, dt = self.meta[k]
            np.ndarray(shp, dtype=dt, buffer=self.shm.buf, offset=o)[...] = x
        self.name = self.shm.name

    def close(self):
        self.shm.close()
        self.shm.unlink()


_WORKER = {}


def _worker_init(name, meta, wdict):
    import numpy as np
    from multiprocessing import shared_memory
    sys.path.insert(0, ROOT)
    shm = shared_memory.SharedMemory(name=name)
    _WORKER["shm"] = shm
    _WORKER["arr"] = {k: np.ndarray(shp, dtype=dt, buffer=shm.buf, offset=o)
                      for k, (o, shp, dt) in meta.items()}
    _WORKER["w"] = wdict


def _oracle_request(arr, w, c, step):
    """The oracle's full step for request c; returns the tokens it emits."""
    import numpy as np
    from oracle import isd
    N, P = w["N"], w["page_size"]
    M = N - 1
    qo = arr["qo_indptr"]
    t0, t1 = int(qo[c]), int(qo[c + 1])
    pages = arr["page_table"][c]
    used = pages[pages >= 0].astype(np.int64)
    table = np.full(pages.shape, -1, dtype=np.int64)
    table[:used.size] = np.arange(used.size)      # the request's pages, in table order
    kc = _bf16_to_f64(arr["k_cache"][used])
    vc = _bf16_to_f64(arr["v_cache"][used])
    q = _bf16_to_f64(arr["q"][t0:t1])
    kn = _bf16_to_f64(arr["k_new"][t0:t1])
    vn = _bf16_to_f64(arr["v_new"][t0:t1])
    sl = arr["seq_lens"][c:c + 1].astype(np.int64)
    sub_qo = np.array([0, t1 - t0])
    isd.isd_attention(q, kn, vn, kc, vc, table[None], sl, sub_qo, P, w["sm_scale"])
    r0, r1 = int(arr["qo0"][c]), int(arr["qo1"][c])
    l0 = _bf16_to_f64(arr["logits0"][r0:r0 + N])
    l1 = _bf16_to_f64(arr["logits1"][r1:r1 + 2 * N - 1])
    o0 = isd.isd_accept(l0, np.array([0, N]), np.array([isd.FRESH]), np.full((1, M), -1),
                        l0, np.zeros(1, dtype=np.int64), N, w["temperature"],
                        isd.PROPOSE_ARGMAX, 0, 0, request_ids=np.array([c]))
    o1 = isd.isd_accept(l1, np.array([0, 2 * N - 1]), o0["next_mode"], o0["next_drafts"],
                        l0, o0["next_mask_row0"], N, w["temperature"], isd.PROPOSE_ARGMAX, 0,
                        step, request_ids=np.array([c]))
    isd.kv_commit(kc, vc, table[None], sl, kn, vn, sub_qo, np.array([int(o1["n_commit"][0])]), P)
    return int(o1["n_out"][0])


def _worker_task(task):
    c, step = task
    return _oracle_request(_WORKER["arr"], _WORKER["w"], c, step)


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        return 1


def host_cpu():
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count() or 1
    return {"nproc": os.cpu_count(), "usable_cores": usable, "model": model}


def _wdict(w, host):
    return {"N": w.N, "page_size": w.page_size, "sm_scale": host["a"]["sm_scale"],
            "temperature": w.temperature}


def cpu_baseline(w, host, budget_s=12.0, one_core_s=8.0):
    """The oracle as it stands, on a bounded sample of the same batch: on every
    usable host core (a spawned process pool, one BLAS thread per process,
    whole requests as tasks) and on one core.  `value` is the all-cores
    figure; `cores` the processes that ran."""
    import multiprocessing as mp
    cpu = host_cpu()
    sb = SharedBatch(host)
    wd = _wdict(w, host)
    try:
        # one core: this process, BLAS held to one thread
        import contextlib
        try:
            from threadpoolctl import threadpool_limits
            one = threadpool_limits(limits=1)
        except Exception:
            one = contextlib.nullcontext()
        arr = _attach(sb)
        with one:
            t0 = time.time()
            tok1 = req1 = 0
            while time.time() - t0 < one_core_s and req1 < w.C:
                tok1 += _oracle_request(arr, wd, req1, 1)
                req1 += 1
            dt1 = time.time() - t0
        del arr
        # every usable core: spawned workers (safe after CUDA is initialised)
        P = cpu["usable_cores"]
        env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in env_keys}
        for k in env_keys:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            with ctx.Pool(P, initializer=_worker_init, initargs=(sb.name, sb.meta, wd)) as pool:
                pool.map(_worker_task, [(c % w.C, 1) for c in range(P)])   # warm-up, untimed
                t0 = time.time()
                tokP = doneP = 0
                tasks = ((i % w.C, 2 + i // w.C) for i in range(10 ** 9))
                pending = [pool.apply_async(_worker_task, (next(tasks),)) for _ in range(2 * P)]
                while pending:
                    r = pending.pop(0)
                    tokP += r.get()
                    doneP += 1
                    if time.time() - t0 < budget_s:
                        pending.append(pool.apply_async(_worker_task, (next(tasks),)))
                dtP = time.time() - t0
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
    finally:
        sb.close()
    return {"value": tokP / dtP, "unit": "tokens/s", "cores": P, "kind": "oracle",
            "nproc": cpu["nproc"], "cpu_model": cpu["model"],
            "sample": f"all cores: {doneP} whole-request steps (attention, accept, commit) of the "
                      f"{w.C}-request batch in {dtP:.1f} s on {P} processes (one BLAS thread "
                      f"each); one core: {req1} requests in {dt1:.1f} s; numpy float64",
            "one_core": {"value": tok1 / dt1, "unit": "tokens/s", "cores": 1}}


def _attach(sb):
    import numpy as np
    return {k: np.ndarray(shp, dtype=dt, buffer=sb.shm.buf, offset=o)
            for k, (o, shp, dt) in sb.meta.items()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from speculative_verify_accept_step_b300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    host = dict(a=wl.attention_inputs(w), b=wl.accept_inputs(w))
    sb = SharedBatch(host)
    arr, wd = _attach(sb), _wdict(w, host)
    try:
        for i in range(args.warmup):
            _oracle_request(arr, wd, i % w.C, i + 1)
        t0 = time.time()
        tokens = done = 0
        for k in range(args.steps):
            # a bounded sample of the batch per step: one request
            tokens += _oracle_request(arr, wd, k % w.C, k + 1)
            done += 1
            if time.time() - t0 > 150.0:   # keep the whole run within a few minutes
                break
        dt = time.time() - t0
    finally:
        del arr
        sb.close()
    v = tokens / dt
    cpu = host_cpu()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": done, "steps_requested": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / done * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; shapes of the workload)",
        "config": {"workload": w.name, "C": w.C, "N": w.N, "V": w.V},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _blas_threads(),
                         "kind": "oracle", "nproc": cpu["nproc"], "cpu_model": cpu["model"],
                         "sample": f"one request of {w.C} per step (full step: attention, "
                                   "accept, commit), numpy float64, this process"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    args = parse()
    sys.path.insert(0, ROOT)
    if args.impl == "reference":
        return run_reference(args)
    from speculative_verify_accept_step_b300.build import build
    if not os.path.exists(os.path.join(ROOT, "speculative_verify_accept_step_b300", "libidlm.so")):
        build()
    if args.leg == "layer":
        print(json.dumps(layer_leg(torch.device("cuda", 0))))
        return
    if args.leg == "lmhead":
        print(json.dumps(lmhead_leg(torch.device("cuda", 0))))
        return
    if args.leg == "loop":
        torch.cuda.set_device(0)
        print(json.dumps(loop_leg(torch.device("cuda", 0))))
        return
    if args.leg == "lora":
        dev = torch.device("cuda", 0)
        out = lora_leg(dev, reps=args.lora_reps, rank=args.lora_rank)
        _, bf16, kind = peaks()
        sus, sus_kind = sustained_bf16()
        out.update({"peak": bf16, "peak_kind": kind, "frac": out["TFLOP/s"] / bf16,
                    "sustained_peak": sus, "frac_of_sustained": out["TFLOP/s"] / sus})
        print(json.dumps(out))
        return
    run_ours(args)


if __name__ == "__main__":
    main()
