"""Benchmark of the MTP speculative-decoding hot path on one GB300 per rank.

Default workload: the ~30B-class dense bf16 target (48 layers, d 6144, GQA
48/8 heads of 128, FFN 24576, vocabulary 262144) at batch 8, context 8192,
k = 4, with the 4-layer width-256 drafter and its 2048-centroid clustered head.

One step = one full speculative step: the drafter proposes k tokens per
sequence (spec_draft), the drafts are replaced at the set acceptance rate
(spec_inject_drafts: a seeded stand-in for real text), and the target verifies
the k+1 rows per sequence in one pass with greedy accept (spec_verify).

value = verify tok/s: B*(k+1) verified positions per verify pass, over the
verify pass's device time (CUDA events on the library's stream). Beside it:
the verify pass's HBM GB/s against the measured copy peak and 8 TB/s, the
whole step time, effective (emitted) tok/s, plain greedy GPU tok/s
(spec_decode) and the speculative / greedy speed-up, an acceptance sweep over
the workload's alphas (S = 64 steps each), e2e through host buffers, the
dominant kernel's roofline, clocks, and the CPU oracle as a baseline.

--impl reference times the CPU oracle (the plain fp64 reference) on the same
workload: each step is one verify pass of the oracle over one sequence.
Multi-GPU: sequences are independent and the weights fit one GPU, so N ranks
run N independent replicas (weak scaling, no collective on the data path).
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_spec_gb300 import configs, synth  # noqa: E402

METRIC = "verify tok/s and HBM GB/s (% of roofline); effective tok/s at set acceptance"
UNIT = "tok/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ncu summaries holding the DRAM traffic of the roofline kernel per workload
TRAFFIC_FILES = {"e2b_bf16_b1_ctx2048_k3": "gemv_tc_e2b_verify_projections_traffic.txt",
                 "dense30b_bf16_b8_ctx8192_k4": "wide_kernel_dense30b_m40_projections_traffic.txt"}


def measured_traffic(workload):
    """DRAM bytes per launch of the roofline kernel from the committed ncu
    summary of this workload, or None when there is none or the kernel's
    sources changed since it was taken."""
    import hashlib
    if workload not in TRAFFIC_FILES:
        return None
    p = os.path.join(ROOT, "profiles", TRAFFIC_FILES[workload])
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if line.startswith("#") or not line.strip():
            continue
        k, v = line.split(None, 1)
        kv[k] = v.strip()
    h = hashlib.sha256()
    for f in kv["sources"].split(","):
        h.update(open(os.path.join(ROOT, f), "rb").read())
    if h.hexdigest() != kv["sources_sha256"]:
        return None
    return float(kv["dram_bytes_read_plus_write_per_launch"])


def verify_bytes(w: configs.Workload, ctx_lens):
    """Algorithmic bytes of one verify pass: every linear weight and the tied
    LM head once, plus KV read (keys/values of all committed positions, all
    layers) and KV write (k+1 new positions)."""
    t = w.target
    kv = t.kv_bytes_per_pos()
    return t.weight_bytes() + sum(ctx_lens) * kv + w.B * (w.k + 1) * kv


def gemv_bytes(t: configs.TargetShape, N, K):
    per = {configs.F32: 4.0, configs.BF16: 2.0, configs.Q4_0: 0.5625}[t.wdtype]
    return N * K * per


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, idx):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(idx), "--query-gpu=" + q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for i, n in enumerate(names):
                    if r[5 + i].strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def setup_workload(w: configs.Workload, steps_total: int, device):
    from speculative_decoding_spec_gb300 import binding
    t = w.target
    tw = synth.make_target(t, device=device)
    dw = synth.make_drafter(w.drafter, device=device)
    ctx = synth.make_context_lengths(w.B, *w.ctx)
    grow = steps_total * (w.k + 1) + w.k + 2
    eng = binding.Engine(tw, dw, n_slots=w.B, B_max=w.B, rows_max=w.k + 1, max_ctx=max(ctx) + grow + 64,
                         shuffle_pages=w.ctx[0] != w.ctx[1])
    for b in range(w.B):
        eng.load_prefilled(b, synth.make_prefilled_kv(t, ctx[b] - 1, device=device, seed=synth.SEED_KV + b))
    first = synth.make_tokens(w.B, t.V, device=device).view(w.B, 1)
    ids = eng.seq_ids(list(range(w.B)))
    eng.spec_prefill(ids, eng._in("first", first))
    eng.sync()
    return tw, dw, eng, ids, ctx


def greedy_reference(eng, ids, w, n_tokens):
    """Target greedy tokens for every absolute position ahead (for the
    acceptance injection); the slot state is saved and restored around it."""
    saved = [x.clone() for x in (eng.seq_len, eng.pending, eng.hid, eng.stats)]
    start = eng.seq_len.clone()
    toks = [eng.pending.clone()]
    for _ in range(n_tokens):
        toks.append(eng.spec_decode(ids, w.B).clone())
    eng.sync()
    for dst, src in zip((eng.seq_len, eng.pending, eng.hid, eng.stats), saved):
        dst.copy_(src)
    ref_len = int(start.max()) + n_tokens + 8
    ref = torch.zeros((w.B, ref_len), dtype=torch.int32, device=eng.device)
    seq = torch.stack(toks, 1)                                   # [B][n+1]
    for b in range(w.B):
        s0 = int(start[b])
        ref[b, s0:s0 + seq.shape[1]] = seq[b]
    torch.cuda.synchronize()
    return ref


WIDE_MIN_ELEMS = 1 << 25   # bf16 matrices this large (with rows of >= 4096 columns) take the
WIDE_MIN_K = 4096          # tcgen05 projection at any row count


def roofline_kernel_name(w):
    """The projection kernel(s) the verify pass of this workload runs, the one
    streaming most of the bytes first."""
    t = w.target
    if t.wdtype == configs.F32:
        return "gemv_kernel (CUDA-core weight-streaming projection)"
    wide = "wide_kernel (tcgen05 weight-streaming projection%s; each launch with its wide_prep_kernel)" % (
        ", Q4_0 dequantised in shared memory" if t.wdtype == configs.Q4_0 else "")
    if w.M > 8:
        return wide
    reg = "gemv_tc_kernel (mma.sync weight-streaming projection)"
    if t.wdtype != configs.BF16:
        return reg
    shapes = [(t.nqkv, t.d), (t.d, t.nq * t.hd), (2 * t.ff, t.d), (t.d, t.ff)]
    large = lambda N, K: N * K >= WIDE_MIN_ELEMS and K >= WIDE_MIN_K
    big = sum(t.L * N * K for N, K in shapes if large(N, K)) + (t.V * t.d if large(t.V, t.d) else 0)
    small = sum(t.L * N * K for N, K in shapes if not large(N, K)) + (0 if large(t.V, t.d) else t.V * t.d)
    if small == 0:
        return wide
    return (wide + " for the large matrices, " + reg + " for the rest") if big >= small else (
        reg + " for the per-layer matrices, " + wide + " for the large ones")


def time_dominant_kernel(tw, w, device, reps=5):
    """Average duration of the weight-streaming projection as the verify runs
    it: every layer's QKV, O, gate/up and down projections and the LM head,
    captured in one CUDA graph (2.5 GB+ of weights per replay, so nothing is
    L2-resident) and timed over several replays with CUDA events."""
    from speculative_decoding_spec_gb300 import binding
    t = w.target
    M = w.M
    shapes = [(tw.wqkv, t.d), (tw.wo, t.nq * t.hd), (tw.wgu, t.d), (tw.wdown, t.ff)]
    xs = {K: torch.randn((M, K), device=device) for K in {t.d, t.nq * t.hd, t.ff}}
    ys = {id(W): torch.empty((M, W.N), device=device) for W, _ in shapes + [(tw.embed, t.d)]}
    seq = [(W, K, l) for l in range(t.L) for W, K in shapes] + [(tw.embed, t.d, 0)]
    for W, K, l in seq[:5]:
        binding.spec_linear(W, xs[K], layer=l, y=ys[id(W)])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for W, K, l in seq:
                binding.spec_linear(W, xs[K], layer=l, y=ys[id(W)])
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    nbytes = sum(gemv_bytes(t, W.N, K) for W, K, _ in seq)
    return nbytes / len(seq), e0.elapsed_time(e1) / reps / len(seq)


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over every rank (the slowest rank's
    times, so that the whole job's throughput is all ranks' work over it); the
    values themselves on a single process."""
    if not torch.distributed.is_available() or not torch.distributed.is_initialized() or \
            torch.distributed.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def cpu_model():
    """The host CPU's model name (lscpu), for the baseline line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


class SavedState:
    """Copy of the slot state, to run several measurements from one start."""

    def __init__(self, eng):
        self.eng = eng
        self.t = [x.clone() for x in (eng.seq_len, eng.pending, eng.hid, eng.stats)]

    def restore(self):
        torch.cuda.synchronize()
        for dst, src in zip((self.eng.seq_len, self.eng.pending, self.eng.hid, self.eng.stats), self.t):
            dst.copy_(src)
        torch.cuda.synchronize()


def run_steps(eng, ids, w, ref, alpha, draws, offs, first, n, ev=None):
    """n speculative steps (draft, injection at alpha, verify) on the library's
    stream; step i uses draws/offsets block first + i. ev: optional list of
    (start, end) CUDA event pairs around each verify."""
    st = eng.stream
    dbuf = eng._buf("draws_step", (w.B * w.k,), torch.float32)
    obuf = eng._buf("offs_step", (w.B * w.k,), torch.int32)
    nb = w.B * w.k
    for i in range(n):
        j = first + i
        with torch.cuda.stream(st):
            dbuf.copy_(draws[j * nb:(j + 1) * nb], non_blocking=True)
            obuf.copy_(offs[j * nb:(j + 1) * nb], non_blocking=True)
        d = eng.spec_draft(ids, w.B, w.k)
        eng.spec_inject_drafts(ids, d, ref, alpha, dbuf, obuf)
        if ev is not None:
            ev[i][0].record(st)
        eng.spec_verify(ids, d)
        if ev is not None:
            ev[i][1].record(st)


def emitted_since(eng, w, stats0):
    s1 = [eng.spec_stats(b) for b in range(w.B)]
    return (sum(b.emitted - a.emitted for a, b in zip(stats0, s1)),
            sum(b.accepted - a.accepted for a, b in zip(stats0, s1)))


def run_gpu(args, w, rank, world):
    from speculative_decoding_spec_gb300 import binding  # noqa: F401
    device = "cuda"
    K, W, S = args.steps, args.warmup, args.sweep_steps
    alphas = list(w.alphas) if w.alphas else [0.0]
    alpha = alphas[-1] if args.alpha is None else args.alpha
    n_blocks = max(K + W + 2 * args.e2e_steps, S + 2) + 2
    tw, dw, eng, ids, ctx = setup_workload(w, n_blocks + 2, device)
    start = SavedState(eng)
    ref = greedy_reference(eng, ids, w, n_blocks * (w.k + 1) + w.k + 2)
    nd = n_blocks * w.B * w.k
    draws = synth.make_alpha_draws(nd, device=device)
    offs = synth.make_wrong_offsets(nd, w.target.V, device=device)
    st = eng.stream

    # ---- timed speculative steps at the set alpha ----
    run_steps(eng, ids, w, ref, alpha, draws, offs, 0, W)
    eng.sync()
    stats0 = [eng.spec_stats(b) for b in range(w.B)]
    launches0 = eng.kernel_launches()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("timed")
    t0.record(st)
    run_steps(eng, ids, w, ref, alpha, draws, offs, W, K, evs)
    t1.record(st)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ck = clocks.stop() if clocks else None
    ms_total = t0.elapsed_time(t1)
    verify_ms = sum(a.elapsed_time(b) for a, b in evs) / K
    if world > 1:
        ms_total, verify_ms = max_over_ranks([ms_total, verify_ms], device)
        torch.distributed.barrier()
    launches = eng.kernel_launches() - launches0
    emitted, accepted = emitted_since(eng, w, stats0)
    ms_step = ms_total / K
    rows = w.B * (w.k + 1)
    ctx_now = [int(x) for x in eng.seq_len.cpu()]
    vbytes = verify_bytes(w, ctx_now)
    hbm_peak, tf_peak, peak_kind = peaks()

    # ---- e2e through host buffers (pinned), copies inside the timed region ----
    # verify: H2D of the step's drafts, spec_verify, D2H of the emitted tokens
    # and counts; the whole step: H2D of ids / draws / offsets, draft,
    # injection, verify, D2H.
    h_d = torch.empty((w.B, w.k), dtype=torch.int32).pin_memory()
    h_ids = torch.arange(w.B, dtype=torch.int32).pin_memory()
    h_out = torch.empty((w.B, w.k + 1), dtype=torch.int32).pin_memory()
    h_ne = torch.empty((w.B,), dtype=torch.int32).pin_memory()
    h_draws = draws.cpu().pin_memory()
    h_offs = offs.cpu().pin_memory()
    dbuf = eng._buf("draws_step", (w.B * w.k,), torch.float32)
    obuf = eng._buf("offs_step", (w.B * w.k,), torch.int32)
    d_dev = eng._buf("e2e_drafts", (w.B, w.k), torch.int32)
    nb = w.B * w.k
    base = W + K
    t_verify = t_step = 0.0
    for i in range(args.e2e_steps):
        j = base + i
        # (untimed) drafts of this step to host memory
        d = eng.spec_draft(ids, w.B, w.k)
        with torch.cuda.stream(st):
            dbuf.copy_(draws[j * nb:(j + 1) * nb], non_blocking=True)
            obuf.copy_(offs[j * nb:(j + 1) * nb], non_blocking=True)
        eng.spec_inject_drafts(ids, d, ref, alpha, dbuf, obuf)
        with torch.cuda.stream(st):
            h_d.copy_(d, non_blocking=True)
        st.synchronize()
        te = time.perf_counter()
        with torch.cuda.stream(st):
            d_dev.copy_(h_d, non_blocking=True)
        out, ne = eng.spec_verify(ids, d_dev)
        with torch.cuda.stream(st):
            h_out.copy_(out, non_blocking=True)
            h_ne.copy_(ne, non_blocking=True)
        st.synchronize()
        t_verify += time.perf_counter() - te
    for i in range(args.e2e_steps):
        j = base + args.e2e_steps + i
        te = time.perf_counter()
        with torch.cuda.stream(st):
            ids.copy_(h_ids, non_blocking=True)
            dbuf.copy_(h_draws[j * nb:(j + 1) * nb], non_blocking=True)
            obuf.copy_(h_offs[j * nb:(j + 1) * nb], non_blocking=True)
        d = eng.spec_draft(ids, w.B, w.k)
        eng.spec_inject_drafts(ids, d, ref, alpha, dbuf, obuf)
        out, ne = eng.spec_verify(ids, d)
        with torch.cuda.stream(st):
            h_out.copy_(out, non_blocking=True)
            h_ne.copy_(ne, non_blocking=True)
        st.synchronize()
        t_step += time.perf_counter() - te
    n_e2e = max(args.e2e_steps, 1)

    # ---- plain greedy decoding on the GPU (spec_decode) from the same start ----
    start.restore()
    for _ in range(W):
        eng.spec_decode(ids, w.B)
    eng.sync()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(st)
    for _ in range(K):
        eng.spec_decode(ids, w.B)
    g1.record(st)
    torch.cuda.synchronize()
    greedy_ms = g0.elapsed_time(g1) / K
    greedy_tok_s = w.B * world / (greedy_ms / 1e3)

    # ---- acceptance sweep: S steps at each alpha, from the same start ----
    sweep = []
    for a in alphas:
        start.restore()
        run_steps(eng, ids, w, ref, a, draws, offs, 0, 2)        # warm
        eng.sync()
        s0 = [eng.spec_stats(b) for b in range(w.B)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        run_steps(eng, ids, w, ref, a, draws, offs, 2, S)
        e1.record(st)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        em, ac = emitted_since(eng, w, s0)
        sweep.append({"alpha": a, "steps": S, "ms_per_step": ms / S,
                      "effective_tok_s": em * world / (ms / 1e3),
                      "emitted_per_step": em / (S * w.B),
                      "expected_emitted_per_step": (1 - a ** (w.k + 1)) / (1 - a) if a < 1 else w.k + 1,
                      "accepted_per_draft": ac / (S * w.B * w.k),
                      "speedup_vs_greedy": (em * world / (ms / 1e3)) / greedy_tok_s})

    gb_avg, gms = time_dominant_kernel(tw, w, device)
    eng.sync()

    value = rows * world / (verify_ms / 1e3)
    eff = emitted * world / (ms_total / 1e3)
    res = {
        "metric": METRIC, "value": value, "unit": UNIT,
        "value_is": "verify tok/s = B*(k+1) / verify pass time (device events, library stream)",
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms_step,
        "ms_per_step_is": "whole speculative step: draft + acceptance injection + verify",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"f32": "f32", "bf16": "bf16", "q4_0": "q4_0/f16-scale, fp32 accumulate"}[w.target.wdtype],
        "data": "synthetic (seeded random weights of the named shape; synthetic KV context)",
        "config": {"workload": w.name, "batch": w.B, "k": w.k, "context": list(w.ctx),
                   "alpha": alpha, "target": {"layers": w.target.L, "d": w.target.d, "vocab": w.target.V,
                                              "weights": w.target.wdtype},
                   "drafter": {"layers": w.drafter.L, "hidden": w.drafter.h,
                               "clustered": w.drafter.clustered},
                   "l2": "inputs larger than L2 (%.2f GB of weights streamed per step)" % (
                       w.target.weight_bytes() / 1e9),
                   "parallelism": "replicas x%d" % world},
        "verify": {"tok_s": value, "ms": verify_ms,
                   "hbm_gbs": vbytes / (verify_ms / 1e3) / 1e9, "bytes": vbytes,
                   "frac_of_measured_copy": vbytes / (verify_ms / 1e3) / 1e9 / hbm_peak,
                   "frac_of_8tbs": vbytes / (verify_ms / 1e3) / 1e9 / 8000.0},
        "draft_plus_inject_ms": ms_step - verify_ms,
        "effective_tok_s": eff,
        "greedy": {"tok_s": greedy_tok_s, "ms_per_token": greedy_ms,
                   "what": "plain greedy decoding on the GPU (spec_decode), B tokens per pass"},
        "speedup_vs_greedy": eff / greedy_tok_s,
        "acceptance": {"alpha_set": alpha, "accepted_per_draft": accepted / max(1, K * w.B * w.k),
                       "emitted_per_step": emitted / max(1, K * w.B),
                       "expected_emitted_per_step": (1 - alpha ** (w.k + 1)) / (1 - alpha) if alpha < 1 else
                       w.k + 1},
        "alpha_sweep": sweep,
        "e2e": {"value": rows * world / (t_verify / n_e2e), "unit": UNIT,
                "what": "verify tok/s through host buffers: H2D of the drafts, spec_verify, D2H of the result",
                "h2d_bytes_per_step": int(h_d.numel() * 4),
                "d2h_bytes_per_step": int(h_out.numel() * 4 + h_ne.numel() * 4),
                "whole_step": {"effective_rows_tok_s": rows * world / (t_step / n_e2e),
                               "ms_per_step": 1e3 * t_step / n_e2e,
                               "h2d_bytes_per_step": int(h_ids.numel() * 4 + nb * 8),
                               "d2h_bytes_per_step": int(h_out.numel() * 4 + h_ne.numel() * 4)}},
        "roofline": {"kernel": roofline_kernel_name(w), "bound": "hbm",
                     "achieved": gb_avg / (gms / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gb_avg / (gms / 1e3) / 1e9 / hbm_peak, "peak_kind": peak_kind,
                     "bytes_per_launch": gb_avg, "ms_per_launch": gms,
                     "traffic": measured_traffic(w.name)},
        "gpu_launches": launches,
        "clocks": ck,
    }
    return res, tw, eng, ctx


def cpu_baseline(w, tw, ctx, budget_s=20.0):
    """The oracle timed on the host cores: one verify pass (k+1 rows) of one
    sequence of the workload, on the same weights and context as the GPU."""
    import oracle
    t0 = time.perf_counter()
    T = oracle.Target(tw)
    s = oracle.Seq(T, ctx[0] + w.k + 4)
    s.load_prefilled(synth.make_prefilled_kv(w.target, ctx[0] - 1, device="cpu" if tw.embed.data.device.type == "cpu"
                                             else "cuda", seed=synth.SEED_KV).cpu())
    first = synth.make_tokens(w.B, w.target.V).view(w.B, 1)[0].numpy()
    oracle.prefill(T, s, first)
    prep = time.perf_counter() - t0
    reps, tv = 0, 0.0
    while reps == 0 or (tv < budget_s and reps < 3):
        sc = s.clone()
        t2 = time.perf_counter()
        oracle.verify(T, sc, synth.make_tokens(w.k, w.target.V, seed=77).numpy())
        tv += time.perf_counter() - t2
        reps += 1
    per = tv / reps
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count()))
    return {"value": (w.k + 1) / per, "unit": UNIT, "cores": threads, "cpu_model": cpu_model(),
            "kind": "oracle",
            "sample": "%d verify pass(es) of %d rows (1 sequence of %d, context %d) of %s; fp64 plain C + OpenMP"
                      % (reps, w.k + 1, w.B, ctx[0], w.name),
            "passes_timed": reps, "seconds_per_verify": per, "setup_s": prep}


def run_reference(args, w):
    """--impl reference: the oracle as the reference arm (same metric/config)."""
    import oracle  # noqa: F401
    device = "cuda" if torch.cuda.is_available() else "cpu"
    tw = synth.make_target(w.target, device=device)
    ctx = synth.make_context_lengths(w.B, *w.ctx)
    cb = cpu_baseline(w, tw, ctx, budget_s=args.ref_budget)
    return {"metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 1,
            "steps": cb["passes_timed"], "warmup": 0, "ms_per_step": 1e3 * cb["seconds_per_verify"],
            "steps_note": "each step is one oracle verify pass over one sequence (k+1 rows); "
                          "the steps actually timed, whatever --steps asked",
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic", "config": {"workload": w.name, "batch": w.B, "k": w.k, "context": list(w.ctx)},
            "cpu_baseline": cb, "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=configs.BENCH_WORKLOAD, choices=sorted(configs.WORKLOADS))
    ap.add_argument("--alpha", type=float, default=None)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--sweep-steps", type=int, default=64, help="steps per alpha of the acceptance sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = configs.WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)))
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    from speculative_decoding_spec_gb300 import build
    # one rank builds the library (if it is not built yet), the others load it
    if rank == 0:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    if rank != 0:
        build.build()
    res, tw, eng, ctx = run_gpu(args, w, rank, world)
    eng.close()
    if rank == 0 and not args.no_cpu_baseline:
        try:
            res["cpu_baseline"] = cpu_baseline(w, tw, ctx)
        except Exception as e:  # the baseline is context; never hide the GPU line
            res["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
