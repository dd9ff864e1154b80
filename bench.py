"""Benchmark of the MTP speculative-decoding hot path on one GB300 per rank.

One step = one full speculative step of the workload: the drafter proposes k
tokens per sequence (spec_draft: in-projection, 4 cross-attention + FFN
layers over the target's last-layer KV pages, out-projection, clustered
head), the drafts are replaced at the set acceptance rate (spec_inject_drafts:
a seeded stand-in for real text), and the target verifies the
k+1 rows per sequence in one pass with greedy accept (spec_verify).

value = verified positions per second over whole steps, B*(k+1)*steps / time.
Also reported: verify-only tok/s and HBM GB/s against the roofline, effective
(emitted) tok/s at the set alpha, e2e through host buffers, the dominant
kernel's roofline, clocks, and the CPU oracle as a baseline.

--impl reference times the CPU oracle (the plain fp64 reference) on the same
workload: each step is one verify pass of the oracle.
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

PERSISTENT = 0
DRAFT_CLUSTER = 0
METRIC = "verify tok/s and HBM GB/s (% of roofline); effective tok/s at set acceptance"
UNIT = "tok/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def measured_traffic():
    """DRAM bytes per launch of the roofline kernel from the committed ncu
    summary, or None when the kernel's sources changed since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "gemv_tc_e2b_verify_projections_traffic.txt")
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
                         shuffle_pages=w.ctx[0] != w.ctx[1], persistent=bool(PERSISTENT),
                         draft_cluster=bool(DRAFT_CLUSTER))
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


def roofline_kernel_name(w):
    """The projection kernel the verify pass of this workload runs."""
    t = w.target
    if t.wdtype in (configs.BF16, configs.Q4_0) and w.M > 8:
        return "wide_kernel (tcgen05 weight-streaming projection%s; each launch with its wide_prep_kernel)" % (
            ", Q4_0 dequantised in shared memory" if t.wdtype == configs.Q4_0 else "")
    if t.wdtype in (configs.BF16, configs.Q4_0):
        return "gemv_tc_kernel (mma.sync weight-streaming projection)"
    return "gemv_kernel (CUDA-core weight-streaming projection)"


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


def run_gpu(args, w, rank, world):
    from speculative_decoding_spec_gb300 import binding
    device = "cuda"
    K, W = args.steps, args.warmup
    tw, dw, eng, ids, ctx = setup_workload(w, K + W + args.e2e_steps + 2, device)
    alpha = w.alphas[-1] if w.alphas else 0.0
    if args.alpha is not None:
        alpha = args.alpha
    ref = greedy_reference(eng, ids, w, (K + W + args.e2e_steps + 2) * (w.k + 1) + w.k + 2)
    nd = (K + W + args.e2e_steps + 2) * w.B * w.k
    draws = synth.make_alpha_draws(nd, device=device)
    offs = synth.make_wrong_offsets(nd, w.target.V, device=device)
    dbuf = eng._buf("draws_step", (w.B * w.k,), torch.float32)
    obuf = eng._buf("offs_step", (w.B * w.k,), torch.int32)
    st = eng.stream

    def step(i, ev=None):
        dbuf.copy_(draws[i * w.B * w.k:(i + 1) * w.B * w.k])
        obuf.copy_(offs[i * w.B * w.k:(i + 1) * w.B * w.k])
        d = eng.spec_draft(ids, w.B, w.k)
        eng.spec_inject_drafts(ids, d, ref, alpha, dbuf, obuf)
        if ev is not None:
            ev[0].record(st)
        out, ne = eng.spec_verify(ids, d)
        if ev is not None:
            ev[1].record(st)
        return out, ne

    for i in range(W):
        step(i)
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
    for i in range(K):
        step(W + i, evs[i])
    t1.record(st)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ck = clocks.stop() if clocks else None
    ms_total = t0.elapsed_time(t1)
    if world > 1:
        tt = torch.tensor([ms_total], device=device)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms_total = float(tt.item())
        torch.distributed.barrier()
    launches = eng.kernel_launches() - launches0
    verify_ms = sum(a.elapsed_time(b) for a, b in evs) / K
    stats1 = [eng.spec_stats(b) for b in range(w.B)]
    emitted = sum(s1.emitted - s0.emitted for s0, s1 in zip(stats0, stats1))
    accepted = sum(s1.accepted - s0.accepted for s0, s1 in zip(stats0, stats1))
    ms_step = ms_total / K
    rows = w.B * (w.k + 1)
    ctx_now = [int(x) for x in eng.seq_len.cpu()]
    vbytes = verify_bytes(w, ctx_now)
    hbm_peak, tf_peak, peak_kind = peaks()

    # e2e: the same step through host buffers (pinned), copies inside the timed region
    h_draws = torch.empty((w.B * w.k,), dtype=torch.float32).pin_memory()
    h_offs = torch.empty((w.B * w.k,), dtype=torch.int32).pin_memory()
    h_ids = torch.arange(w.B, dtype=torch.int32).pin_memory()
    h_out = torch.empty((w.B, w.k + 1), dtype=torch.int32).pin_memory()
    h_ne = torch.empty((w.B,), dtype=torch.int32).pin_memory()
    base = W + K
    h_draws_all = draws.cpu().pin_memory()
    h_offs_all = offs.cpu().pin_memory()
    torch.cuda.synchronize()
    te = time.perf_counter()
    for i in range(args.e2e_steps):
        j = base + i
        h_draws.copy_(h_draws_all[j * w.B * w.k:(j + 1) * w.B * w.k])
        h_offs.copy_(h_offs_all[j * w.B * w.k:(j + 1) * w.B * w.k])
        with torch.cuda.stream(st):
            ids.copy_(h_ids, non_blocking=True)
            dbuf.copy_(h_draws, non_blocking=True)
            obuf.copy_(h_offs, non_blocking=True)
        d = eng.spec_draft(ids, w.B, w.k)
        eng.spec_inject_drafts(ids, d, ref, alpha, dbuf, obuf)
        out, ne = eng.spec_verify(ids, d)
        with torch.cuda.stream(st):
            h_out.copy_(out, non_blocking=True)
            h_ne.copy_(ne, non_blocking=True)
        st.synchronize()
    e2e_s = (time.perf_counter() - te) / max(args.e2e_steps, 1)

    gb_avg, gms = time_dominant_kernel(tw, w, device)
    eng.sync()

    res = {
        "metric": METRIC, "value": rows * K * world / (ms_total / 1e3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": ms_step,
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
        "verify": {"tok_s": rows * world / (verify_ms / 1e3), "ms": verify_ms,
                   "hbm_gbs": vbytes / (verify_ms / 1e3) / 1e9, "bytes": vbytes,
                   "frac_of_measured_copy": vbytes / (verify_ms / 1e3) / 1e9 / hbm_peak,
                   "frac_of_8tbs": vbytes / (verify_ms / 1e3) / 1e9 / 8000.0},
        "draft_plus_inject_ms": ms_step - verify_ms,
        "effective_tok_s": emitted * world / (ms_total / 1e3),
        "acceptance": {"alpha_set": alpha, "accepted_per_draft": accepted / max(1, K * w.B * w.k),
                       "emitted_per_step": emitted / max(1, K * w.B),
                       "expected_emitted_per_step": (1 - alpha ** (w.k + 1)) / (1 - alpha) if alpha < 1 else
                       w.k + 1},
        "e2e": {"value": rows * world / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": int(h_ids.numel() * 4 + h_draws.numel() * 4 + h_offs.numel() * 4),
                "d2h_bytes_per_step": int(h_out.numel() * 4 + h_ne.numel() * 4)},
        "roofline": {"kernel": roofline_kernel_name(w), "bound": "hbm",
                     "achieved": gb_avg / (gms / 1e3) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                     "frac": gb_avg / (gms / 1e3) / 1e9 / hbm_peak, "peak_kind": peak_kind,
                     "bytes_per_launch": gb_avg, "ms_per_launch": gms,
                     "traffic": measured_traffic() if w.name == configs.BENCH_WORKLOAD else None},
        "gpu_launches": launches,
        "persistent_pass": bool(PERSISTENT),
        "fused_drafter": bool(DRAFT_CLUSTER),
        "clocks": ck,
    }
    return res, tw, eng, ctx


def cpu_baseline(w, tw, eng, ctx, budget_s=20.0, impl_line=False):
    """The oracle timed on the host cores: one verify pass (k+1 rows) of one
    sequence of the workload, on the same weights and context as the GPU."""
    import oracle
    t0 = time.perf_counter()
    T = oracle.Target(tw)
    s = oracle.Seq(T, ctx[0] + w.k + 4)
    s.load_prefilled(synth.make_prefilled_kv(w.target, ctx[0] - 1, device="cpu" if tw.embed.data.device.type == "cpu"
                                             else "cuda", seed=synth.SEED_KV).cpu())
    first = synth.make_tokens(w.B, w.target.V).view(w.B, 1)[0].numpy()
    prep = time.perf_counter() - t0
    reps, tv = 0, 0.0
    while reps == 0 or (tv < budget_s and reps < 3):
        sc = s.clone()
        t1 = time.perf_counter()
        oracle.prefill(T, sc, first)
        t2 = time.perf_counter()
        oracle.verify(T, sc, synth.make_tokens(w.k, w.target.V, seed=77).numpy())
        tv += time.perf_counter() - t2
        reps += 1
    per = tv / reps
    return {"value": (w.k + 1) / per, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": "%d verify pass(es) of %d rows (1 sequence, context %d) of %s; fp64 plain C + OpenMP"
                      % (reps, w.k + 1, ctx[0], w.name),
            "seconds_per_verify": per, "setup_s": prep}


def run_reference(args, w):
    """--impl reference: the oracle as the reference arm (same metric/config)."""
    import oracle  # noqa: F401
    device = "cuda" if torch.cuda.is_available() else "cpu"
    tw = synth.make_target(w.target, device=device)
    ctx = synth.make_context_lengths(w.B, *w.ctx)
    cb = cpu_baseline(w, tw, None, ctx, budget_s=args.ref_budget)
    return {"metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * cb["seconds_per_verify"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic", "config": {"workload": w.name, "batch": 1, "k": w.k, "context": list(w.ctx)},
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
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=20.0)
    ap.add_argument("--persistent", type=int, default=0,
                    help="1: one persistent kernel per target pass; 0: one kernel per step")
    ap.add_argument("--draft-cluster", type=int, default=0,
                    help="1: all drafter steps in one thread-block-cluster launch; 0: one kernel per operation")
    args = ap.parse_args()
    global PERSISTENT, DRAFT_CLUSTER
    PERSISTENT = args.persistent
    DRAFT_CLUSTER = args.draft_cluster
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
    build.build()
    res, tw, eng, ctx = run_gpu(args, w, rank, world)
    if rank == 0 and not args.no_cpu_baseline:
        try:
            res["cpu_baseline"] = cpu_baseline(w, tw, eng, ctx)
        except Exception as e:  # the baseline is context; never hide the GPU line
            res["cpu_baseline"] = {"value": None, "error": str(e)[:200]}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
