"""Small, self-contained GPU cases for profiling the hot kernels with ncu.
Each summary under profiles/ names the case and the ncu command it ran.

    python profile_cases.py projections
        every projection of one verify pass of the E2B-shaped bf16 target
        (24 layers x QKV, O, gate/up, down, then the LM head; M = 4 rows),
        run twice. About 2.5 GB of weights, so nothing stays in L2.
    python profile_cases.py projections_wide
        one layer of the E4B-shaped bf16 target (QKV, O, gate/up, down) and
        its LM head at M = 40 rows (batch 8, k = 4): the tcgen05 path, run
        twice. About 0.86 GB of weights.
    python profile_cases.py projections_30b
        one layer of the ~30B-class bf16 target (QKV, O, gate/up, down: 1.08
        GB) at M = 40 rows (batch 8, k = 4), run twice: the per-layer matrix
        shapes of the bench's roofline kernel.
    python profile_cases.py layer_and_head_30b
        the same layer followed by the LM head (262144 x 6144 bf16, 3.2 GB),
        run twice: one of each projection shape of a verify pass.
    python profile_cases.py projections_30b_m5
        the same shapes at M = 5 rows (batch 1, k = 4).
    python profile_cases.py projections_wide_q4
        one layer of the E2B-shaped Q4_0 target and its LM head at M = 20
        rows (batch 4, k = 4): the tcgen05 path with shared-memory
        dequantisation, run twice. About 0.24 GB of codes and scales.
    python profile_cases.py verify_q4b4
        three verify passes of the E2B-shaped Q4_0 batch-4 workload (ctx
        4096, k = 4; about 1.6 GB on the device).
    python profile_cases.py draft
        three draft calls (k = 3) on the E2B-shaped workload.
    python profile_cases.py verify
        three verify passes (k = 3) of the E2B-shaped workload.
    python profile_cases.py attention_30b
        the verify attention of the ~30B-class model at batch 8, context
        8192, k = 4 (one layer's cache: 268 MB), three launches.
    python profile_cases.py lmhead_30b
        the ~30B-class model's LM head (262144 x 6144 bf16, 3.2 GB) at M = 40
        rows, twice.
    python profile_cases.py step_30b_b8
        the bench's workload (~30B-class bf16, batch 8, context 8192, k = 4):
        two speculative steps (draft, then verify) inside an NVTX range
        "step" after the set-up (about 70 GB on the device).
    python profile_cases.py verify_moe
        the mixture-of-experts workload (batch 8, context 4096, k = 4): two
        verify passes inside an NVTX range "verify".

Inputs are the seeded synthetic weights and caches of the workloads; nothing
here checks results (the tests do).
"""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from speculative_decoding_spec_gb300 import binding, configs, synth  # noqa: E402

WORKLOAD = "e2b_bf16_b1_ctx2048_k3"


def _engine(w):
    t = w.target
    tw = synth.make_target(t, device="cuda")
    dw = synth.make_drafter(w.drafter, device="cuda")
    ctx = synth.make_context_lengths(w.B, *w.ctx)
    eng = binding.Engine(tw, dw, n_slots=w.B, B_max=w.B, rows_max=w.k + 1, max_ctx=max(ctx) + 64)
    for b in range(w.B):
        eng.load_prefilled(b, synth.make_prefilled_kv(t, ctx[b] - 1, device="cuda", seed=synth.SEED_KV + b))
    ids = eng.seq_ids(list(range(w.B)))
    eng.spec_prefill(ids, eng._in("first", synth.make_tokens(w.B, t.V, device="cuda").view(w.B, 1)))
    eng.sync()
    return tw, eng, ids


def projections(w):
    t = w.target
    tw = synth.make_target(t, device="cuda")
    shapes = [(tw.wqkv, t.d), (tw.wo, t.nq * t.hd), (tw.wgu, t.d), (tw.wdown, t.ff)]
    seq = [(W, K, l) for l in range(t.L) for W, K in shapes] + [(tw.embed, t.d, 0)]
    xs = {K: torch.randn((w.M, K), device="cuda") for K in {t.d, t.nq * t.hd, t.ff}}
    ys = {id(W): torch.empty((w.M, W.N), device="cuda") for W, _, _ in seq}
    for _ in range(2):
        for W, K, l in seq:
            binding.spec_linear(W, xs[K], layer=l, y=ys[id(W)])
        torch.cuda.synchronize()


def _one_layer_and_head(t, M, seed, head=True):
    g = torch.Generator(device="cuda").manual_seed(seed)
    shapes = [(t.nqkv, t.d), (t.d, t.nq * t.hd), (2 * t.ff, t.d), (t.d, t.ff)] + ([(t.V, t.d)] if head else [])
    seq = [(synth.make_matrix(g, t.wdtype, 1, N, K, t.wstd, "cuda"), K) for N, K in shapes]
    xs = {K: torch.randn((M, K), device="cuda") for _, K in seq}
    ys = [torch.empty((M, W.N), device="cuda") for W, _ in seq]
    for _ in range(2):
        for (W, K), y in zip(seq, ys):
            binding.spec_linear(W, xs[K], y=y)
        torch.cuda.synchronize()


def projections_wide(w):
    _one_layer_and_head(configs.E4B, 40, 3)


def projections_30b(w):
    _one_layer_and_head(configs.DENSE30B, 40, 5, head=False)


def layer_and_head_30b(w):
    _one_layer_and_head(configs.DENSE30B, 40, 5, head=True)


def projections_30b_m5(w):
    _one_layer_and_head(configs.DENSE30B, 5, 5, head=False)


def projections_wide_q4(w):
    _one_layer_and_head(configs.E2B_Q4, 20, 4)


def verify_q4b4(w):
    verify(configs.WORKLOADS["e2b_q4_0_b4_ctx4096_k4"])


def draft(w):
    _, eng, ids = _engine(w)
    for _ in range(3):
        eng.spec_draft(ids, w.B, w.k)
    eng.sync()


def verify(w):
    _, eng, ids = _engine(w)
    d = eng._in("d", torch.arange(1, 1 + w.B * w.k, dtype=torch.int32).view(w.B, w.k))
    for _ in range(3):
        eng.spec_verify(ids, d)
    eng.sync()


def attention_30b(w):
    t = configs.DENSE30B
    B, R, ctx = 8, 5, 8192
    shape = configs.TargetShape(**{**t.__dict__, "L": 1})
    pages = (ctx + 63) // 64
    g = torch.Generator(device="cuda").manual_seed(9)
    pool = torch.randn((1, B * pages, 2, t.nkv, 64, t.hd), generator=g, device="cuda").to(torch.bfloat16)
    bt = synth.make_page_table(B, pages, B * pages, shuffle=True, device="cuda")
    ids = torch.arange(B, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), ctx - R, dtype=torch.int32, device="cuda")
    q = torch.randn((B * R, t.nq * t.hd), generator=g, device="cuda")
    for _ in range(3):
        binding.spec_attention(shape, pool, bt, 0, ids, lens, R, t.nq, 1, q)
    torch.cuda.synchronize()


def lmhead_30b(w):
    t = configs.DENSE30B
    g = torch.Generator(device="cuda").manual_seed(6)
    W = synth.make_matrix(g, t.wdtype, 1, t.V, t.d, t.wstd, "cuda")
    x = torch.randn((40, t.d), device="cuda")
    y = torch.empty((40, t.V), device="cuda")
    for _ in range(2):
        binding.spec_linear(W, x, y=y)
    torch.cuda.synchronize()


def _steps(w, nvtx, n, draft=True):
    _, eng, ids = _engine(w)
    d0 = eng._in("d0", torch.arange(1, 1 + w.B * w.k, dtype=torch.int32).view(w.B, w.k))
    # one untimed round so that every call shape is captured before the range
    if draft:
        eng.spec_draft(ids, w.B, w.k)
    eng.spec_verify(ids, d0)
    eng.sync()
    torch.cuda.nvtx.range_push(nvtx)
    for _ in range(n):
        d = eng.spec_draft(ids, w.B, w.k) if draft else d0
        eng.spec_verify(ids, d)
    eng.sync()
    torch.cuda.nvtx.range_pop()


def step_30b_b8(w):
    _steps(configs.WORKLOADS["dense30b_bf16_b8_ctx8192_k4"], "step", 2)


def verify_moe(w):
    _steps(configs.WORKLOADS["moe_bf16_b8_ctx4096_k4"], "verify", 2, draft=False)


CASES = {"projections": projections, "projections_wide": projections_wide, "projections_30b": projections_30b,
         "layer_and_head_30b": layer_and_head_30b,
         "projections_30b_m5": projections_30b_m5, "projections_wide_q4": projections_wide_q4,
         "verify_q4b4": verify_q4b4, "draft": draft, "verify": verify, "attention_30b": attention_30b,
         "lmhead_30b": lmhead_30b, "step_30b_b8": step_30b_b8, "verify_moe": verify_moe}


def main(argv):
    if len(argv) != 1 or argv[0] not in CASES:
        print(__doc__)
        return 2
    from speculative_decoding_spec_gb300 import build
    build.build()
    CASES[argv[0]](configs.WORKLOADS[WORKLOAD])
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
