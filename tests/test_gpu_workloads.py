"""GPU parity at the workloads' full sizes (E2B-, E4B- and ~30B-shaped
targets with the 4-layer clustered drafter), through the C ABI.

Each long context is a synthetic cache for positions [0, ctx-1) followed by
one real target pass at ctx-1 (spec_prefill with R = 1), on the GPU and in the
oracle alike. The oracle then checks, on the same inputs: the pending token
and hidden state, the drafter's k tokens (margin rule), the verify pass's
logits for every row (relative tolerance) and its emitted tokens. Batched
workloads check a sample of sequences in the oracle (rows are independent).
On the GPU alone, speculative steps at the workload's acceptance rate must
emit exactly the GPU's plain greedy tokens."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu


def _setup(w, steps_extra=64, persistent=False, draft_cluster=False):
    t = w.target
    tw = synth.make_target(t, device="cuda")
    dw = synth.make_drafter(w.drafter, device="cuda")
    ctx = synth.make_context_lengths(w.B, *w.ctx)
    eng = binding.Engine(tw, dw, n_slots=w.B, B_max=w.B, rows_max=w.k + 1, max_ctx=max(ctx) + steps_extra,
                         shuffle_pages=True, persistent=persistent,
                         draft_cluster=draft_cluster)
    kvs = []
    for b in range(w.B):
        kv = synth.make_prefilled_kv(t, ctx[b] - 1, device="cuda", seed=synth.SEED_KV + b)
        eng.load_prefilled(b, kv)
        kvs.append(kv)
    first = synth.make_tokens(w.B, t.V, device="cuda").view(w.B, 1)
    ids = eng.seq_ids(list(range(w.B)))
    eng.spec_prefill(ids, eng._in("first", first))
    eng.sync()
    return tw, dw, eng, ids, ctx, kvs, first.cpu()


@pytest.mark.parametrize("name,sample,persistent,draft_cluster", [
    ("e2b_bf16_b1_ctx2048_k3", [0], False, False),
    ("e2b_bf16_b1_ctx2048_k3", [0], True, True),
    ("e2b_q4_0_b1_ctx4096_k4", [0], False, True),
    ("e2b_q4_0_b4_ctx4096_k4", [1, 3], False, False),
    ("e2b_q4_0_b4_ctx4096_k4", [2], False, True),
    ("e4b_bf16_b8_ragged_k4", [0, 5], False, False),
    ("e4b_bf16_b8_ragged_k4", [3], False, True),
])
def test_workload_matches_oracle(name, sample, persistent, draft_cluster):
    w = configs.WORKLOADS[name]
    t = w.target
    tw, dw, eng, ids, ctx, kvs, first = _setup(w, persistent=persistent, draft_cluster=draft_cluster)
    # GPU: draft, then verify the drafted rows with full logits
    d = eng.spec_draft(ids, w.B, w.k).clone()
    logits = torch.empty((w.B * (w.k + 1), t.V), dtype=torch.float32, device="cuda")
    eng.sync()
    pend = eng.pending.clone().cpu()
    hid = eng.hid.clone().cpu()
    out, ne = eng.spec_verify(ids, d, logits)
    eng.sync()
    T, D = oracle.Target(tw), oracle.Drafter(dw)
    tol = TOL[t.wdtype]
    for b in sample:
        s = oracle.Seq(T, ctx[b] + w.k + 8)
        s.load_prefilled(kvs[b].cpu())
        oracle.prefill(T, s, first[b].numpy())
        assert int(pend[b]) == s.pending
        assert_rows_close(hid[b:b + 1].numpy(), s.hid[None], tol, "%s seq %d hidden" % (name, b))
        ref_d, mg_d = oracle.draft(T, D, s.clone(), w.k)
        compare_tokens(d[b].cpu().numpy(), ref_d, mg_d)
        drafts = d[b].cpu().numpy()
        am, mg, _, lg = oracle.forward(T, s.clone(), [s.pending] + list(drafts), want_logits=True)
        rows = logits[b * (w.k + 1):(b + 1) * (w.k + 1)].cpu().numpy()
        assert_rows_close(rows, lg, tol, "%s seq %d verify logits" % (name, b))
        em, _ = oracle.verify(T, s, drafts)
        n = int(ne[b])
        compare_tokens(out[b, :n].cpu().numpy(), em, mg)
        if np.all(mg[:len(em)] > 0.05):
            assert n == len(em)


@pytest.mark.parametrize("name", sorted(configs.WORKLOADS))
def test_speculative_equals_greedy_on_gpu(name):
    """Speculative steps with drafts injected at the workload's acceptance rate
    emit exactly the tokens of the GPU's own plain greedy decoding."""
    w = configs.WORKLOADS[name]
    if w.prompt:
        pytest.skip("covered by the tiny end-to-end tests")
    steps = 4
    tw, dw, eng, ids, ctx, kvs, first = _setup(w, steps_extra=(steps + 2) * (w.k + 1) + 64)
    saved = [x.clone() for x in (eng.seq_len, eng.pending, eng.hid, eng.stats)]
    n_ref = steps * (w.k + 1) + w.k + 2
    start = eng.seq_len.clone()
    toks = [eng.pending.clone()]
    for _ in range(n_ref):
        toks.append(eng.spec_decode(ids, w.B).clone())
    eng.sync()
    greedy = torch.stack(toks, 1).cpu()                     # [B][n_ref+1], from the pending token
    for dst, src in zip((eng.seq_len, eng.pending, eng.hid, eng.stats), saved):
        dst.copy_(src)
    ref_len = int(start.max()) + n_ref + 8
    ref = torch.zeros((w.B, ref_len), dtype=torch.int32)
    for b in range(w.B):
        ref[b, int(start[b]):int(start[b]) + greedy.shape[1]] = greedy[b]
    ref = ref.cuda()
    alpha = w.alphas[-1] if w.alphas else 0.5
    draws = synth.make_alpha_draws(steps * w.B * w.k, device="cuda")
    offs = synth.make_wrong_offsets(steps * w.B * w.k, w.target.V, device="cuda")
    emitted = [[] for _ in range(w.B)]
    for st in range(steps):
        d = eng.spec_draft(ids, w.B, w.k)
        sl = slice(st * w.B * w.k, (st + 1) * w.B * w.k)
        eng.spec_inject_drafts(ids, d, ref, alpha, eng._in("dr", draws[sl].contiguous()),
                               eng._in("of", offs[sl].contiguous()))
        out, ne = eng.spec_verify(ids, d)
        eng.sync()
        for b in range(w.B):
            n = int(ne[b])
            assert 1 <= n <= w.k + 1
            emitted[b] += out[b, :n].cpu().tolist()
    for b in range(w.B):
        assert emitted[b] == greedy[b, 1:1 + len(emitted[b])].tolist(), (name, b)
    eng.close()
