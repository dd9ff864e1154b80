"""GPU parity of the lenient verify (spec_verify_topm): drafts are kept while
each ranks among the target's top-m tokens of its row ("Accelerating Gemini
Nano on Pixel with frozen multi-token prediction" (ai-news-spoon), "Future
directions": relaxing the strict draft/verification token match; the rule is
this repository's reading).

Drafts are picked at known ranks with the oracle's teacher-forced rows (so the
expected accept count is known), verified on the GPU, and compared with the
oracle's lenient verify: emitted tokens, counts and the slot state, wherever
the oracle's decision is more than 0.05 of logit away from flipping. The
cache rows of accepted non-greedy drafts are then exercised by plain greedy
decoding from the new state on both sides."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import MARGIN, TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]


def _drafts_at_ranks(T, s, ranks):
    d = []
    for r in ranks:
        _, _, _, lg = oracle.forward(T, s.clone(), [s.pending] + d, want_logits=True)
        row = lg[len(d)].astype(np.float32).astype(np.float64)
        d.append(int(np.lexsort((np.arange(len(row)), -row))[r]))
    return d


def _setup(tshape, dshape, ctx_prompt=True, w=None):
    tw = synth.make_target(tshape, device="cuda")
    dw = synth.make_drafter(dshape, device="cuda")
    T = oracle.Target(tw)
    eng = binding.Engine(tw, dw, n_slots=1, B_max=1, rows_max=64, max_ctx=512, shuffle_pages=True)
    prompt = synth.make_tokens(64, tshape.V)
    ids = eng.seq_ids([0])
    eng.spec_prefill(ids, eng._in("prompt", prompt.view(1, -1).cuda()))
    eng.sync()
    s = oracle.Seq(T, 512)
    oracle.prefill(T, s, prompt.numpy())
    return tw, T, eng, ids, s


@pytest.mark.parametrize("dt", [configs.F32, configs.BF16])
@pytest.mark.parametrize("ranks,m", [([1, 0, 2], 2), ([1, 1, 1], 2), ([0, 3, 0], 3), ([0, 0, 0], 1), ([2, 0, 1], 1)])
def test_topm_verify_matches_oracle(dt, ranks, m):
    tshape = W.target if dt == configs.F32 else dataclasses.replace(W.target, wdtype=dt, kvdtype=configs.BF16)
    dshape = W.drafter if dt == configs.F32 else dataclasses.replace(W.drafter, wdtype=dt)
    tw, T, eng, ids, s0 = _setup(tshape, dshape)
    drafts = _drafts_at_ranks(T, s0, ranks)
    d = eng._in("drafts", torch.tensor([drafts], dtype=torch.int32).cuda())
    logits = torch.empty((len(drafts) + 1, tshape.V), dtype=torch.float32, device="cuda")
    out, ne = eng.spec_verify_topm(ids, d, m, logits)
    eng.sync()
    out, ne = out.clone(), ne.clone()
    s = s0.clone()
    em, mg, dec = oracle.verify_topm(T, s, drafts, m)
    _, _, _, lg = oracle.forward(T, s0.clone(), [s0.pending] + drafts, want_logits=True)
    assert_rows_close(logits.cpu().numpy(), lg, TOL[tshape.wdtype], "lenient verify logits")
    n = int(ne[0])
    A = len(em) - 1
    st = eng.spec_stats(0)
    assert st.passes == 1 and st.accepted == n - 1 and st.emitted == n
    if np.all(dec[:min(A + 1, len(drafts))] > MARGIN) and mg[A] > MARGIN:
        assert n == len(em) and list(out[0, :n].cpu().numpy()) == list(em)
        assert int(eng.seq_len[0]) == s.len and int(eng.pending[0]) == s.pending
        assert_rows_close(eng.hid[0:1].cpu().numpy(), s.hid[None], TOL[tshape.wdtype], "hidden after lenient")
        # the committed cache rows (accepted drafts included) drive later decoding
        toks = [int(eng.spec_decode(ids, 1)[0]) for _ in range(6)]
        eng.sync()
        G, gm = oracle.greedy(T, s, 6)
        compare_tokens(toks, G, gm)
    assert 1 <= n <= len(drafts) + 1
    assert np.all(out[0, n:].cpu().numpy() == -1)
    eng.close()


def test_topm_one_equals_spec_verify_on_gpu():
    """top_m = 1 reproduces spec_verify's greedy accept bit for bit."""
    tshape = dataclasses.replace(W.target, wdtype=configs.BF16, kvdtype=configs.BF16)
    dshape = dataclasses.replace(W.drafter, wdtype=configs.BF16)
    tw, T, eng, ids, s0 = _setup(tshape, dshape)
    saved = [x.clone() for x in (eng.seq_len, eng.pending, eng.hid, eng.stats)]
    drafts = _drafts_at_ranks(T, s0, [0, 0, 1])
    d = eng._in("drafts", torch.tensor([drafts], dtype=torch.int32).cuda())
    o1, n1 = eng.spec_verify(ids, d)
    o1, n1 = o1.clone(), n1.clone()
    eng.sync()
    st1 = [x.clone() for x in (eng.seq_len, eng.pending, eng.hid)]
    for dst, src in zip((eng.seq_len, eng.pending, eng.hid, eng.stats), saved):
        dst.copy_(src)
    o2, n2 = eng.spec_verify_topm(ids, d, 1)
    eng.sync()
    assert torch.equal(o1, o2) and torch.equal(n1, n2)
    for a, b in zip(st1, (eng.seq_len, eng.pending, eng.hid)):
        assert torch.equal(a, b)
    eng.close()
