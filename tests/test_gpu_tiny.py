"""GPU parity on the tiny workload (2-layer d=256 target, 1-layer width-64
drafter, vocabulary 4096, 64-token prompt, k = 3), through the C ABI. The
fp32 model is the configured workload; the same shapes with bf16 and Q4_0
weights (bf16 KV) exercise the other weight paths end to end."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import MARGIN, TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]
CAP = 512


def _variant(dt):
    if dt == configs.F32:
        return W.target, W.drafter
    t = dataclasses.replace(W.target, wdtype=dt, kvdtype=configs.BF16)
    d = dataclasses.replace(W.drafter, wdtype=dt)
    return t, d


@pytest.fixture(scope="module", params=[configs.F32, configs.BF16, configs.Q4_0])
def models(request):
    tshape, dshape = _variant(request.param)
    tw = synth.make_target(tshape, device="cuda")
    dw = synth.make_drafter(dshape, device="cuda")
    prompt = synth.make_tokens(64, W.target.V)
    T, D = oracle.Target(tw), oracle.Drafter(dw)
    s0 = oracle.Seq(T, CAP)
    oracle.prefill(T, s0, prompt.numpy())
    return tw, dw, T, D, prompt, s0


def _engine(tw, dw, graphs=True):
    return binding.Engine(tw, dw, n_slots=2, B_max=2, rows_max=64, max_ctx=CAP, shuffle_pages=True,
                          graphs=graphs)


def _prefilled(models, graphs=True):
    tw, dw, T, D, prompt, s0 = models
    eng = _engine(tw, dw, graphs)
    ids = eng.seq_ids([1])
    eng.spec_prefill(ids, eng._in("prompt", prompt.view(1, -1).cuda()))
    eng.sync()
    return eng, ids


def test_prefill_two_sequences_matches_oracle(models):
    """Two 64-token prompts in one prefill: 128 rows, which the bf16 / Q4_0
    projections run as two 64-row passes (the tail after the second)."""
    tw, dw, T, D, prompt, s0 = models
    eng = _engine(tw, dw)
    ids = eng.seq_ids([0, 1])
    second = synth.make_tokens(64, W.target.V, seed=synth.SEED_KV + 7)
    both = torch.stack([second, prompt]).cuda()
    eng.spec_prefill(ids, eng._in("prompts", both))
    eng.sync()
    s1 = oracle.Seq(T, CAP)
    m1 = oracle.prefill(T, s1, second.numpy())
    tol = TOL[tw.shape.wdtype]
    for slot, ref in ((0, s1), (1, s0)):
        assert int(eng.seq_len[slot]) == 64
        assert_rows_close(eng.hid[slot:slot + 1].cpu().numpy(), ref.hid[None], tol, "prefill hidden %d" % slot)
    assert int(eng.pending[1]) == s0.pending
    if m1 > MARGIN:
        assert int(eng.pending[0]) == s1.pending
    eng.close()


def test_prefill_matches_oracle(models):
    tw, dw, T, D, prompt, s0 = models
    eng, ids = _prefilled(models)
    assert int(eng.seq_len[1]) == 64
    assert int(eng.pending[1]) == s0.pending
    assert_rows_close(eng.hid[1:2].cpu().numpy(), s0.hid[None], TOL[tw.shape.wdtype], "prefill hidden")


@pytest.mark.parametrize("graphs", [True, False])
def test_verify_logits_and_accept_match_oracle(models, graphs):
    """Verify pass logits and accepted tokens, with and without CUDA graphs."""
    tw, dw, T, D, prompt, s0 = models
    eng, ids = _prefilled(models, graphs)
    eng.close()
    G, _ = oracle.greedy(T, s0.clone(), 8)
    for drafts in ([G[0], G[1], 7], [G[0], G[1], G[2]], [5, 6, 7]):
        eng2, ids2 = _prefilled(models, graphs)
        d = eng2._in("drafts", torch.tensor([drafts], dtype=torch.int32).cuda())
        logits = torch.empty((4, W.target.V), dtype=torch.float32, device="cuda")
        out, ne = eng2.spec_verify(ids2, d, logits)
        eng2.sync()
        s = s0.clone()
        am, mg, hid, lg = oracle.forward(T, s.clone(), [s.pending] + list(drafts), want_logits=True)
        assert_rows_close(logits.cpu().numpy(), lg, TOL[tw.shape.wdtype], "verify logits")
        em, _ = oracle.verify(T, s, np.array(drafts))
        n = int(ne[0])
        got = out[0, :n].cpu().numpy()
        if np.all(mg > MARGIN):
            assert n == len(em) and np.array_equal(got, em)
            assert int(eng2.seq_len[1]) == s.len and int(eng2.pending[1]) == s.pending
        assert np.all(out[0, n:].cpu().numpy() == -1)
        eng2.close()


def test_greedy_decode_matches_oracle(models):
    tw, dw, T, D, prompt, s0 = models
    eng, ids = _prefilled(models)
    toks = []
    for _ in range(24):
        toks.append(int(eng.spec_decode(ids, 1)[0]))
    eng.sync()
    G, mg = oracle.greedy(T, s0.clone(), 24)
    n = compare_tokens(toks, G, mg)
    assert n >= 1


@pytest.mark.parametrize("alpha", [0.0, 0.5, 0.8, 1.0])
def test_speculative_output_equals_greedy(models, alpha):
    """The pages' invariant on the GPU: tokens emitted by speculative steps
    equal plain greedy decoding, bit for bit (same kernels, row results that
    do not depend on the number of verified rows), and the oracle's greedy
    sequence under the margin rule."""
    tw, dw, T, D, prompt, s0 = models
    k, steps = W.k, 16
    eng, ids = _prefilled(models)
    n_ref = 64 + steps * (k + 1) + k + 2
    ref = torch.zeros((2, n_ref + 8), dtype=torch.int32, device="cuda")
    greedy = []
    for _ in range(steps * (k + 1) + k + 1):
        greedy.append(int(eng.spec_decode(ids, 1)[0]))
    eng.sync()
    # ref[slot][pos] = token at absolute position pos (pending sits at 64)
    ref[1, 64] = int(s0.pending)
    ref[1, 65:65 + len(greedy)] = torch.tensor(greedy, dtype=torch.int32)
    eng2, ids2 = _prefilled(models)
    draws = synth.make_alpha_draws(steps * k, device="cuda")
    offs = synth.make_wrong_offsets(steps * k, W.target.V, device="cuda")
    emitted, per_step = [], []
    for st in range(steps):
        d = eng2.spec_draft(ids2, 1, k)
        dr = eng2._in("draws", draws[st * k:(st + 1) * k].contiguous())
        of = eng2._in("offs", offs[st * k:(st + 1) * k].contiguous())
        eng2.spec_inject_drafts(ids2, d, ref, alpha, dr, of)
        out, ne = eng2.spec_verify(ids2, d)
        eng2.sync()
        n = int(ne[0])
        assert 1 <= n <= k + 1
        per_step.append(n)
        emitted += out[0, :n].cpu().tolist()
    assert emitted == greedy[:len(emitted)]
    if alpha == 1.0:
        assert per_step == [k + 1] * steps
    if alpha == 0.0:
        assert per_step == [1] * steps
    G, mg = oracle.greedy(T, s0.clone(), len(emitted))
    compare_tokens(emitted, G, mg)
    st = eng2.spec_stats(1)
    assert st.passes == steps and st.emitted == sum(per_step)
    assert st.accepted == st.emitted - st.passes and st.drafted == steps * k


def test_drafter_matches_oracle(models):
    """The k drafted tokens against the oracle's drafter (margin rule)."""
    tw, dw, T, D, prompt, s0 = models
    eng, ids = _prefilled(models)
    d = eng.spec_draft(ids, 1, W.k)
    eng.sync()
    ref, mg = oracle.draft(T, D, s0.clone(), W.k)
    compare_tokens(d[0].cpu().numpy(), ref, mg)


def test_step_emits_greedy_tokens(models):
    tw, dw, T, D, prompt, s0 = models
    eng, ids = _prefilled(models)
    toks = []
    for _ in range(6):
        out, ne = eng.spec_step(ids, 1, W.k)
        eng.sync()
        toks += out[0, :int(ne[0])].cpu().tolist()
    G, mg = oracle.greedy(T, s0.clone(), len(toks))
    compare_tokens(toks, G, mg)
