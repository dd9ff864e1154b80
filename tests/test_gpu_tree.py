"""GPU parity of tree verify (spec_verify_tree): a tree of draft nodes rooted
at the pending token verified in one pass with a tree attention mask, greedy
accept along the matching branch, and the accepted nodes' keys and values moved
to consecutive positions ("Accelerating Gemini Nano on Pixel with frozen
multi-token prediction" (ai-news-spoon), "Future directions": branching
possibilities explored in parallel; the rule is this repository's reading).

Trees are built from the oracle's greedy tokens (the greedy branch among wrong
siblings, a star, a chain, a tree whose match sits below a wrong node) on the
fp32 model (CUDA-core attention), the bf16 model (register-fragment
attention, head_dim 64) and an E2B-shaped model (tcgen05 attention, head_dim
128). Emitted tokens, counts, the slot state and the hidden state are compared
with the oracle's tree verify; greedy decoding afterwards reads the moved cache
rows and is compared with the oracle's."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import MARGIN, TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]
E2B_4L = dataclasses.replace(configs.E2B, L=4)


def _shapes(name):
    if name == "tiny_f32":
        return W.target, W.drafter
    if name == "tiny_bf16":
        return (dataclasses.replace(W.target, wdtype=configs.BF16, kvdtype=configs.BF16),
                dataclasses.replace(W.drafter, wdtype=configs.BF16))
    d = configs.WORKLOADS["e2b_bf16_b1_ctx2048_k3"].drafter
    return E2B_4L, dataclasses.replace(d, bh=E2B_4L.d)


def _trees(G, V):
    bad = lambda x, o: int((x + o) % V)
    return {
        "greedy_branch": ([bad(G[0], 1), G[0], bad(G[1], 2), G[1], bad(G[1], 3), G[2], G[2]],
                          [-1, -1, 1, 1, 1, 3, 0]),
        "star": ([bad(G[0], 5), G[0], bad(G[0], 9), G[0]], [-1, -1, -1, -1]),
        "chain": ([G[0], G[1], bad(G[2], 4)], [-1, 0, 1]),
        "below_wrong": ([bad(G[0], 1), bad(G[0], 2), G[0]], [-1, -1, 0]),
    }


@pytest.mark.parametrize("name", ["tiny_f32", "tiny_bf16", "e2b_4layer"])
@pytest.mark.parametrize("tree", ["greedy_branch", "star", "chain", "below_wrong"])
def test_tree_verify_matches_oracle(name, tree):
    tshape, dshape = _shapes(name)
    tw = synth.make_target(tshape, device="cuda")
    dw = synth.make_drafter(dshape, device="cuda")
    T = oracle.Target(tw)
    cap = 256
    eng = binding.Engine(tw, dw, n_slots=1, B_max=1, rows_max=128, max_ctx=cap, shuffle_pages=True)
    prompt = synth.make_tokens(70, tshape.V)
    ids = eng.seq_ids([0])
    eng.spec_prefill(ids, eng._in("prompt", prompt.view(1, -1).cuda()))
    eng.sync()
    s0 = oracle.Seq(T, cap)
    oracle.prefill(T, s0, prompt.numpy())
    G, gm = oracle.greedy(T, s0.clone(), 4)
    tokens, parents = _trees(G, tshape.V)[tree]
    n = len(tokens)
    out, ne = eng.spec_verify_tree(ids, eng._in("tt", torch.tensor([tokens], dtype=torch.int32).cuda()),
                                   eng._in("tp", torch.tensor([parents], dtype=torch.int32).cuda()))
    eng.sync()
    out, ne = out.clone().cpu(), ne.clone().cpu()
    st = eng.spec_stats(0)
    seq_len, pending, hid = int(eng.seq_len[0]), int(eng.pending[0]), eng.hid.cpu().clone()
    s = s0.clone()
    em, mg = oracle.verify_tree(T, s, tokens, parents)
    k = int(ne[0])
    assert 1 <= k <= n + 1 and np.all(out[0, k:].numpy() == -1)
    assert st.passes == 1 and st.emitted == k and st.accepted == k - 1 and st.drafted == n
    if np.all(mg > MARGIN):
        assert list(out[0, :k].numpy()) == list(em)
        assert seq_len == s.len and pending == s.pending
        assert_rows_close(hid[0:1].numpy(), s.hid[None], TOL[tshape.wdtype], "%s %s hidden" % (name, tree))
        toks = [int(eng.spec_decode(ids, 1)[0]) for _ in range(6)]
        eng.sync()
        Gn, gmn = oracle.greedy(T, s, 6)
        compare_tokens(toks, Gn, gmn)
    eng.close()


def test_tree_batch_two_sequences():
    """Two sequences with different trees in one pass (tcgen05 attention)."""
    tshape, dshape = _shapes("e2b_4layer")
    tw = synth.make_target(tshape, device="cuda")
    dw = synth.make_drafter(dshape, device="cuda")
    T = oracle.Target(tw)
    cap = 256
    eng = binding.Engine(tw, dw, n_slots=2, B_max=2, rows_max=128, max_ctx=cap, shuffle_pages=True)
    prompts = torch.stack([synth.make_tokens(70, tshape.V, seed=synth.SEED_TOKENS + b) for b in range(2)])
    ids = eng.seq_ids([0, 1])
    eng.spec_prefill(ids, eng._in("prompts", prompts.cuda()))
    eng.sync()
    seqs, trees = [], []
    for b, kind in enumerate(["greedy_branch", "star"]):
        s = oracle.Seq(T, cap)
        oracle.prefill(T, s, prompts[b].numpy())
        G, _ = oracle.greedy(T, s.clone(), 4)
        tk, pa = _trees(G, tshape.V)[kind]
        tk, pa = (tk + [0] * 7)[:7], (pa + [-1] * 7)[:7]   # both padded to 7 nodes
        seqs.append(s)
        trees.append((tk, pa))
    out, ne = eng.spec_verify_tree(ids, eng._in("tt", torch.tensor([t[0] for t in trees], dtype=torch.int32).cuda()),
                                   eng._in("tp", torch.tensor([t[1] for t in trees], dtype=torch.int32).cuda()))
    eng.sync()
    for b in range(2):
        em, mg = oracle.verify_tree(T, seqs[b], *trees[b])
        k = int(ne[b])
        if np.all(mg > MARGIN):
            assert list(out[b, :k].cpu().numpy()) == list(em)
            assert int(eng.seq_len[b]) == seqs[b].len and int(eng.pending[b]) == seqs[b].pending
    eng.close()
