"""Pins of the oracle's tree verify (CPU only): drafts form a tree rooted at
the pending token; greedy accept follows the matching child from the root
("Accelerating Gemini Nano on Pixel with frozen multi-token prediction"
(ai-news-spoon), "Future directions": branching possibilities explored in
parallel; the accept rule is this repository's reading).

* a chain is exactly the linear verify (tokens, state, cache);
* a tree holding the greedy path on some branch, among wrong siblings, emits
  exactly the greedy tokens along it and leaves the greedy decoder's state;
* a star (every node a child of the root) accepts the lowest-index node whose
  token is the target's choice, and only that one;
* nodes off the accepted path leave no trace in the committed cache."""
import numpy as np
import pytest

import oracle
from speculative_decoding_spec_gb300 import configs, synth


@pytest.fixture(scope="module")
def tiny():
    w = configs.WORKLOADS["tiny_f32_b1_k3"]
    T = oracle.Target(synth.make_target(w.target))
    s = oracle.Seq(T, 256)
    oracle.prefill(T, s, synth.make_tokens(64, w.target.V).numpy())
    return w, T, s


def _same_state(a, b):
    L = a.len
    return (a.len == b.len and a.pending == b.pending and np.array_equal(a.hid, b.hid)
            and np.array_equal(a.kv[:, :, :, :L], b.kv[:, :, :, :L]))


def test_chain_is_linear_verify(tiny):
    w, T, s0 = tiny
    G, _ = oracle.greedy(T, s0.clone(), 4)
    for drafts in ([G[0], G[1], 7], [G[0], G[1], G[2]], [5, 6, 7]):
        a, b = s0.clone(), s0.clone()
        e1, _ = oracle.verify(T, a, drafts)
        e2, _ = oracle.verify_tree(T, b, drafts, [-1, 0, 1])
        assert list(e1) == list(e2)
        assert _same_state(a, b)


def test_greedy_branch_among_wrong_siblings(tiny):
    w, T, s0 = tiny
    G, _ = oracle.greedy(T, s0.clone(), 4)
    V = w.target.V
    bad = lambda x, o: int((x + o) % V)
    # node: 0 bad, 1 G0 (root children); 2 bad, 3 G1, 4 bad (children of node 1);
    # 5 G2 (child of node 3); 6 G2 as a child of a wrong node
    tokens = [bad(G[0], 1), G[0], bad(G[1], 2), G[1], bad(G[1], 3), G[2], G[2]]
    parents = [-1, -1, 1, 1, 1, 3, 0]
    s = s0.clone()
    em, mg = oracle.verify_tree(T, s, tokens, parents)
    assert list(em) == list(G[:4])
    g = s0.clone()
    oracle.greedy(T, g, 4)
    assert _same_state(s, g)


def test_star_accepts_lowest_matching_child(tiny):
    w, T, s0 = tiny
    G, _ = oracle.greedy(T, s0.clone(), 2)
    V = w.target.V
    tokens = [int((G[0] + 5) % V), G[0], int((G[0] + 9) % V), G[0]]
    s = s0.clone()
    em, _ = oracle.verify_tree(T, s, tokens, [-1, -1, -1, -1])
    assert list(em) == list(G[:2])
    g = s0.clone()
    oracle.verify(T, g, [G[0]])
    assert _same_state(s, g)


def test_no_match_emits_root_choice(tiny):
    w, T, s0 = tiny
    G, _ = oracle.greedy(T, s0.clone(), 1)
    V = w.target.V
    tokens = [int((G[0] + 1) % V), int((G[0] + 2) % V), G[0]]
    s = s0.clone()
    em, _ = oracle.verify_tree(T, s, tokens, [-1, -1, 0])   # G0 only below a wrong node
    assert list(em) == [G[0]] and s.len == s0.len + 1
