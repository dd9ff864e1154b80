"""Pins of the oracle's lenient verify (CPU only): a draft is kept while it
ranks among the target's top-m tokens of its row ("Accelerating Gemini Nano on
Pixel with frozen multi-token prediction" (ai-news-spoon), "Future directions":
relaxing the strict draft/verification token match; the rule is this
repository's reading).

* rank: against a stable library sort of the binary32 logits by (logit
  descending, index ascending), with ties planted;
* top_m = 1 is the greedy accept, exactly (tokens, counts, cache state);
* top_m = vocabulary accepts every draft and ends with the target's choice at
  the last row;
* drafts picked at known ranks (teacher-forced rows) are accepted exactly up to
  the first one ranked m or worse;
* 1..k+1 tokens per step."""
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


def _library_rank(logits, tok):
    f = np.asarray(logits, np.float64).astype(np.float32)
    order = np.lexsort((np.arange(len(f)), -f.astype(np.float64)))   # logit desc, index asc
    return int(np.nonzero(order == tok)[0][0])


def test_rank_matches_library_sort_with_ties():
    rng = np.random.default_rng(3)
    lg = rng.standard_normal(200)
    lg[[10, 20, 30]] = lg[5]                 # exact ties
    lg[40] = np.nextafter(lg[5], np.inf)     # differs only in double: equal as binary32
    for tok in [5, 10, 20, 30, 40, 0, 199, int(np.argmax(lg))]:
        assert oracle.rank_f32(lg, tok) == _library_rank(lg, tok)


def _drafts_at_ranks(T, s, ranks):
    """Draft j = the token ranked ranks[j] at row j, rows teacher-forced on the
    drafts before them."""
    d = []
    for r in ranks:
        _, _, _, lg = oracle.forward(T, s.clone(), [s.pending] + d, want_logits=True)
        row = lg[len(d)].astype(np.float32).astype(np.float64)
        order = np.lexsort((np.arange(len(row)), -row))
        d.append(int(order[r]))
    return d


def test_top1_is_greedy_accept(tiny):
    w, T, s0 = tiny
    G, _ = oracle.greedy(T, s0.clone(), 4)
    for drafts in ([G[0], G[1], 7], [G[0], G[1], G[2]], [5, 6, 7], _drafts_at_ranks(T, s0, [0, 1, 0])):
        a, b = s0.clone(), s0.clone()
        e1, _ = oracle.verify(T, a, drafts)
        e2, _, _ = oracle.verify_topm(T, b, drafts, 1)
        assert list(e1) == list(e2)
        assert (a.len, a.pending) == (b.len, b.pending)
        assert np.array_equal(a.hid, b.hid) and np.array_equal(a.kv, b.kv)


def test_whole_vocabulary_accepts_everything(tiny):
    w, T, s0 = tiny
    drafts = [11, 2222, 3333]
    s = s0.clone()
    em, _, _ = oracle.verify_topm(T, s, drafts, w.target.V)
    am, _, _, _ = oracle.forward(T, s0.clone(), [s0.pending] + drafts)
    assert list(em) == drafts + [int(am[-1])]
    assert s.len == s0.len + 4


@pytest.mark.parametrize("ranks,m,A", [
    ([1, 0, 2], 2, 2),
    ([1, 1, 1], 2, 3),
    ([0, 3, 0], 3, 1),
    ([4, 0, 0], 4, 0),
    ([2, 2, 2], 3, 3),
])
def test_accept_up_to_first_draft_outside_top_m(tiny, ranks, m, A):
    w, T, s0 = tiny
    drafts = _drafts_at_ranks(T, s0, ranks)
    s = s0.clone()
    em, mg, dec = oracle.verify_topm(T, s, drafts, m)
    assert 1 <= len(em) <= len(drafts) + 1
    assert len(em) == A + 1
    assert list(em[:A]) == drafts[:A]
    am, _, _, _ = oracle.forward(T, s0.clone(), [s0.pending] + drafts)
    assert em[A] == am[A]
    assert s.len == s0.len + A + 1 and s.pending == em[A]
    assert np.all(dec[:A] >= 0) and (A == len(drafts) or dec[A] >= 0)
