"""Pins of the oracle's mixture-of-experts target (CPU only). The pages name a
26B mixture-of-experts target without its layer ("Gemma 4 acceleration: faster
inference with multi-token prediction drafters" (cafe.daangn.com), "MTP
drafter internal optimisations"); the reading here: router scores on the FFN's
normalised input, the top_k experts by score (ties to the lower id), softmax
weights over the chosen scores, gated-GELU experts.

* top-k selection against a stable library sort, ties included;
* one expert, top_k 1: exactly the dense layer with that expert's weights;
* every expert chosen: the layer output is the softmax-weighted sum of the
  experts' outputs, each expert's output taken from a dense one-expert model;
* identical experts: the output is that one expert's (weights sum to 1);
* speculative output equals greedy output on a mixture-of-experts target."""
import copy
import dataclasses

import numpy as np
import pytest

import oracle
from speculative_decoding_spec_gb300 import configs, synth

MOE = dataclasses.replace(configs.TINY_MOE, L=1, wstd=0.1)


def rms(x, g, eps=1e-6):
    return x / np.sqrt(np.mean(x * x) + eps) * g


def test_topk_matches_library_sort_with_ties():
    rng = np.random.default_rng(4)
    sc = rng.standard_normal(64)
    sc[[3, 7, 9]] = sc[40]
    sc[11] = np.nextafter(sc[40], np.inf)      # equal once rounded to binary32
    for k in (1, 4, 8, 20):
        idx, gap = oracle.topk_f32(sc, k)
        f = sc.astype(np.float32).astype(np.float64)
        want = np.lexsort((np.arange(64), -f))[:k]
        assert list(idx) == list(want)


def _dense_twin(tw, e):
    """A dense model whose FFN is expert e of layer 0."""
    shape = dataclasses.replace(tw.shape, n_experts=0, top_k=0, ff_e=0, ff=tw.shape.ff_e)
    d = copy.deepcopy(tw)
    d.shape = shape
    d.wgu = synth.WTensor(tw.wgu_e.dtype, 1, 2 * shape.ff, shape.d, tw.wgu_e.data[e:e + 1].clone())
    d.wdown = synth.WTensor(tw.wdown_e.dtype, 1, shape.d, shape.ff, tw.wdown_e.data[e:e + 1].clone())
    d.router = d.wgu_e = d.wdown_e = None
    return d


def _resid(tw, toks):
    T = oracle.Target(tw)
    return oracle.forward_resid(T, oracle.Seq(T, 16), toks)[4]


def test_single_expert_is_the_dense_layer():
    shape = dataclasses.replace(MOE, n_experts=1, top_k=1)
    tw = synth.make_target(shape)
    toks = np.array([3, 500, 77], np.int32)
    assert np.array_equal(_resid(tw, toks), _resid(_dense_twin(tw, 0), toks))


def test_all_experts_chosen_is_softmax_weighted_sum():
    shape = dataclasses.replace(MOE, n_experts=4, top_k=4)
    tw = synth.make_target(shape)
    tw.wo.data.zero_()                       # attention adds nothing: the FFN sees E[tok]
    toks = np.array([9, 1234], np.int32)
    got = _resid(tw, toks)
    E = tw.embed.data[0].double().numpy()
    want = []
    for r, t in enumerate(toks):
        xn = rms(E[t], tw.g_ffn[0].double().numpy())
        z = tw.router.data[0].double().numpy() @ xn
        w = np.exp(z - z.max())
        w /= w.sum()
        outs = []
        for e in range(4):
            dense = _dense_twin(tw, e)
            dense.wo.data.zero_()
            outs.append(_resid(dense, toks)[r] - E[t])
        want.append(E[t] + sum(w[e] * outs[e] for e in range(4)))
    assert np.abs(got - np.array(want)).max() / np.abs(np.array(want)).max() < 1e-12


def test_identical_experts_give_that_expert():
    shape = dataclasses.replace(MOE, n_experts=5, top_k=3)
    tw = synth.make_target(shape)
    tw.wgu_e.data[:] = tw.wgu_e.data[0:1].clone()
    tw.wdown_e.data[:] = tw.wdown_e.data[0:1].clone()
    toks = np.array([42, 4000], np.int32)
    a, b = _resid(tw, toks), _resid(_dense_twin(tw, 0), toks)
    assert np.abs(a - b).max() / np.abs(b).max() < 1e-13


def test_speculative_equals_greedy_on_moe_target():
    tw = synth.make_target(configs.TINY_MOE)
    T = oracle.Target(tw)
    s0 = oracle.Seq(T, 256)
    oracle.prefill(T, s0, synth.make_tokens(40, configs.TINY_MOE.V).numpy())
    G, _ = oracle.greedy(T, s0.clone(), 14)
    s, out = s0.clone(), []
    for st in range(5):
        n = len(out)
        d = [G[n], G[n + 1], 11] if st % 2 == 0 else [G[n], 5, 6]
        em, _ = oracle.verify(T, s, d)
        out += list(em)
    assert out == list(G[:len(out)])
