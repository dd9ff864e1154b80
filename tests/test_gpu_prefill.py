"""Long prompts: the target processes the whole context before drafting
starts, the drafter has no prefill of its own ("Accelerating Gemini Nano on
Pixel with frozen multi-token prediction" (ai-news-spoon), "Zero-copy
architecture"). spec_prefill takes a prompt longer than one target pass and
runs it as consecutive causal passes (each pass's rows attend to the cached
keys of the passes before it). Checked against the oracle's one-pass prefill
of the whole prompt: the pending token, the hidden state, and then greedy
decoding from the new state (which reads every cached position)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import MARGIN, TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]
E2B_4L = dataclasses.replace(configs.E2B, L=4)   # E2B shapes (d 1536, GQA 12/4, head_dim 128), 4 layers


def _shapes(name):
    if name == "tiny_f32":
        return W.target, W.drafter
    if name == "tiny_bf16":
        return (dataclasses.replace(W.target, wdtype=configs.BF16, kvdtype=configs.BF16),
                dataclasses.replace(W.drafter, wdtype=configs.BF16))
    return E2B_4L, configs.WORKLOADS["e2b_bf16_b1_ctx2048_k3"].drafter


@pytest.mark.parametrize("name,plen,B", [("tiny_f32", 512, 1), ("tiny_bf16", 512, 1), ("tiny_bf16", 300, 2),
                                         ("e2b_4layer", 200, 1)])
def test_long_prompt_matches_oracle(name, plen, B):
    tshape, dshape = _shapes(name)
    dshape = dataclasses.replace(dshape, bh=tshape.d)
    tw = synth.make_target(tshape, device="cuda")
    dw = synth.make_drafter(dshape, device="cuda")
    cap = plen + 64
    eng = binding.Engine(tw, dw, n_slots=B, B_max=B, rows_max=plen, max_ctx=cap, shuffle_pages=True)
    prompts = torch.stack([synth.make_tokens(plen, tshape.V, seed=synth.SEED_TOKENS + b) for b in range(B)])
    ids = eng.seq_ids(list(range(B)))
    eng.spec_prefill(ids, eng._in("prompts", prompts.cuda()))
    eng.sync()
    seq_len, pending, hid = eng.seq_len.cpu().clone(), eng.pending.cpu().clone(), eng.hid.cpu().clone()
    toks = [[] for _ in range(B)]
    for _ in range(6):
        t = eng.spec_decode(ids, B).cpu()
        for b in range(B):
            toks[b].append(int(t[b]))
    eng.sync()
    T = oracle.Target(tw)
    tol = TOL[tshape.wdtype]
    for b in range(B):
        s = oracle.Seq(T, cap)
        mlast = oracle.prefill(T, s, prompts[b].numpy())
        assert int(seq_len[b]) == plen
        assert_rows_close(hid[b:b + 1].numpy(), s.hid[None], tol, "%s prompt hidden %d" % (name, b))
        if mlast > MARGIN:
            assert int(pending[b]) == s.pending
            G, gm = oracle.greedy(T, s, 6)
            compare_tokens(toks[b], G, gm)
    eng.close()
