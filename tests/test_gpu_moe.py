"""GPU parity of the mixture-of-experts target on small models (the full-size
mixture-of-experts workload runs through the workload tests): a 64-token
prompt, a verify pass with drafts, and greedy decoding, against the oracle
(router scores, top-k routing with softmax weights, gated-GELU experts). fp32
and bf16 weights with head_dim 64, and a head_dim 128 model with 16 experts
(tensor-core attention)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import MARGIN, TOL, assert_rows_close, compare_tokens

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]
MOE_HD128 = dataclasses.replace(configs.TINY_MOE, d=512, nq=4, nkv=2, hd=128, n_experts=16, top_k=2, ff_e=512,
                                wdtype=configs.BF16, kvdtype=configs.BF16)


@pytest.mark.parametrize("name", ["f32", "bf16", "hd128"])
def test_moe_target_matches_oracle(name):
    if name == "f32":
        t = configs.TINY_MOE
    elif name == "bf16":
        t = dataclasses.replace(configs.TINY_MOE, wdtype=configs.BF16, kvdtype=configs.BF16)
    else:
        t = MOE_HD128
    dsh = dataclasses.replace(W.drafter, bh=t.d, nq=t.nq, hd=t.hd, nkv=t.nkv, wdtype=t.wdtype)
    tw = synth.make_target(t, device="cuda")
    dw = synth.make_drafter(dsh, device="cuda")
    eng = binding.Engine(tw, dw, n_slots=1, B_max=1, rows_max=64, max_ctx=256, shuffle_pages=True)
    prompt = synth.make_tokens(64, t.V)
    ids = eng.seq_ids([0])
    eng.spec_prefill(ids, eng._in("prompt", prompt.view(1, -1).cuda()))
    eng.sync()
    T = oracle.Target(tw)
    s0 = oracle.Seq(T, 256)
    mlast = oracle.prefill(T, s0, prompt.numpy())
    tol = TOL[t.wdtype]
    assert_rows_close(eng.hid[0:1].cpu().numpy(), s0.hid[None], tol, "moe %s prompt hidden" % name)
    if mlast > MARGIN:
        assert int(eng.pending[0]) == s0.pending
    G, gm = oracle.greedy(T, s0.clone(), 8)
    drafts = [int(G[0]), int(G[1]), 7]
    logits = torch.empty((4, t.V), dtype=torch.float32, device="cuda")
    out, ne = eng.spec_verify(ids, eng._in("d", torch.tensor([drafts], dtype=torch.int32).cuda()), logits)
    eng.sync()
    _, mg, _, lg = oracle.forward(T, s0.clone(), [s0.pending] + drafts, want_logits=True)
    assert_rows_close(logits.cpu().numpy(), lg, tol, "moe %s verify logits" % name)
    s = s0.clone()
    em, _ = oracle.verify(T, s, drafts)
    n = int(ne[0])
    compare_tokens(out[0, :n].cpu().numpy(), em, mg)
    toks = [int(eng.spec_decode(ids, 1)[0]) for _ in range(5)]
    eng.sync()
    if np.all(mg[:len(em)] > MARGIN) and n == len(em):
        Gs, gms = oracle.greedy(T, s, 5)
        compare_tokens(toks, Gs, gms)
    eng.close()
