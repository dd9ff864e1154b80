"""Failure detection through the C ABI, in the forms that fault no GPU.

* Invalid calls are refused on the host with SPEC_EINVAL / SPEC_ESTATE before
  anything is launched, and leave the slot state untouched.
* A sequence whose committed length the caller set past its pages: the
  device-side bounds checks skip every out-of-range cache access, record the
  violation in the context's error word, and the accept step then leaves the
  slot state as it was; spec_sync reports SPEC_ECAPACITY (and clears the word).
* A draft token outside the vocabulary: recorded on the device, reported by
  spec_sync as SPEC_EINVAL, state unchanged.
* A bounded device wait that runs out: a test-only option makes the split
  merge of the tensor-core attention wait for one arrival more than there are
  splits (a count nothing completes); after about a second the wait gives up,
  the launch records a timeout and the pass commits nothing; spec_sync
  reports SPEC_ETIMEOUT.
After each failure the same context serves a correct pass (checked against the
oracle), so the context stays usable."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import TOL, assert_rows_close

pytestmark = pytest.mark.gpu
W = configs.WORKLOADS["tiny_f32_b1_k3"]


@pytest.fixture(scope="module", params=[configs.F32, configs.BF16])
def setup(request):
    import dataclasses
    t = W.target if request.param == configs.F32 else dataclasses.replace(W.target, wdtype=configs.BF16,
                                                                          kvdtype=configs.BF16)
    d = W.drafter if request.param == configs.F32 else dataclasses.replace(W.drafter, wdtype=configs.BF16)
    tw = synth.make_target(t, device="cuda")
    dw = synth.make_drafter(d, device="cuda")
    prompt = synth.make_tokens(64, t.V)
    T = oracle.Target(tw)
    s0 = oracle.Seq(T, 256)
    oracle.prefill(T, s0, prompt.numpy())
    return tw, dw, prompt, T, s0


def _engine(setup, drafter=True):
    tw, dw, prompt, T, s0 = setup
    eng = binding.Engine(tw, dw if drafter else None, n_slots=2, B_max=2, rows_max=64, max_ctx=128,
                         shuffle_pages=True)
    ids = eng.seq_ids([0])
    eng.spec_prefill(ids, eng._in("prompt", prompt.view(1, -1).cuda()))
    eng.sync()
    return eng, ids


def _state(eng):
    torch.cuda.synchronize()
    return [x.clone().cpu() for x in (eng.seq_len, eng.pending, eng.hid, eng.stats)]


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def _verify_matches_oracle(eng, ids, setup):
    tw, dw, prompt, T, s0 = setup
    G, _ = oracle.greedy(T, s0.clone(), 3)
    drafts = [int(G[0]), int(G[1]), 5]
    d = eng._in("drafts", torch.tensor([drafts], dtype=torch.int32).cuda())
    logits = torch.empty((4, tw.shape.V), dtype=torch.float32, device="cuda")
    eng.spec_verify(ids, d, logits)
    eng.sync()
    _, _, _, lg = oracle.forward(T, s0.clone(), [s0.pending] + drafts, want_logits=True)
    assert_rows_close(logits.cpu().numpy(), lg, TOL[tw.shape.wdtype], "verify after a failure")


def test_invalid_calls_refused_on_host(setup):
    eng, ids = _engine(setup)
    L = binding.lib()
    st = eng.stream.cuda_stream
    before = _state(eng)
    out = torch.zeros((2, 9), dtype=torch.int32, device="cuda")
    ne = torch.zeros((2,), dtype=torch.int32, device="cuda")
    dr = torch.zeros((2, 8), dtype=torch.int32, device="cuda")
    p = lambda t: t.data_ptr()
    E = binding.SPEC_EINVAL
    assert L.spec_verify(eng.ctx, 1, p(ids), 64, p(dr), p(out), p(ne), None, st) == E     # k + 1 > rows_max
    assert L.spec_verify(eng.ctx, 1, p(ids), -1, p(dr), p(out), p(ne), None, st) == E
    assert L.spec_verify(eng.ctx, 1, p(ids), 3, None, p(out), p(ne), None, st) == E        # no drafts
    assert L.spec_verify(eng.ctx, 1, p(ids), 3, p(dr), None, p(ne), None, st) == E         # no output
    assert L.spec_verify(eng.ctx, 3, p(ids), 3, p(dr), p(out), p(ne), None, st) == E       # B > B_max
    assert L.spec_verify(eng.ctx, 0, p(ids), 3, p(dr), p(out), p(ne), None, st) == E
    assert L.spec_verify(eng.ctx, 1, None, 3, p(dr), p(out), p(ne), None, st) == E
    assert L.spec_draft(eng.ctx, 1, p(ids), 0, p(dr), st) == E
    assert L.spec_draft(eng.ctx, 1, p(ids), 17, p(dr), st) == E
    assert L.spec_prefill(eng.ctx, 1, p(ids), 65, p(dr), st) == E                          # R > rows_max
    assert L.spec_decode(eng.ctx, 1, p(ids), None, st) == E
    assert L.spec_stats(eng.ctx, 5, None, st) == E
    assert _same(before, _state(eng))
    assert L.spec_sync(eng.ctx, st) == binding.SPEC_OK
    _verify_matches_oracle(eng, ids, setup)
    eng.close()
    nod, ids2 = _engine(setup, drafter=False)
    assert L.spec_draft(nod.ctx, 1, p(ids2), 3, p(dr), nod.stream.cuda_stream) == binding.SPEC_ESTATE
    nod.close()


def test_over_capacity_length_is_caught_on_device(setup):
    """128 positions of pages per sequence; the caller sets seq_len to 126 and
    verifies 4 rows (positions 126..129)."""
    eng, ids = _engine(setup)
    good = _state(eng)
    eng.seq_len[0] = 126
    torch.cuda.synchronize()
    before = _state(eng)
    d = eng._in("drafts", torch.tensor([[1, 2, 3]], dtype=torch.int32).cuda())
    eng.spec_verify(ids, d)
    rc = binding.lib().spec_sync(eng.ctx, eng.stream.cuda_stream)
    assert rc == binding.SPEC_ECAPACITY
    assert _same(before, _state(eng))                  # no commit, no stats
    assert binding.lib().spec_sync(eng.ctx, eng.stream.cuda_stream) == binding.SPEC_OK   # word cleared
    # the caller restores its saved state; the context serves a correct pass
    for dst, src in zip((eng.seq_len, eng.pending, eng.hid, eng.stats), good):
        dst.copy_(src.cuda())
    _verify_matches_oracle(eng, ids, setup)
    eng.close()


def test_token_outside_vocabulary_is_caught_on_device(setup):
    eng, ids = _engine(setup)
    before = _state(eng)
    V = setup[0].shape.V
    d = eng._in("drafts", torch.tensor([[1, V + 7, 3]], dtype=torch.int32).cuda())
    eng.spec_verify(ids, d)
    assert binding.lib().spec_sync(eng.ctx, eng.stream.cuda_stream) == binding.SPEC_EINVAL
    assert _same(before, _state(eng))
    _verify_matches_oracle(eng, ids, setup)
    eng.close()


HD128 = configs.TargetShape(L=2, d=256, nq=4, nkv=2, hd=128, ff=512, V=1024, wdtype=configs.BF16,
                            kvdtype=configs.BF16, wstd=0.02)
HD128_DRAFTER = configs.DrafterShape(L=1, h=64, bh=256, ff=256, nq=4, hd=128, nkv=2, V=1024,
                                     wdtype=configs.BF16, wstd=0.02, clustered=False)


def test_attention_wait_that_runs_out_reports_timeout():
    """A 300-position context splits each (sequence, KV head) over several
    CTAs of the tensor-core attention, whose merge then waits on the pair's
    arrivals."""
    tw = synth.make_target(HD128, device="cuda")
    dw = synth.make_drafter(HD128_DRAFTER, device="cuda")
    ctx = 300
    eng = binding.Engine(tw, dw, n_slots=1, B_max=1, rows_max=8, max_ctx=512, shuffle_pages=True)
    kv = synth.make_prefilled_kv(HD128, ctx - 1, device="cuda")
    eng.load_prefilled(0, kv)
    first = synth.make_tokens(1, HD128.V, device="cuda").view(1, 1)
    ids = eng.seq_ids([0])
    eng.spec_prefill(ids, eng._in("first", first))
    eng.sync()
    before = _state(eng)
    drafts = [3, 4, 5]
    d = eng._in("drafts", torch.tensor([drafts], dtype=torch.int32).cuda())
    eng.set_option(binding.SPEC_OPT_TEST_ATTN_WAIT, 1)
    eng.spec_verify(ids, d)
    assert binding.lib().spec_sync(eng.ctx, eng.stream.cuda_stream) == binding.SPEC_ETIMEOUT
    assert _same(before, _state(eng))
    eng.set_option(binding.SPEC_OPT_TEST_ATTN_WAIT, 0)
    logits = torch.empty((4, HD128.V), dtype=torch.float32, device="cuda")
    eng.spec_verify(ids, d, logits)
    eng.sync()
    T = oracle.Target(tw)
    s = oracle.Seq(T, 512)
    s.load_prefilled(kv.cpu())
    oracle.prefill(T, s, first.cpu().numpy()[0])
    _, _, _, lg = oracle.forward(T, s, [s.pending] + drafts, want_logits=True)
    assert_rows_close(logits.cpu().numpy(), lg, TOL[configs.BF16], "verify after a timeout")
    eng.close()
