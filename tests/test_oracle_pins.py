"""Closed-form pins of the oracle's composition (CPU only).

The single operations (RMSNorm, RoPE, GELU, attention, linear, argmax) are
pinned one by one elsewhere. These tests pin how the oracle's target forward
and drafter put them together, by zeroing chosen weights so that the model
reduces to something with an independent closed form:

* target, attention and FFN switched off (W_o = W_down = 0): the residual
  stream is the embedding row and the logits are E . N_final(E[tok]) (tied
  head, final RMSNorm with its gain, no embedding scale);
* queries switched off (W_q = 0): every score is 0, so each row's attention is
  the plain mean of the values of keys 0..pos (causal, the row's own key
  included, GQA head h reading KV head h / group);
* the FFN through the odd part of GELU, GELU(z) - GELU(-z) = z: flipping the
  sign of the gate rows changes the output by W_down((W_g xn) * (W_u xn)),
  which holds only for gate rows first, GELU on the gate and the FFN norm's
  own gain;
* RoPE inside attention through its complex form: with pair i of a head read
  as z = v[i] + 1j v[i + hd/2], a query at position p and a key at position
  p' score Re(sum_i z_q z_k* e^{1j (p - p') w_i}) / sqrt(hd), w_i =
  theta^(-2i/hd), which fixes every key's and query's absolute position;
* drafter: the same reductions for its input projection and recurrence
  (W_o' = W_down' = 0), its cross-attention over exactly the committed
  positions [0, len) of the target's last layer (W_q' = 0, garbage written
  past len), its query position len + j - 1 (complex RoPE form against the
  cached keys), and its FFN (odd GELU part).

Sources: the target layer and drafter step the oracle states ("Gemma 4's MTP
drafter explained" (molayo1419.me), "What is different about Gemma 4's
drafter?"; "Accelerating Gemini Nano on Pixel with frozen multi-token
prediction" (ai-news-spoon), "The late-exit strategy", "Zero-copy
architecture").
"""
import copy

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import configs, synth

SHAPE = configs.TargetShape(L=2, d=128, nq=4, nkv=2, hd=32, ff=256, V=512, wdtype=configs.F32,
                            kvdtype=configs.F32, wstd=0.05)
DSHAPE = configs.DrafterShape(L=2, h=64, bh=128, ff=256, nq=4, hd=32, nkv=2, V=512,
                              wdtype=configs.F32, wstd=0.05, clustered=False)
TOL = 1e-9


def rms(x, g, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(g, np.float64)


def f64(t):
    return t.detach().double().cpu().numpy()


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def target(shape=SHAPE, **zero):
    tw = synth.make_target(shape)
    tw = copy.deepcopy(tw)
    for name in zero:
        getattr(tw, name).data.zero_()
    return tw


def qkv_rows(shape):
    qd, kd = shape.nq * shape.hd, shape.nkv * shape.hd
    return slice(0, qd), slice(qd, qd + kd), slice(qd + kd, qd + 2 * kd)


def complex_pairs(v, hd):
    """Pairs (i, i + hd/2) of every head as complex numbers [..., heads, hd/2]."""
    v = np.asarray(v, np.float64).reshape(v.shape[:-1] + (-1, hd))
    return v[..., : hd // 2] + 1j * v[..., hd // 2:]


def freqs(hd, theta=10000.0):
    return theta ** (-2.0 * np.arange(hd // 2) / hd)


# ------------------------------------------------------------------ target
@pytest.mark.parametrize("dtype", [configs.F32, configs.BF16])
def test_target_without_attention_and_ffn_is_tied_head_on_embedding(dtype):
    shape = configs.TargetShape(**{**SHAPE.__dict__, "wdtype": dtype})
    tw = target(shape, wo=1, wdown=1)
    T = oracle.Target(tw)
    toks = np.array([3, 77, 400], np.int32)
    am, mg, hid, lg, res = oracle.forward_resid(T, oracle.Seq(T, 16), toks)
    E = f64(tw.embed.data[0].float())
    assert rel(res, E[toks]) < TOL
    n = rms(E[toks], f64(tw.g_final))
    assert rel(hid, n) < TOL
    assert rel(lg, n @ E.T) < TOL
    assert list(am) == list(np.argmax(np.float32(n @ E.T), axis=1))


def test_target_attention_with_zero_queries_is_causal_mean_of_values():
    """W_q = 0 and W_gate/up = 0: row r at position p adds W_o . mean_{p' <= p} v_{p'}
    per query head (KV head h // group), layer after layer; values pass
    through the fp32 cache."""
    tw = target(wgu=1)
    qs, ks, vs = qkv_rows(SHAPE)
    tw.wqkv.data[:, qs, :] = 0
    T = oracle.Target(tw)
    s = oracle.Seq(T, 32)
    toks = np.array([5, 9, 130, 9, 511, 0], np.int32)
    oracle.prefill(T, s, toks[:3])                 # positions 0..2 committed
    _, _, _, _, res = oracle.forward_resid(T, s, toks[3:])   # positions 3..5, not committed

    E = f64(tw.embed.data[0])
    x = E[toks].copy()
    grp, hd = SHAPE.nq // SHAPE.nkv, SHAPE.hd
    for l in range(SHAPE.L):
        xn = rms(x, f64(tw.g_attn[l]))
        v = np.float32(xn @ f64(tw.wqkv.data[l, vs]).T).astype(np.float64)   # [pos][nkv*hd]
        att = np.zeros((len(toks), SHAPE.nq * hd))
        for p in range(len(toks)):
            mean = v[: p + 1].mean(axis=0).reshape(SHAPE.nkv, hd)
            att[p] = np.concatenate([mean[h // grp] for h in range(SHAPE.nq)])
        x = x + att @ f64(tw.wo.data[l]).T
    assert rel(res, x[3:]) < 1e-7   # fp32 cache rounding of values is mirrored above


def test_target_ffn_through_odd_part_of_gelu():
    """One layer, W_o = 0: x(W_g) - x(-W_g) = W_down((W_g xn) * (W_u xn)),
    xn = RMSNorm(E[tok]) with the FFN gain."""
    shape = configs.TargetShape(**{**SHAPE.__dict__, "L": 1})
    tw = target(shape, wo=1)
    tw.g_attn.mul_(-3.0)                           # the FFN must not read this gain
    toks = np.array([17, 250], np.int32)
    outs = []
    for sign in (1.0, -1.0):
        t2 = copy.deepcopy(tw)
        t2.wgu.data[0, : shape.ff] *= sign
        T = oracle.Target(t2)
        outs.append(oracle.forward_resid(T, oracle.Seq(T, 8), toks)[4])
    E = f64(tw.embed.data[0])
    xn = rms(E[toks], f64(tw.g_ffn[0]))
    Wg, Wu = f64(tw.wgu.data[0, : shape.ff]), f64(tw.wgu.data[0, shape.ff:])
    want = ((xn @ Wg.T) * (xn @ Wu.T)) @ f64(tw.wdown.data[0]).T
    assert rel(outs[0] - outs[1], want) < 1e-9


def test_target_rope_positions_in_attention_complex_form():
    """One layer, no FFN: rows at positions 3 and 4 attend keys 0..3 and 0..4;
    scores from the complex form of RoPE, softmax, mean of fp32 values."""
    shape = configs.TargetShape(**{**SHAPE.__dict__, "L": 1, "wstd": 0.2})
    tw = target(shape, wgu=1)
    T = oracle.Target(tw)
    s = oracle.Seq(T, 16)
    toks = np.array([11, 300, 42, 7, 99], np.int32)
    oracle.prefill(T, s, toks[:3])
    _, _, _, _, res = oracle.forward_resid(T, s, toks[3:])

    hd, grp = shape.hd, shape.nq // shape.nkv
    qs, ks, vs = qkv_rows(shape)
    E = f64(tw.embed.data[0])
    xn = rms(E[toks], f64(tw.g_attn[0]))
    W = f64(tw.wqkv.data[0])
    zq = complex_pairs(xn @ W[qs].T, hd)            # [pos][nq][hd/2], before rotation
    zk = complex_pairs(xn @ W[ks].T, hd)            # [pos][nkv][hd/2]
    v = np.float32(xn @ W[vs].T).astype(np.float64).reshape(len(toks), shape.nkv, hd)
    w = freqs(hd)
    want = []
    for p in (3, 4):
        att = []
        for h in range(shape.nq):
            sc = np.array([np.real(np.sum(zq[p, h] * np.conj(zk[j, h // grp]) * np.exp(1j * (p - j) * w)))
                           for j in range(p + 1)]) / np.sqrt(hd)
            pr = np.exp(sc - sc.max())
            pr /= pr.sum()
            att.append(pr @ v[: p + 1, h // grp])
        want.append(E[toks[p]] + np.concatenate(att) @ f64(tw.wo.data[0]).T)
    # keys pass through the fp32 cache after rotation: agreement to fp32 level
    assert rel(res, np.array(want)) < 1e-6


# ------------------------------------------------------------------ drafter
def _drafter_setup(**zero):
    tw = synth.make_target(SHAPE)
    T = oracle.Target(tw)
    s = oracle.Seq(T, 64)
    oracle.prefill(T, s, synth.make_tokens(20, SHAPE.V).numpy())
    # garbage past the committed length: a drafter reading beyond len sees it
    s.kv[:, :, :, s.len:, :] = 1e3 * np.random.default_rng(5).standard_normal(
        s.kv[:, :, :, s.len:, :].shape).astype(np.float32)
    dw = copy.deepcopy(synth.make_drafter(DSHAPE))
    for name in zero:
        getattr(dw, name).data.zero_()
    return tw, T, s, dw


def _u0(tw, dw, h_prev, tok):
    E = f64(tw.embed.data[0])
    cat = np.concatenate([rms(h_prev, f64(dw.g_in_h)), rms(E[tok], f64(dw.g_in_e))])
    return f64(dw.w_in.data[0]) @ cat


def test_drafter_without_attention_and_ffn_is_in_out_projection_recurrence():
    """W_o' = W_down' = 0: u = W_in [N(h_{j-1}); N(E[tok_{j-1}])], h_j = W_out u,
    the head reads N_out(u); h_0 is the target's hidden, tok_0 the pending token,
    and each later step starts from the previous step's h_j and draft."""
    tw, T, s, dw = _drafter_setup(wo=1, wdown=1)
    D = oracle.Drafter(dw)
    k = 3
    d, mg, ub, hn = oracle.draft_states(T, D, s, k)
    h, tok = s.hid.copy(), s.pending
    for j in range(k):
        u = _u0(tw, dw, h, tok)
        assert rel(ub[j], rms(u, f64(dw.g_out))) < TOL
        h = f64(dw.w_out.data[0]) @ u
        assert rel(hn[j], h) < TOL
        tok = int(d[j])


def test_drafter_cross_attention_reads_exactly_committed_positions():
    """W_q' = 0, no FFN: each layer adds W_o' . (mean of the target's last-layer
    values over positions [0, len)) per query head; nothing past len counts."""
    tw, T, s, dw = _drafter_setup(wq=1, wgu=1)
    D = oracle.Drafter(dw)
    k = 2
    d, mg, ub, hn = oracle.draft_states(T, D, s, k)
    grp, hd = DSHAPE.nq // DSHAPE.nkv, DSHAPE.hd
    V = s.kv[SHAPE.L - 1, 1, :, : s.len, :].astype(np.float64)      # [nkv][len][hd]
    att = np.concatenate([V[h // grp].mean(axis=0) for h in range(DSHAPE.nq)])
    h, tok = s.hid.copy(), s.pending
    for j in range(k):
        u = _u0(tw, dw, h, tok)
        for l in range(DSHAPE.L):
            u = u + f64(dw.wo.data[l]) @ att
        h = f64(dw.w_out.data[0]) @ u
        assert rel(hn[j], h) < TOL
        assert rel(ub[j], rms(u, f64(dw.g_out))) < TOL
        tok = int(d[j])


def test_drafter_query_position_complex_form():
    """One drafter layer, no FFN: step j's query is rotated to position
    len + j - 1 and scored against the cached (already rotated) keys."""
    tw, T, s, dw = _drafter_setup(wgu=1)
    dw.wq.data.mul_(8.0)                              # sharper attention: positions matter
    dsh = configs.DrafterShape(**{**DSHAPE.__dict__, "L": 1})
    dw.shape = dsh
    for name in ("wq", "wo", "wgu", "wdown"):
        wt = getattr(dw, name)
        wt.data, wt.L = wt.data[:1].contiguous(), 1
    dw.g_attn, dw.g_ffn = dw.g_attn[:1].contiguous(), dw.g_ffn[:1].contiguous()
    D = oracle.Drafter(dw)
    k = 2
    d, mg, ub, hn = oracle.draft_states(T, D, s, k)
    hd, grp = DSHAPE.hd, DSHAPE.nq // DSHAPE.nkv
    Kc = s.kv[SHAPE.L - 1, 0, :, : s.len, :].astype(np.float64)     # rotated keys [nkv][len][hd]
    Vc = s.kv[SHAPE.L - 1, 1, :, : s.len, :].astype(np.float64)
    zk = complex_pairs(Kc, hd)[:, :, 0, :]                          # [nkv][len][hd/2]
    w = freqs(hd)
    h, tok = s.hid.copy(), s.pending
    for j in range(1, k + 1):
        u = _u0(tw, dw, h, tok)
        q = f64(dw.wq.data[0]) @ rms(u, f64(dw.g_attn[0]))
        zq = complex_pairs(q, hd)                                   # [nq][hd/2]
        pos = s.len + j - 1
        att = []
        for hh in range(DSHAPE.nq):
            rot = zq[hh] * np.exp(1j * pos * w)
            sc = np.real(np.conj(zk[hh // grp]) @ rot) / np.sqrt(hd)
            pr = np.exp(sc - sc.max())
            pr /= pr.sum()
            att.append(pr @ Vc[hh // grp])
        u = u + f64(dw.wo.data[0]) @ np.concatenate(att)
        h = f64(dw.w_out.data[0]) @ u
        assert rel(hn[j - 1], h) < 1e-9
        tok = int(d[j - 1])


def test_drafter_ffn_through_odd_part_of_gelu():
    """One step, W_o' = 0: h(W_g') - h(-W_g') = W_out . sum_l W_down'_l((W_g' un)
    * (W_u' un)) with one layer, un = N(u) under the FFN gain; the attention
    gain has no effect."""
    tw, T, s, dw = _drafter_setup(wo=1)
    dsh = configs.DrafterShape(**{**DSHAPE.__dict__, "L": 1})
    dw.shape = dsh
    for name in ("wq", "wo", "wgu", "wdown"):
        wt = getattr(dw, name)
        wt.data, wt.L = wt.data[:1].contiguous(), 1
    dw.g_attn, dw.g_ffn = dw.g_attn[:1].contiguous() * -2.0, dw.g_ffn[:1].contiguous()
    hs = []
    for sign in (1.0, -1.0):
        d2 = copy.deepcopy(dw)
        d2.wgu.data[0, : dsh.ff] *= sign
        hs.append(oracle.draft_states(T, oracle.Drafter(d2), s, 1)[3][0])
    u = _u0(tw, dw, s.hid.copy(), s.pending)
    un = rms(u, f64(dw.g_ffn[0]))
    Wg, Wu = f64(dw.wgu.data[0, : dsh.ff]), f64(dw.wgu.data[0, dsh.ff:])
    want = f64(dw.w_out.data[0]) @ (f64(dw.wdown.data[0]) @ ((Wg @ un) * (Wu @ un)))
    assert rel(hs[0] - hs[1], want) < 1e-9
