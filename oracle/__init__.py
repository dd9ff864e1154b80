"""ctypes wrapper of the CPU oracle (liboracle.so built from oracle.c).

TEST INFRASTRUCTURE: only tests/, the smoke check and the benchmark's
CPU-baseline leg import this package. It takes host copies of the seeded
inputs (speculative_decoding_spec_gb300.synth) and never calls the CUDA
library.
"""
import ctypes as C
import os

import numpy as np
import torch

from . import build as _build

_DT = {"f32": 0, "bf16": 1, "q4_0": 2}
_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        d, i, p = C.c_double, C.c_int, C.c_void_p
        _lib.or_bf16_to_double.restype = d
        _lib.or_bf16_to_double.argtypes = [C.c_uint16]
        _lib.or_f16_to_double.restype = d
        _lib.or_f16_to_double.argtypes = [C.c_uint16]
        _lib.or_round_kv.restype = C.c_float
        _lib.or_round_kv.argtypes = [d, i]
        _lib.or_dequant_row.argtypes = [C.POINTER(OrW), i, C.c_int64, p]
        _lib.or_linear.argtypes = [C.POINTER(OrW), i, i, p, i, p]
        _lib.or_rmsnorm.argtypes = [p, i, p, d, p]
        _lib.or_rope.argtypes = [p, i, C.c_int64, d]
        _lib.or_gelu.restype = d
        _lib.or_gelu.argtypes = [d]
        _lib.or_attend.argtypes = [p, p, p, i, i, p]
        _lib.or_argmax_f32.restype = i
        _lib.or_argmax_f32.argtypes = [p, i, p]
        _lib.or_forward.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), p, i, p, p, p, p]
        _lib.or_forward_resid.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), p, i, p, p, p, p, p]
        _lib.or_draft_states.argtypes = [C.POINTER(OrModel), C.POINTER(OrDrafter), C.POINTER(OrSeq),
                                         i, p, p, p, p]
        _lib.or_prefill.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), p, i, p]
        _lib.or_accept.restype = i
        _lib.or_accept.argtypes = [i, p, p]
        _lib.or_verify.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), i, p, p, p, p]
        _lib.or_rank_f32.restype = i
        _lib.or_rank_f32.argtypes = [p, i, i]
        _lib.or_verify_topm.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), i, p, i, p, p, p, p]
        _lib.or_verify_tree.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), i, p, p, p, p, p]
        _lib.or_topk_f32.argtypes = [p, i, i, p, p]
        _lib.or_greedy.argtypes = [C.POINTER(OrModel), C.POINTER(OrSeq), i, p, p]
        _lib.or_draft.argtypes = [C.POINTER(OrModel), C.POINTER(OrDrafter), C.POINTER(OrSeq), i,
                                  p, p]
        _lib.or_draft_head.restype = i
        _lib.or_draft_head.argtypes = [C.POINTER(OrDrafter), p, p]
    return _lib


class OrW(C.Structure):
    _fields_ = [("dtype", C.c_int), ("data", C.c_void_p), ("scales", C.c_void_p)]


class OrModel(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("L", "d", "nq", "nkv", "hd", "ff", "V", "kv_dtype")] + [
        ("eps", C.c_double), ("theta", C.c_double), ("embed", OrW), ("wqkv", OrW), ("wo", OrW),
        ("wgu", OrW), ("wdown", OrW), ("g_attn", C.c_void_p), ("g_ffn", C.c_void_p),
        ("g_final", C.c_void_p), ("n_experts", C.c_int), ("top_k", C.c_int), ("ff_e", C.c_int),
        ("router", OrW), ("wgu_e", OrW), ("wdown_e", OrW)]


class OrDrafter(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("L", "h", "bh", "ff", "nq", "hd", "nkv", "clustered",
                                       "n_centroids", "top_c", "cluster_size", "V")] + [
        ("w_in", OrW), ("g_in_h", C.c_void_p), ("g_in_e", C.c_void_p), ("wq", OrW), ("wo", OrW),
        ("wgu", OrW), ("wdown", OrW), ("g_attn", C.c_void_p), ("g_ffn", C.c_void_p),
        ("g_out", C.c_void_p), ("w_out", OrW), ("vocab", OrW), ("centroids", OrW),
        ("perm", C.c_void_p)]


class OrSeq(C.Structure):
    _fields_ = [("kv", C.c_void_p), ("cap", C.c_int), ("len", C.c_int), ("pending", C.c_int),
                ("hid", C.c_void_p)]


def _np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        t = t.view(torch.int16)
        return t.numpy().view(np.uint16)
    if t.dtype == torch.float16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class _Keep:
    """Holds host arrays alive while the C structs point at them."""

    def __init__(self):
        self.arrays = []

    def arr(self, t):
        a = t if isinstance(t, np.ndarray) else _np(t)
        a = np.ascontiguousarray(a)
        self.arrays.append(a)
        return a

    def w(self, wt) -> OrW:
        data = self.arr(wt.data)
        sc = self.arr(wt.scales) if wt.scales is not None else None
        return OrW(_DT[wt.dtype], _ptr(data), _ptr(sc) if sc is not None else None)


class Target:
    """Host copy of a synthetic target model (synth.TargetWeights)."""

    def __init__(self, tw):
        s = tw.shape
        self.shape = s
        self.keep = _Keep()
        k = self.keep
        self.m = OrModel(L=s.L, d=s.d, nq=s.nq, nkv=s.nkv, hd=s.hd, ff=s.ff, V=s.V,
                         kv_dtype=_DT[s.kvdtype], eps=s.eps, theta=s.theta,
                         embed=k.w(tw.embed), wqkv=k.w(tw.wqkv), wo=k.w(tw.wo), wgu=k.w(tw.wgu),
                         wdown=k.w(tw.wdown), g_attn=_ptr(k.arr(tw.g_attn)),
                         g_ffn=_ptr(k.arr(tw.g_ffn)), g_final=_ptr(k.arr(tw.g_final)))
        if getattr(s, "n_experts", 0):
            self.m.n_experts, self.m.top_k, self.m.ff_e = s.n_experts, s.top_k, s.ff_e
            self.m.router, self.m.wgu_e, self.m.wdown_e = k.w(tw.router), k.w(tw.wgu_e), k.w(tw.wdown_e)


class Drafter:
    """Host copy of synthetic drafter weights (synth.DrafterWeights)."""

    def __init__(self, dw):
        s = dw.shape
        self.shape = s
        self.keep = _Keep()
        k = self.keep
        self.m = OrDrafter(L=s.L, h=s.h, bh=s.bh, ff=s.ff, nq=s.nq, hd=s.hd, nkv=s.nkv,
                           clustered=int(s.clustered), n_centroids=s.n_centroids, top_c=s.top_c,
                           cluster_size=s.cluster_size, V=s.V, w_in=k.w(dw.w_in),
                           g_in_h=_ptr(k.arr(dw.g_in_h)), g_in_e=_ptr(k.arr(dw.g_in_e)),
                           wq=k.w(dw.wq), wo=k.w(dw.wo), wgu=k.w(dw.wgu), wdown=k.w(dw.wdown),
                           g_attn=_ptr(k.arr(dw.g_attn)), g_ffn=_ptr(k.arr(dw.g_ffn)),
                           g_out=_ptr(k.arr(dw.g_out)), w_out=k.w(dw.w_out),
                           vocab=k.w(dw.vocab),
                           centroids=k.w(dw.centroids) if dw.centroids is not None else OrW(),
                           perm=_ptr(k.arr(dw.perm)) if dw.perm is not None else None)


class Seq:
    """One sequence: its cache (float [L][2][nkv][cap][hd]) and decode state."""

    def __init__(self, target: Target, cap: int):
        s = target.shape
        self.target = target
        self.kv = np.zeros((s.L, 2, s.nkv, cap, s.hd), dtype=np.float32)
        self.hid = np.zeros((s.d,), dtype=np.float64)
        self.c = OrSeq(kv=_ptr(self.kv), cap=cap, len=0, pending=0, hid=_ptr(self.hid))

    @property
    def len(self):
        return self.c.len

    @property
    def pending(self):
        return self.c.pending

    def load_prefilled(self, contig: torch.Tensor) -> None:
        """Adopt cache contents [L][2][nkv][n][hd] for positions [0, n)."""
        n = contig.shape[3]
        self.kv[:, :, :, :n, :] = contig.float().cpu().numpy()
        self.c.len = n

    def set_state(self, length: int, pending: int) -> None:
        self.c.len = length
        self.c.pending = pending

    def clone(self) -> "Seq":
        o = Seq.__new__(Seq)
        o.target = self.target
        o.kv = self.kv.copy()
        o.hid = self.hid.copy()
        o.c = OrSeq(kv=_ptr(o.kv), cap=self.c.cap, len=self.c.len, pending=self.c.pending,
                    hid=_ptr(o.hid))
        return o


def _i32(x):
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def forward(t: Target, s: Seq, tokens, want_logits=False):
    """Forward R rows at positions len..len+R-1 (len not advanced).
    Returns (argmax[R], margin[R], hidden[R][d], logits[R][V] or None)."""
    tok = _i32(tokens)
    R = tok.shape[0]
    am = np.zeros(R, np.int32)
    mg = np.zeros(R, np.float64)
    hid = np.zeros((R, t.shape.d), np.float64)
    lg = np.zeros((R, t.shape.V), np.float64) if want_logits else None
    rc = lib().or_forward(C.byref(t.m), C.byref(s.c), _ptr(tok), R,
                          _ptr(lg) if lg is not None else None, _ptr(am), _ptr(mg), _ptr(hid))
    assert rc == 0, "or_forward failed (capacity?)"
    return am, mg, hid, lg


def forward_resid(t: Target, s: Seq, tokens):
    """forward() plus the residual stream after the last layer (before the
    final RMSNorm). Returns (argmax, margin, hidden, logits, resid[R][d])."""
    tok = _i32(tokens)
    R = tok.shape[0]
    am = np.zeros(R, np.int32)
    mg = np.zeros(R, np.float64)
    hid = np.zeros((R, t.shape.d), np.float64)
    lg = np.zeros((R, t.shape.V), np.float64)
    res = np.zeros((R, t.shape.d), np.float64)
    rc = lib().or_forward_resid(C.byref(t.m), C.byref(s.c), _ptr(tok), R, _ptr(lg), _ptr(am),
                                _ptr(mg), _ptr(hid), _ptr(res))
    assert rc == 0, "or_forward_resid failed (capacity?)"
    return am, mg, hid, lg, res


def prefill(t: Target, s: Seq, tokens) -> float:
    tok = _i32(tokens)
    mg = C.c_double()
    rc = lib().or_prefill(C.byref(t.m), C.byref(s.c), _ptr(tok), tok.shape[0], C.addressof(mg))
    assert rc == 0
    return mg.value


def verify(t: Target, s: Seq, drafts):
    """One greedy verify step. Returns (emitted tokens, margins[k+1])."""
    d = _i32(drafts)
    k = d.shape[0]
    out = np.zeros(k + 1, np.int32)
    ne = np.zeros(1, np.int32)
    mg = np.zeros(k + 1, np.float64)
    rc = lib().or_verify(C.byref(t.m), C.byref(s.c), k, _ptr(d) if k else None, _ptr(out),
                         _ptr(ne), _ptr(mg))
    assert rc == 0
    return out[: ne[0]].copy(), mg


def verify_topm(t: Target, s: Seq, drafts, top_m: int):
    """Lenient verify step. Returns (emitted tokens, margins[k+1], decision[k])."""
    d = _i32(drafts)
    k = d.shape[0]
    out = np.zeros(k + 1, np.int32)
    ne = np.zeros(1, np.int32)
    mg = np.zeros(k + 1, np.float64)
    dec = np.zeros(max(k, 1), np.float64)
    rc = lib().or_verify_topm(C.byref(t.m), C.byref(s.c), k, _ptr(d) if k else None, top_m, _ptr(out),
                              _ptr(ne), _ptr(mg), _ptr(dec))
    assert rc == 0
    return out[: ne[0]].copy(), mg, dec[:k]


def verify_tree(t: Target, s: Seq, tokens, parents):
    """Tree verify step. Returns (emitted tokens, margins[n+1]: per node, root first)."""
    tk, pa = _i32(tokens), _i32(parents)
    n = tk.shape[0]
    out = np.zeros(n + 1, np.int32)
    ne = np.zeros(1, np.int32)
    mg = np.zeros(n + 1, np.float64)
    rc = lib().or_verify_tree(C.byref(t.m), C.byref(s.c), n, _ptr(tk), _ptr(pa), _ptr(out), _ptr(ne), _ptr(mg))
    assert rc == 0, "or_verify_tree failed (bad parents or capacity)"
    return out[: ne[0]].copy(), mg


def topk_f32(scores, k: int):
    sc = np.ascontiguousarray(np.asarray(scores, np.float64))
    idx = np.zeros(k, np.int32)
    gap = C.c_double()
    lib().or_topk_f32(_ptr(sc), sc.shape[0], k, _ptr(idx), C.addressof(gap))
    return idx, gap.value


def rank_f32(logits, tok: int) -> int:
    lg = np.ascontiguousarray(np.asarray(logits, np.float64))
    return lib().or_rank_f32(_ptr(lg), lg.shape[0], tok)


def greedy(t: Target, s: Seq, n: int):
    out = np.zeros(n, np.int32)
    mg = np.zeros(n, np.float64)
    rc = lib().or_greedy(C.byref(t.m), C.byref(s.c), n, _ptr(out), _ptr(mg))
    assert rc == 0
    return out, mg


def accept(drafts, t) -> int:
    d, tt = _i32(drafts), _i32(t)
    return lib().or_accept(d.shape[0], _ptr(d) if d.shape[0] else None, _ptr(tt))


def draft(t: Target, dr: Drafter, s: Seq, k: int):
    out = np.zeros(k, np.int32)
    mg = np.zeros(k, np.float64)
    rc = lib().or_draft(C.byref(t.m), C.byref(dr.m), C.byref(s.c), k, _ptr(out), _ptr(mg))
    assert rc == 0
    return out, mg


def draft_states(t: Target, dr: Drafter, s: Seq, k: int):
    """draft() plus per-step states: (drafts, margins, u_bar[k][h], h_next[k][bh])."""
    out = np.zeros(k, np.int32)
    mg = np.zeros(k, np.float64)
    ub = np.zeros((k, dr.shape.h), np.float64)
    hn = np.zeros((k, dr.shape.bh), np.float64)
    rc = lib().or_draft_states(C.byref(t.m), C.byref(dr.m), C.byref(s.c), k, _ptr(out), _ptr(mg),
                               _ptr(ub), _ptr(hn))
    assert rc == 0
    return out, mg, ub, hn


def draft_head(dr: Drafter, u_bar) -> tuple:
    u = np.ascontiguousarray(np.asarray(u_bar, np.float64))
    mg = C.c_double()
    tok = lib().or_draft_head(C.byref(dr.m), _ptr(u), C.addressof(mg))
    return tok, mg.value


# ---- single operations, for the pins ----
def rmsnorm(x, g, eps):
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    g = np.ascontiguousarray(np.asarray(g, np.float32))
    out = np.zeros_like(x)
    lib().or_rmsnorm(_ptr(x), x.shape[0], _ptr(g), eps, _ptr(out))
    return out


def rope(v, pos, theta=10000.0):
    v = np.array(v, np.float64)
    lib().or_rope(_ptr(v), v.shape[0], pos, theta)
    return v


def gelu(x: float) -> float:
    return lib().or_gelu(x)


def attend(q, K, V):
    q = np.ascontiguousarray(np.asarray(q, np.float64))
    K = np.ascontiguousarray(np.asarray(K, np.float32))
    V = np.ascontiguousarray(np.asarray(V, np.float32))
    o = np.zeros(q.shape[0], np.float64)
    lib().or_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], q.shape[0], _ptr(o))
    return o


def linear(wt, x, layer=0):
    """y = x . W^T for layer `layer` of a WTensor stack, x [M][K] float64."""
    keep = _Keep()
    w = keep.w(wt)
    # offset to the layer by building a one-layer view
    if layer:
        sub = type(wt)(wt.dtype, 1, wt.N, wt.K, wt.data[layer:layer + 1],
                       wt.scales[layer:layer + 1] if wt.scales is not None else None)
        w = keep.w(sub)
    x = np.ascontiguousarray(np.asarray(x, np.float64))
    M = x.shape[0]
    y = np.zeros((M, wt.N), np.float64)
    lib().or_linear(C.byref(w), wt.N, wt.K, _ptr(x), M, _ptr(y))
    return y


def dequant_row(wt, n: int, layer: int = 0):
    keep = _Keep()
    sub = type(wt)(wt.dtype, 1, wt.N, wt.K, wt.data[layer:layer + 1],
                   wt.scales[layer:layer + 1] if wt.scales is not None else None)
    w = keep.w(sub)
    out = np.zeros(wt.K, np.float64)
    lib().or_dequant_row(C.byref(w), wt.K, n, _ptr(out))
    return out


def round_kv(x: float, dtype: str) -> float:
    return lib().or_round_kv(x, _DT[dtype])


def argmax_f32(logits):
    lg = np.ascontiguousarray(np.asarray(logits, np.float64))
    mg = C.c_double()
    return lib().or_argmax_f32(_ptr(lg), lg.shape[0], C.addressof(mg)), mg.value
