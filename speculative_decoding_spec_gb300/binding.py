"""ctypes binding of libspec_gb300.so (include/spec.h), same names as the C ABI.

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels. PyTorch provides device memory and streams. If the library has
not been built, every entry point raises instead of falling back to anything.
"""
import ctypes as C
import math
import os
from typing import Optional

import torch

from . import synth
from .configs import BF16, F32, PAGE, Q4_0

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libspec_gb300.so")

SPEC_OK, SPEC_EINVAL, SPEC_ECAPACITY, SPEC_ESTATE, SPEC_ECUDA, SPEC_ETIMEOUT, SPEC_EUNSUPPORTED = range(7)
DTYPES = {F32: 0, BF16: 1, Q4_0: 2}

EXPORTS = ["spec_workspace_bytes", "spec_init", "spec_prefill", "spec_draft", "spec_verify", "spec_step",
           "spec_decode", "spec_inject_drafts", "spec_stats", "spec_sync", "spec_set_graphs",
           "spec_kernel_launches", "spec_status_str", "spec_destroy", "spec_linear",
           "spec_linear_workspace_bytes", "spec_linear_noalloc", "spec_set_option",
           "spec_attention_workspace_bytes", "spec_attention", "spec_verify_topm", "spec_verify_tree"]
SPEC_OPT_GRAPHS, SPEC_OPT_PREFETCH, SPEC_OPT_TEST_ATTN_WAIT = 1, 4, 8
SPEC_OPT_WIDE_TRACE = 7
SPEC_LINEAR_NOALLOC_MAX_ROWS = 523776


class spec_matrix(C.Structure):
    _fields_ = [("dtype", C.c_int32), ("data", C.c_void_p), ("scales", C.c_void_p)]


class spec_model_desc(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layers", "d_model", "n_q_heads", "n_kv_heads", "head_dim",
                                          "d_ff", "vocab", "w_dtype", "kv_dtype")] + [
        ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("n_experts", C.c_int32), ("top_k", C.c_int32),
        ("d_ff_expert", C.c_int32)]


class spec_weights(C.Structure):
    _fields_ = [("embed", spec_matrix), ("wqkv", spec_matrix), ("wo", spec_matrix), ("wgu", spec_matrix),
                ("wdown", spec_matrix), ("g_attn", C.c_void_p), ("g_ffn", C.c_void_p),
                ("g_final", C.c_void_p), ("router", spec_matrix), ("wgu_e", spec_matrix),
                ("wdown_e", spec_matrix)]


class spec_drafter_desc(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_layers", "hidden", "d_ff", "n_q_heads", "clustered",
                                          "n_centroids", "top_c", "w_dtype")]


class spec_drafter_weights(C.Structure):
    _fields_ = [("w_in", spec_matrix), ("g_in_h", C.c_void_p), ("g_in_e", C.c_void_p),
                ("wq", spec_matrix), ("wo", spec_matrix), ("wgu", spec_matrix), ("wdown", spec_matrix),
                ("g_attn", C.c_void_p), ("g_ffn", C.c_void_p), ("g_out", C.c_void_p),
                ("w_out", spec_matrix), ("vocab", spec_matrix), ("centroids", spec_matrix),
                ("perm", C.c_void_p)]


class spec_kv_desc(C.Structure):
    _fields_ = [("pool", C.c_void_p), ("n_pages", C.c_int32), ("page_size", C.c_int32),
                ("block_table", C.c_void_p), ("max_pages_per_seq", C.c_int32), ("n_slots", C.c_int32)]


class spec_state(C.Structure):
    _fields_ = [("seq_len", C.c_void_p), ("pending", C.c_void_p), ("hid", C.c_void_p),
                ("stats", C.c_void_p)]


class spec_stats_t(C.Structure):
    _fields_ = [("passes", C.c_int64), ("drafted", C.c_int64), ("accepted", C.c_int64),
                ("emitted", C.c_int64), ("tokens_per_pass", C.c_double)]


_lib = None


def lib():
    """Load the CUDA library; raises if it has not been built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libspec_gb300.so is not built; run `python -c \"import __graft_entry__ as g; "
                           "g.build()\"` first")
    L = C.CDLL(LIB_PATH)
    p, i32, st = C.c_void_p, C.c_int32, C.c_int
    L.spec_workspace_bytes.restype = C.c_size_t
    L.spec_workspace_bytes.argtypes = [p, p, i32, i32, i32]
    L.spec_init.restype = st
    L.spec_init.argtypes = [p, p, p, p, p, p, i32, i32, p, C.c_size_t, p, C.POINTER(p)]
    L.spec_prefill.restype = st
    L.spec_prefill.argtypes = [p, i32, p, i32, p, p]
    L.spec_draft.restype = st
    L.spec_draft.argtypes = [p, i32, p, i32, p, p]
    L.spec_verify.restype = st
    L.spec_verify.argtypes = [p, i32, p, i32, p, p, p, p, p]
    L.spec_step.restype = st
    L.spec_step.argtypes = [p, i32, p, i32, p, p, p]
    L.spec_decode.restype = st
    L.spec_decode.argtypes = [p, i32, p, p, p]
    L.spec_inject_drafts.restype = st
    L.spec_inject_drafts.argtypes = [p, i32, p, i32, p, p, i32, C.c_float, p, p, p]
    L.spec_stats.restype = st
    L.spec_stats.argtypes = [p, i32, C.POINTER(spec_stats_t), p]
    L.spec_sync.restype = st
    L.spec_sync.argtypes = [p, p]
    L.spec_set_graphs.restype = st
    L.spec_set_graphs.argtypes = [p, i32]
    L.spec_kernel_launches.restype = C.c_int64
    L.spec_kernel_launches.argtypes = [p]
    L.spec_status_str.restype = C.c_char_p
    L.spec_status_str.argtypes = [st]
    L.spec_linear_workspace_bytes.restype = C.c_size_t
    L.spec_linear_workspace_bytes.argtypes = [i32, i32, i32]
    L.spec_linear.restype = st
    L.spec_linear.argtypes = [C.POINTER(spec_matrix), i32, i32, p, i32, p, C.c_float, p, p, C.c_size_t, p]
    L.spec_set_option.restype = st
    L.spec_set_option.argtypes = [p, i32, C.c_int64]
    L.spec_linear_noalloc.restype = st
    L.spec_linear_noalloc.argtypes = [C.POINTER(spec_matrix), i32, i32, p, i32, p, C.c_float, p, p]
    L.spec_attention_workspace_bytes.restype = C.c_size_t
    L.spec_attention_workspace_bytes.argtypes = [p, i32, i32, i32, i32]
    L.spec_attention.restype = st
    L.spec_attention.argtypes = [p, p, i32, i32, p, p, i32, i32, i32, p, p, p, C.c_size_t, p]
    L.spec_verify_topm.restype = st
    L.spec_verify_topm.argtypes = [p, i32, p, i32, p, i32, p, p, p, p]
    L.spec_verify_tree.restype = st
    L.spec_verify_tree.argtypes = [p, i32, p, i32, p, p, p, p, p, p]
    L.spec_destroy.restype = None
    L.spec_destroy.argtypes = [p]
    _lib = L
    return L


class SpecError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__("%s failed: %s (%d)" % (fn, lib().spec_status_str(code).decode(), code))
        self.code = code


def check(fn, code):
    if code != SPEC_OK:
        raise SpecError(fn, code)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _mat(w) -> spec_matrix:
    return spec_matrix(DTYPES[w.dtype], _ptr(w.data), _ptr(w.scales))


def model_desc(t) -> spec_model_desc:
    return spec_model_desc(t.L, t.d, t.nq, t.nkv, t.hd, t.ff, t.V, DTYPES[t.wdtype], DTYPES[t.kvdtype],
                           t.eps, t.theta, getattr(t, "n_experts", 0), getattr(t, "top_k", 0),
                           getattr(t, "ff_e", 0))


def drafter_desc(d) -> spec_drafter_desc:
    return spec_drafter_desc(d.L, d.h, d.ff, d.nq, int(d.clustered), d.n_centroids, d.top_c,
                             DTYPES[d.wdtype])


def spec_linear(w, x: torch.Tensor, gain: Optional[torch.Tensor] = None, eps: float = 1e-6,
                layer: int = 0, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y = (RMSNorm(x) * gain if gain is given else x) . W[layer]^T on the
    library's weight-streaming kernel (x float32 [M][K] on the device)."""
    L = lib()
    sub = synth.WTensor(w.dtype, 1, w.N, w.K, w.data[layer], w.scales[layer] if w.scales is not None else None)
    m = _mat(sub)
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    ws = _linear_ws(x.device, L.spec_linear_workspace_bytes(w.N, w.K, M))
    check("spec_linear", L.spec_linear(C.byref(m), w.N, w.K, _ptr(x), M, _ptr(gain), eps, _ptr(y),
                                       _ptr(ws), ws.numel(), s.cuda_stream))
    return y


def spec_linear_noalloc(w, x: torch.Tensor, gain: Optional[torch.Tensor] = None, eps: float = 1e-6,
                        layer: int = 0, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """spec_linear through the entry point that allocates nothing (its scratch
    is a fixed array inside the library; see include/spec.h)."""
    L = lib()
    sub = synth.WTensor(w.dtype, 1, w.N, w.K, w.data[layer], w.scales[layer] if w.scales is not None else None)
    m = _mat(sub)
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, w.N), dtype=torch.float32, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    check("spec_linear_noalloc", L.spec_linear_noalloc(C.byref(m), w.N, w.K, _ptr(x), M, _ptr(gain), eps,
                                                       _ptr(y), s.cuda_stream))
    return y


def spec_attention(t, pool: torch.Tensor, block_table: torch.Tensor, layer: int, seq_ids: torch.Tensor,
                   seq_len: torch.Tensor, R: int, n_q_heads: int, key_extra: int, q: torch.Tensor,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One attention launch over a paged cache (include/spec.h spec_attention).
    pool [L][n_pages][2][nkv][64][hd] in the cache dtype of shape t,
    block_table int32 [n_slots][max_pages], q float32 [B*R][n_q_heads*hd]."""
    L = lib()
    md = model_desc(t)
    kv = spec_kv_desc(_ptr(pool), pool.shape[1], PAGE, _ptr(block_table), block_table.shape[1],
                      block_table.shape[0])
    B = seq_ids.shape[0]
    if out is None:
        out = torch.empty_like(q)
    nbytes = L.spec_attention_workspace_bytes(C.byref(md), B, R, n_q_heads, block_table.shape[1])
    if nbytes == 0:
        raise SpecError("spec_attention_workspace_bytes", SPEC_EINVAL)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    s = stream if stream is not None else torch.cuda.current_stream()
    check("spec_attention", L.spec_attention(C.byref(md), C.byref(kv), layer, B, _ptr(seq_ids), _ptr(seq_len),
                                             R, n_q_heads, key_extra, _ptr(q), _ptr(out), _ptr(ws), nbytes,
                                             s.cuda_stream))
    out.workspace = ws      # error word in its first int
    return out


_LINEAR_WS = {}


def _linear_ws(device, nbytes):
    """A zeroed workspace per device, grown on demand (the kernel leaves it zeroed)."""
    key = str(device)
    ws = _LINEAR_WS.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _LINEAR_WS[key] = ws
    return ws


class Engine:
    """Owns the torch allocations (KV pool, block table, slot state, workspace)
    around one spec_ctx and forwards calls to the C ABI on its own stream."""

    def __init__(self, tw, dw=None, n_slots=1, B_max=1, rows_max=4, max_ctx=256, shuffle_pages=False,
                 device="cuda", graphs=True):
        L = lib()
        t = tw.shape
        self.tw, self.dw, self.shape = tw, dw, t
        self.device = device
        self.pages_per_seq = int(math.ceil(max_ctx / PAGE))
        self.n_pages = n_slots * self.pages_per_seq
        kvdt = torch.float32 if t.kvdtype == F32 else torch.bfloat16
        self.pool = torch.zeros((t.L, self.n_pages, 2, t.nkv, PAGE, t.hd), dtype=kvdt, device=device)
        self.block_table = synth.make_page_table(n_slots, self.pages_per_seq, self.n_pages, shuffle_pages,
                                                 device=device)
        self.seq_len = torch.zeros(n_slots, dtype=torch.int32, device=device)
        self.pending = torch.zeros(n_slots, dtype=torch.int32, device=device)
        self.hid = torch.zeros((n_slots, t.d), dtype=torch.float32, device=device)
        self.stats = torch.zeros((n_slots, 4), dtype=torch.int64, device=device)
        self.n_slots, self.B_max, self.rows_max = n_slots, B_max, rows_max
        self.stream = torch.cuda.Stream(device=device)
        self._md = model_desc(t)
        moe = getattr(tw, "router", None) is not None
        self._w = spec_weights(_mat(tw.embed), _mat(tw.wqkv), _mat(tw.wo), _mat(tw.wgu), _mat(tw.wdown),
                               _ptr(tw.g_attn), _ptr(tw.g_ffn), _ptr(tw.g_final),
                               _mat(tw.router) if moe else spec_matrix(), _mat(tw.wgu_e) if moe else spec_matrix(),
                               _mat(tw.wdown_e) if moe else spec_matrix())
        self._dd = self._dw = None
        if dw is not None:
            self._dd = drafter_desc(dw.shape)
            self._dw = spec_drafter_weights(
                _mat(dw.w_in), _ptr(dw.g_in_h), _ptr(dw.g_in_e), _mat(dw.wq), _mat(dw.wo), _mat(dw.wgu),
                _mat(dw.wdown), _ptr(dw.g_attn), _ptr(dw.g_ffn), _ptr(dw.g_out), _mat(dw.w_out),
                _mat(dw.vocab), _mat(dw.centroids) if dw.centroids is not None else spec_matrix(),
                _ptr(dw.perm))
        self._kv = spec_kv_desc(_ptr(self.pool), self.n_pages, PAGE, _ptr(self.block_table),
                                self.pages_per_seq, n_slots)
        self._st = spec_state(_ptr(self.seq_len), _ptr(self.pending), _ptr(self.hid), _ptr(self.stats))
        dd = C.byref(self._dd) if self._dd is not None else None
        nbytes = L.spec_workspace_bytes(C.byref(self._md), dd, B_max, rows_max, self.pages_per_seq)
        if nbytes == 0:
            raise SpecError("spec_workspace_bytes", SPEC_EINVAL)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.stream.wait_stream(torch.cuda.current_stream())
        ctx = C.c_void_p()
        check("spec_init", L.spec_init(C.byref(self._md), C.byref(self._w), dd,
                                       C.byref(self._dw) if self._dw is not None else None,
                                       C.byref(self._kv), C.byref(self._st), B_max, rows_max,
                                       _ptr(self.workspace), nbytes, self.stream.cuda_stream,
                                       C.byref(ctx)))
        self.ctx = ctx
        if not graphs:
            check("spec_set_graphs", L.spec_set_graphs(ctx, 0))
        self._bufs = {}

    # -- helpers ------------------------------------------------------------
    def _buf(self, name, shape, dtype=torch.int32):
        key = (name, tuple(shape), dtype)
        b = self._bufs.get(key)
        if b is None:
            b = torch.empty(shape, dtype=dtype, device=self.device)
            self._bufs[key] = b
        return b

    def _in(self, name, t: torch.Tensor):
        """Copy an input into a persistent device buffer (stable pointers let
        the library replay its captured graphs)."""
        b = self._buf(name, t.shape, t.dtype)
        self.enter()
        with torch.cuda.stream(self.stream):
            b.copy_(t, non_blocking=True)
        return b

    def enter(self):
        self.stream.wait_stream(torch.cuda.current_stream())

    def leave(self):
        """Order later work on torch's current stream after the library's."""
        torch.cuda.current_stream().wait_stream(self.stream)

    def sync(self):
        check("spec_sync", lib().spec_sync(self.ctx, self.stream.cuda_stream))

    def seq_ids(self, ids):
        return self._in("seq_ids", torch.as_tensor(ids, dtype=torch.int32))

    # -- the C ABI --------------------------------------------------------------
    def spec_prefill(self, seq_ids: torch.Tensor, tokens: torch.Tensor):
        self.enter()
        B, R = tokens.shape
        check("spec_prefill", lib().spec_prefill(self.ctx, B, _ptr(seq_ids), R, _ptr(tokens),
                                                 self.stream.cuda_stream))
        self.leave()

    def spec_verify(self, seq_ids, drafts: torch.Tensor, logits: Optional[torch.Tensor] = None):
        self.enter()
        B, k = drafts.shape
        out = self._buf("out_tokens", (B, k + 1))
        ne = self._buf("n_emitted", (B,))
        check("spec_verify", lib().spec_verify(self.ctx, B, _ptr(seq_ids), k, _ptr(drafts) if k else None,
                                               _ptr(out), _ptr(ne), _ptr(logits), self.stream.cuda_stream))
        self.leave()
        return out, ne

    def spec_verify_topm(self, seq_ids, drafts: torch.Tensor, top_m: int, logits: Optional[torch.Tensor] = None):
        self.enter()
        B, k = drafts.shape
        out = self._buf("out_tokens", (B, k + 1))
        ne = self._buf("n_emitted", (B,))
        check("spec_verify_topm", lib().spec_verify_topm(self.ctx, B, _ptr(seq_ids), k, _ptr(drafts), int(top_m),
                                                         _ptr(out), _ptr(ne), _ptr(logits), self.stream.cuda_stream))
        self.leave()
        return out, ne

    def spec_verify_tree(self, seq_ids, tokens: torch.Tensor, parents: torch.Tensor,
                         logits: Optional[torch.Tensor] = None):
        self.enter()
        B, n = tokens.shape
        out = self._buf("out_tokens", (B, n + 1))
        ne = self._buf("n_emitted", (B,))
        check("spec_verify_tree", lib().spec_verify_tree(self.ctx, B, _ptr(seq_ids), n, _ptr(tokens), _ptr(parents),
                                                         _ptr(out), _ptr(ne), _ptr(logits), self.stream.cuda_stream))
        self.leave()
        return out, ne

    def spec_draft(self, seq_ids, B: int, k: int):
        self.enter()
        d = self._buf("drafts", (B, k))
        check("spec_draft", lib().spec_draft(self.ctx, B, _ptr(seq_ids), k, _ptr(d), self.stream.cuda_stream))
        self.leave()
        return d

    def spec_step(self, seq_ids, B: int, k: int):
        self.enter()
        out = self._buf("out_tokens", (B, k + 1))
        ne = self._buf("n_emitted", (B,))
        check("spec_step", lib().spec_step(self.ctx, B, _ptr(seq_ids), k, _ptr(out), _ptr(ne),
                                           self.stream.cuda_stream))
        self.leave()
        return out, ne

    def spec_decode(self, seq_ids, B: int):
        self.enter()
        out = self._buf("decode_out", (B,))
        check("spec_decode", lib().spec_decode(self.ctx, B, _ptr(seq_ids), _ptr(out), self.stream.cuda_stream))
        self.leave()
        return out

    def spec_inject_drafts(self, seq_ids, drafts, ref, alpha, draws, offsets):
        B, k = drafts.shape
        check("spec_inject_drafts", lib().spec_inject_drafts(
            self.ctx, B, _ptr(seq_ids), k, _ptr(drafts), _ptr(ref), ref.shape[1], float(alpha), _ptr(draws),
            _ptr(offsets), self.stream.cuda_stream))
        self.leave()

    def spec_stats(self, slot: int) -> spec_stats_t:
        s = spec_stats_t()
        check("spec_stats", lib().spec_stats(self.ctx, slot, C.byref(s), self.stream.cuda_stream))
        return s

    def set_option(self, option: int, value: int):
        check("spec_set_option", lib().spec_set_option(self.ctx, option, int(value)))

    def kernel_launches(self) -> int:
        return lib().spec_kernel_launches(self.ctx)

    def load_prefilled(self, slot: int, contig: torch.Tensor):
        """Adopt cache contents [L][2][nkv][n][hd] for positions [0, n) of a slot
        (synthetic long contexts) and set its committed length to n."""
        synth.scatter_to_pages(self.pool, contig, self.block_table[slot])
        self.seq_len[slot] = contig.shape[3]

    def close(self):
        if getattr(self, "ctx", None):
            self.stream.synchronize()
            lib().spec_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
