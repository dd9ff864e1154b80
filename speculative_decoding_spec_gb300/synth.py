"""Seeded synthetic inputs: weights, prompts, KV contents, page tables, draws.

This module serves both the CUDA path and the CPU oracle, so it holds none of
the method's arithmetic: it only draws random numbers, casts them to the
storage dtype and lays them out. Recipe (no dataset or trained checkpoint is
available, so these stand in for the pages' coding / summarisation prompts):

* linear weights, embedding (tied LM head) and drafter tables: N(0, wstd),
  wstd = 0.02 (0.01 for the ~30B model), stored in the model's weight dtype;
  Q4_0 weights: codes uniform on 0..15, fp16 scales |N(0, 0.004)|;
* mixture-of-experts targets: router and expert matrices N(0, wstd) like the
  rest (the dense FFN matrices are then small placeholders, unused);
* norm gains: 1 + N(0, 0.1) per element, from their own seeded stream (so that
  a gain read from the wrong layer or the wrong norm changes the result);
* the drafter's clustered vocabulary: a random permutation of the token ids
  sorted into 2048 balanced clusters; for float tables each member row is its
  centroid row plus N(0, wstd/2) noise, so the top clusters hold the best rows;
* prompts / first tokens: uniform over the vocabulary;
* pre-filled KV for long contexts: N(0, 1) in the cache dtype (keys taken as
  already rotated);
* page tables: a seeded shuffle of the page pool.
Seeds: weights 0, KV 1, tokens 2, acceptance draws 3; gains: the weight seed + 1000.
"""
from dataclasses import dataclass
from typing import Dict, List, Optional

import torch

from .configs import BF16, F32, PAGE, Q4_0, DrafterShape, TargetShape

SEED_WEIGHTS, SEED_KV, SEED_TOKENS, SEED_ALPHA = 0, 1, 2, 3
SEED_GAINS = 1000       # offset of the norm-gain stream from the weight seed
GAIN_STD = 0.1


@dataclass
class WTensor:
    """A stack of L matrices [N][K] in one storage format.

    f32 / bf16: data [L, N, K].  q4_0: data uint8 [L, N, K/2] (codes; element i
    of a 32-block is the low nibble of byte i for i < 16, the high nibble of
    byte i-16 otherwise) and scales fp16 [L, N, K/32]."""
    dtype: str
    L: int
    N: int
    K: int
    data: torch.Tensor
    scales: Optional[torch.Tensor] = None

    def nbytes(self) -> int:
        n = self.data.numel() * self.data.element_size()
        if self.scales is not None:
            n += self.scales.numel() * self.scales.element_size()
        return n


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(g, shape, std, dtype, device, chunk_rows=4096) -> torch.Tensor:
    """N(0, std) drawn in float32 row chunks (bounded temporary memory), cast."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1, shape[-1])
    for r0 in range(0, flat.shape[0], chunk_rows):
        r1 = min(flat.shape[0], r0 + chunk_rows)
        flat[r0:r1] = (torch.randn((r1 - r0, shape[-1]), generator=g, device=device) * std).to(dtype)
    return out


def _gains(seed: int, device):
    """Draws RMSNorm gain vectors 1 + N(0, GAIN_STD) (float32) one after another
    from one seeded stream."""
    g = _gen(seed, device)

    def draw(*shape):
        return 1.0 + torch.randn(shape, generator=g, device=device) * GAIN_STD
    return draw


def _q4_0(g, L, N, K, device, chunk_rows=4096) -> WTensor:
    codes = torch.empty((L, N, K // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((L, N, K // 32), dtype=torch.float16, device=device)
    cf, sf = codes.view(-1, K // 2), scales.view(-1, K // 32)
    for r0 in range(0, cf.shape[0], chunk_rows):
        r1 = min(cf.shape[0], r0 + chunk_rows)
        c = torch.randint(0, 16, (r1 - r0, K // 32, 32), generator=g, device=device,
                          dtype=torch.int32)
        cf[r0:r1] = (c[..., :16] | (c[..., 16:] << 4)).to(torch.uint8).view(r1 - r0, K // 2)
        sf[r0:r1] = (torch.randn((r1 - r0, K // 32), generator=g, device=device) * 0.004).abs().half()
    return WTensor(Q4_0, L, N, K, codes, scales)


def make_matrix(g, dtype: str, L: int, N: int, K: int, std: float, device) -> WTensor:
    if dtype == Q4_0:
        assert K % 32 == 0
        return _q4_0(g, L, N, K, device)
    tdt = torch.float32 if dtype == F32 else torch.bfloat16
    return WTensor(dtype, L, N, K, _normal(g, (L, N, K), std, tdt, device))


@dataclass
class TargetWeights:
    shape: TargetShape
    embed: WTensor          # [V][d]; also the tied LM head
    wqkv: WTensor           # L x [(nq+2nkv)hd][d]
    wo: WTensor             # L x [d][nq hd]
    wgu: WTensor            # L x [2ff][d]: gate rows then up rows
    wdown: WTensor          # L x [d][ff]
    g_attn: torch.Tensor    # f32 [L][d]
    g_ffn: torch.Tensor     # f32 [L][d]
    g_final: torch.Tensor   # f32 [d]
    router: Optional[WTensor] = None    # mixture of experts: L x [E][d]
    wgu_e: Optional[WTensor] = None     # (L*E) x [2 ff_e][d]: gate rows then up rows
    wdown_e: Optional[WTensor] = None   # (L*E) x [d][ff_e]

    def matrices(self) -> List[WTensor]:
        m = [self.embed, self.wqkv, self.wo, self.wgu, self.wdown]
        return m + ([self.router, self.wgu_e, self.wdown_e] if self.router is not None else [])


def make_target(t: TargetShape, device="cpu", seed=SEED_WEIGHTS) -> TargetWeights:
    g = _gen(seed, device)
    w = lambda L, N, K: make_matrix(g, t.wdtype, L, N, K, t.wstd, device)
    embed = w(1, t.V, t.d)
    wqkv = w(t.L, t.nqkv, t.d)
    wo = w(t.L, t.d, t.nq * t.hd)
    if t.n_experts:
        # mixture of experts: no dense FFN; router and experts drawn like the rest
        wgu = w(t.L, 8, t.d)
        wdown = w(t.L, t.d, 8)
        router = w(t.L, t.n_experts, t.d)
        wgu_e = w(t.L * t.n_experts, 2 * t.ff_e, t.d)
        wdown_e = w(t.L * t.n_experts, t.d, t.ff_e)
    else:
        wgu = w(t.L, 2 * t.ff, t.d)
        wdown = w(t.L, t.d, t.ff)
        router = wgu_e = wdown_e = None
    gains = _gains(seed + SEED_GAINS, device)
    return TargetWeights(t, embed, wqkv, wo, wgu, wdown, gains(t.L, t.d), gains(t.L, t.d),
                         gains(t.d), router, wgu_e, wdown_e)


@dataclass
class DrafterWeights:
    shape: DrafterShape
    w_in: WTensor           # [h][2 bh]
    g_in_h: torch.Tensor    # f32 [bh]
    g_in_e: torch.Tensor    # f32 [bh]
    wq: WTensor             # L x [nq hd][h]
    wo: WTensor             # L x [h][nq hd]
    wgu: WTensor            # L x [2ff][h]
    wdown: WTensor          # L x [h][ff]
    g_attn: torch.Tensor    # f32 [L][h]
    g_ffn: torch.Tensor     # f32 [L][h]
    g_out: torch.Tensor     # f32 [h]
    w_out: WTensor          # [bh][h]
    vocab: WTensor          # [V][h] (cluster-sorted when clustered)
    centroids: Optional[WTensor]   # [C][h]
    perm: Optional[torch.Tensor]   # int32 [V]: token id of sorted row p

    def matrices(self) -> List[WTensor]:
        m = [self.w_in, self.wq, self.wo, self.wgu, self.wdown, self.w_out, self.vocab]
        return m + ([self.centroids] if self.centroids is not None else [])


def make_drafter(dsh: DrafterShape, device="cpu", seed=SEED_WEIGHTS + 100) -> DrafterWeights:
    g = _gen(seed, device)
    w = lambda L, N, K: make_matrix(g, dsh.wdtype, L, N, K, dsh.wstd, device)
    w_in = w(1, dsh.h, 2 * dsh.bh)
    wq = w(dsh.L, dsh.nq * dsh.hd, dsh.h)
    wo = w(dsh.L, dsh.h, dsh.nq * dsh.hd)
    wgu = w(dsh.L, 2 * dsh.ff, dsh.h)
    wdown = w(dsh.L, dsh.h, dsh.ff)
    w_out = w(1, dsh.bh, dsh.h)
    centroids, perm = None, None
    if dsh.clustered:
        C, cs = dsh.n_centroids, dsh.cluster_size
        perm = torch.randperm(dsh.V, generator=g, device=device).to(torch.int32)
        if dsh.wdtype == Q4_0:
            centroids = w(1, C, dsh.h)
            vocab = w(1, dsh.V, dsh.h)
        else:
            tdt = torch.float32 if dsh.wdtype == F32 else torch.bfloat16
            cen = torch.randn((C, dsh.h), generator=g, device=device) * dsh.wstd
            noise = torch.randn((C, cs, dsh.h), generator=g, device=device) * (dsh.wstd / 2)
            members = (cen[:, None, :] + noise).reshape(1, dsh.V, dsh.h)
            centroids = WTensor(dsh.wdtype, 1, C, dsh.h, cen.reshape(1, C, dsh.h).to(tdt))
            vocab = WTensor(dsh.wdtype, 1, dsh.V, dsh.h, members.to(tdt))
    else:
        vocab = w(1, dsh.V, dsh.h)
    gains = _gains(seed + SEED_GAINS, device)
    return DrafterWeights(dsh, w_in, gains(dsh.bh), gains(dsh.bh), wq, wo, wgu, wdown,
                          gains(dsh.L, dsh.h), gains(dsh.L, dsh.h), gains(dsh.h), w_out, vocab,
                          centroids, perm)


def make_tokens(n: int, V: int, device="cpu", seed=SEED_TOKENS) -> torch.Tensor:
    return torch.randint(0, V, (n,), generator=_gen(seed, device), device=device,
                         dtype=torch.int64).to(torch.int32)


def make_context_lengths(B: int, lo: int, hi: int, seed=SEED_TOKENS + 10) -> List[int]:
    if lo == hi:
        return [lo] * B
    g = _gen(seed, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


def make_prefilled_kv(t: TargetShape, n_pos: int, device="cpu", seed=SEED_KV) -> torch.Tensor:
    """Cache contents for positions [0, n_pos) of one sequence, contiguous
    [L][2][nkv][n_pos][hd] in the cache dtype, N(0, 1)."""
    tdt = torch.float32 if t.kvdtype == F32 else torch.bfloat16
    g = _gen(seed, device)
    out = torch.empty((t.L, 2, t.nkv, n_pos, t.hd), dtype=tdt, device=device)
    for l in range(t.L):
        out[l] = torch.randn((2, t.nkv, n_pos, t.hd), generator=g, device=device).to(tdt)
    return out


def make_page_table(B: int, pages_per_seq: int, n_pages: int, shuffle: bool, device="cpu",
                    seed=SEED_KV + 10) -> torch.Tensor:
    """Block table int32 [B][pages_per_seq]: distinct page ids of a pool of n_pages."""
    assert B * pages_per_seq <= n_pages
    if shuffle:
        ids = torch.randperm(n_pages, generator=_gen(seed, "cpu"))[: B * pages_per_seq]
    else:
        ids = torch.arange(B * pages_per_seq)
    return ids.to(torch.int32).view(B, pages_per_seq).to(device)


def scatter_to_pages(pool: torch.Tensor, contig: torch.Tensor, block_row: torch.Tensor) -> None:
    """Copy contiguous cache contents [L][2][nkv][n][hd] of one sequence into a
    paged pool [L][n_pages][2][nkv][PAGE][hd] through its block-table row."""
    L, _, nkv, n, hd = contig.shape
    for p0 in range(0, n, PAGE):
        p1 = min(n, p0 + PAGE)
        page = int(block_row[p0 // PAGE])
        pool[:, page, :, :, : p1 - p0, :] = contig[:, :, :, p0:p1, :].to(pool.dtype)


def make_alpha_draws(n: int, device="cpu", seed=SEED_ALPHA) -> torch.Tensor:
    """Uniform draws in [0, 1) deciding each injected draft (float32 [n])."""
    return torch.rand((n,), generator=_gen(seed, device), device=device)


def make_wrong_offsets(n: int, V: int, device="cpu", seed=SEED_ALPHA + 1) -> torch.Tensor:
    """Uniform offsets in [1, V-1] used to build a draft that differs from the
    target's token (int32 [n])."""
    return torch.randint(1, V, (n,), generator=_gen(seed, device), device=device,
                         dtype=torch.int64).to(torch.int32)
