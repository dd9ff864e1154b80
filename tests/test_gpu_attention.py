"""Kernel-level parity of the paged attention (spec_attention, the kernels the
verify pass and the drafter run) against the oracle's attention at fp32-level
tolerance.

The cache holds exact bf16 (or fp32) keys and values; the queries are fp32.
For every (row, query head) the oracle computes softmax(q K^T / sqrt(hd)) V
over exactly the keys that row may see, read from a contiguous copy of the
paged cache: [0, seq_len + i] for verify row i (key_extra = 1: the row's own
key and those of earlier rows of the pass included), [0, seq_len) for the
drafter's rows (key_extra = 0). A mask that is off by one key, a dropped last
page or a wrong GQA mapping moves some output by far more than the 1e-4
relative tolerance used here (the end-to-end logits tolerance of 2e-2 could
not see a one-key error over thousands of keys).

Cases: single sequences whose visible key counts straddle the 64-key pages
(1, 63, 64, 65 keys) and long contexts (2048, 8192), at the GQA groups of the
E2B- (12/4), E4B- (20/4) and ~30B-class (48/8) models with head_dim 128 and
of the tiny bf16 model (4/4, head_dim 64); verify rows (R = 4, 5), one-row
decode and the drafter's rows; a ragged batch of 8 with shuffled pages (the
batched launch)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import rel_rows

pytestmark = pytest.mark.gpu
TOL = 1e-4
PAGE = configs.PAGE


def _shape(nq, nkv, hd, kv=configs.BF16):
    return configs.TargetShape(L=2, d=256, nq=nq, nkv=nkv, hd=hd, ff=256, V=256, wdtype=configs.BF16,
                               kvdtype=kv, wstd=0.02)


def _run(t, lens, R, key_extra, layer=1, seed=0):
    """Random cache for every slot up to its visible keys, random queries;
    returns (gpu out, oracle out) as [B*R][nq][hd]."""
    B = len(lens)
    g = torch.Generator(device="cuda").manual_seed(seed)
    need = [L_ + (R if key_extra else 0) for L_ in lens]
    max_pages = max(1, (max(need) + PAGE - 1) // PAGE)
    n_pages = B * max_pages
    dt = torch.bfloat16 if t.kvdtype == configs.BF16 else torch.float32
    pool = torch.randn((t.L, n_pages, 2, t.nkv, PAGE, t.hd), generator=g, device="cuda").to(dt)
    bt = synth.make_page_table(B, max_pages, n_pages, shuffle=B > 1, device="cuda", seed=seed + 10)
    seq_ids = torch.arange(B, dtype=torch.int32, device="cuda")
    seq_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    q = torch.randn((B * R, t.nq * t.hd), generator=g, device="cuda")
    out = binding.spec_attention(t, pool, bt, layer, seq_ids, seq_len, R, t.nq, key_extra, q)
    torch.cuda.synchronize()
    assert int(out.workspace[:4].view(torch.int32)[0]) == 0
    # oracle on a contiguous copy of each sequence's keys/values
    poolc = pool[layer].float().cpu().numpy()          # [n_pages][2][nkv][64][hd]
    btc = bt.cpu().numpy()
    qc = q.cpu().numpy().astype(np.float64).reshape(B * R, t.nq, t.hd)
    ref = np.zeros_like(qc)
    grp = t.nq // t.nkv
    for b in range(B):
        n_all = need[b]
        pages = [poolc[btc[b, p]] for p in range((n_all + PAGE - 1) // PAGE)]
        K = np.concatenate([pg[0] for pg in pages], axis=1)[:, :n_all]   # [nkv][n][hd]
        V = np.concatenate([pg[1] for pg in pages], axis=1)[:, :n_all]
        for i in range(R):
            nk = lens[b] + i + 1 if key_extra else lens[b]
            for h in range(t.nq):
                ref[b * R + i, h] = oracle.attend(qc[b * R + i, h], np.ascontiguousarray(K[h // grp, :nk]),
                                                  np.ascontiguousarray(V[h // grp, :nk]))
    return out.cpu().numpy().reshape(B * R, t.nq, t.hd), ref


def _check(gpu, ref, what):
    r = rel_rows(gpu.reshape(-1, gpu.shape[-1]), ref.reshape(-1, ref.shape[-1]))
    assert r.max() <= TOL, "%s: worst (row, head) relative error %.3e" % (what, r.max())


GQA = {"e2b": (12, 4, 128), "e4b": (20, 4, 128), "dense30b": (48, 8, 128), "tiny_bf16": (4, 4, 64)}


@pytest.mark.parametrize("model", sorted(GQA))
@pytest.mark.parametrize("keys_last_row", [1, 63, 64, 65, 2048])
def test_verify_rows_single_sequence(model, keys_last_row):
    t = _shape(*GQA[model])
    R = 5 if model in ("e4b", "dense30b") else 4
    seq_len = max(keys_last_row - R, 0)
    R = min(R, keys_last_row) if seq_len == 0 else R
    gpu, ref = _run(t, [seq_len], R, 1)
    _check(gpu, ref, "%s verify seq_len %d R %d" % (model, seq_len, R))


@pytest.mark.parametrize("model", ["e2b", "dense30b"])
@pytest.mark.parametrize("ctx", [8192])
def test_verify_rows_long_context(model, ctx):
    t = _shape(*GQA[model])
    gpu, ref = _run(t, [ctx - 5], 5, 1, seed=3)
    _check(gpu, ref, "%s verify ctx %d" % (model, ctx))


@pytest.mark.parametrize("model", sorted(GQA))
@pytest.mark.parametrize("seq_len", [1, 64, 65, 4095])
def test_decode_row(model, seq_len):
    t = _shape(*GQA[model])
    gpu, ref = _run(t, [seq_len - 1], 1, 1, seed=4)
    _check(gpu, ref, "%s decode" % model)


@pytest.mark.parametrize("model", sorted(GQA))
@pytest.mark.parametrize("seq_len", [1, 63, 64, 65, 2048])
def test_drafter_rows(model, seq_len):
    t = _shape(*GQA[model])
    gpu, ref = _run(t, [seq_len], 1, 0, layer=1, seed=5)
    _check(gpu, ref, "%s drafter" % model)


@pytest.mark.parametrize("model", ["e4b", "dense30b"])
@pytest.mark.parametrize("key_extra,R", [(1, 5), (0, 1), (1, 1)])
def test_ragged_batch_shuffled_pages(model, key_extra, R):
    t = _shape(*GQA[model])
    lens = [1024, 8187, 1, 63, 4096, 65, 3000, 64]
    gpu, ref = _run(t, lens, R, key_extra, seed=6)
    _check(gpu, ref, "%s batch key_extra %d R %d" % (model, key_extra, R))


@pytest.mark.parametrize("key_extra,R", [(1, 4), (0, 1)])
def test_fp32_cache(key_extra, R):
    t = _shape(4, 4, 64, kv=configs.F32)
    gpu, ref = _run(t, [130], R, key_extra, seed=7)
    _check(gpu, ref, "fp32 cache")
