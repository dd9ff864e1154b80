"""Model and workload shapes.

Shapes only: no arithmetic of the method lives here. The target models are
synthetic decoders shaped like the pages' E2B / E4B edge models and a ~30B dense
model; the drafter is the 4-layer, width-256 head that reads the target's
backbone-width hidden state ("Gemma 4's MTP drafter explained" (molayo1419.me),
section "What is different about Gemma 4's drafter?": hidden_size 256,
backbone_hidden_size 1536 for E2B and 2560 for E4B, 4 layers; num_centroids 2048
for the clustered output shortcut).
"""
from dataclasses import dataclass, field, replace
from typing import Optional, Tuple

F32, BF16, Q4_0 = "f32", "bf16", "q4_0"
PAGE = 64  # tokens per KV page


@dataclass(frozen=True)
class TargetShape:
    L: int
    d: int
    nq: int
    nkv: int
    hd: int
    ff: int
    V: int
    wdtype: str
    kvdtype: str
    wstd: float
    eps: float = 1e-6
    theta: float = 10000.0
    n_experts: int = 0            # mixture of experts: experts per layer (0: dense FFN)
    top_k: int = 0                # experts each row uses
    ff_e: int = 0                 # width of one expert's FFN

    @property
    def nqkv(self) -> int:
        return (self.nq + 2 * self.nkv) * self.hd

    def weight_bytes(self) -> int:
        """Bytes of every linear weight plus the tied embedding / LM head."""
        per = {F32: 4.0, BF16: 2.0, Q4_0: 0.5 + 2.0 / 32}[self.wdtype]
        ffn = 3 * self.d * self.ff if not self.n_experts else self.n_experts * (3 * self.d * self.ff_e + self.d)
        layer = self.d * self.nqkv + self.d * self.nq * self.hd + ffn
        return int(round((self.L * layer + self.V * self.d) * per))

    def kv_bytes_per_pos(self) -> int:
        """K and V of one position over all layers."""
        return self.L * 2 * self.nkv * self.hd * (4 if self.kvdtype == F32 else 2)


@dataclass(frozen=True)
class DrafterShape:
    L: int
    h: int
    bh: int
    ff: int
    nq: int
    hd: int
    nkv: int
    V: int
    wdtype: str
    wstd: float
    clustered: bool
    n_centroids: int = 0
    top_c: int = 0

    @property
    def cluster_size(self) -> int:
        return self.V // self.n_centroids if self.clustered else 0


@dataclass(frozen=True)
class Workload:
    name: str
    target: TargetShape
    drafter: DrafterShape
    B: int
    ctx: Tuple[int, int]          # context length range [lo, hi] (lo == hi: fixed)
    k: int
    alphas: Tuple[float, ...]
    prompt: bool = False          # True: real prefill of a uniform random prompt of length ctx
    steps: int = 16

    @property
    def M(self) -> int:
        return self.B * (self.k + 1)


def _drafter(t: TargetShape, L: int, h: int, clustered: bool, wdtype: Optional[str] = None):
    return DrafterShape(L=L, h=h, bh=t.d, ff=4 * h, nq=t.nq, hd=t.hd, nkv=t.nkv, V=t.V,
                        wdtype=wdtype or t.wdtype, wstd=t.wstd, clustered=clustered,
                        n_centroids=2048 if clustered else 0, top_c=32 if clustered else 0)


TINY = TargetShape(L=2, d=256, nq=4, nkv=4, hd=64, ff=1024, V=4096, wdtype=F32, kvdtype=F32,
                   wstd=0.02)
E2B = TargetShape(L=24, d=1536, nq=12, nkv=4, hd=128, ff=6144, V=262144, wdtype=BF16,
                  kvdtype=BF16, wstd=0.02)
E2B_Q4 = replace(E2B, wdtype=Q4_0)
E4B = TargetShape(L=32, d=2560, nq=20, nkv=4, hd=128, ff=10240, V=262144, wdtype=BF16,
                  kvdtype=BF16, wstd=0.02)
DENSE30B = TargetShape(L=48, d=6144, nq=48, nkv=8, hd=128, ff=24576, V=262144, wdtype=BF16,
                       kvdtype=BF16, wstd=0.01)

# Mixture-of-experts targets ("Gemma 4 acceleration: faster inference with
# multi-token prediction drafters" (cafe.daangn.com), "MTP drafter internal
# optimisations": a 26B mixture-of-experts model, little gain at batch 1 because
# of routing, about 2.2x at batch 4-8). The pages give no layer shapes: these
# are synthetic, with each row using top_k of n_experts gated-GELU experts.
TINY_MOE = TargetShape(L=2, d=256, nq=4, nkv=4, hd=64, ff=256, V=4096, wdtype=F32, kvdtype=F32, wstd=0.02,
                       n_experts=8, top_k=2, ff_e=256)
MOE = TargetShape(L=16, d=2048, nq=16, nkv=8, hd=128, ff=1024, V=262144, wdtype=BF16, kvdtype=BF16,
                  wstd=0.02, n_experts=64, top_k=4, ff_e=1024)

WORKLOADS = {
    "tiny_f32_b1_k3": Workload("tiny_f32_b1_k3", TINY, _drafter(TINY, 1, 64, False), B=1,
                               ctx=(64, 64), k=3, alphas=(), prompt=True, steps=16),
    "e2b_bf16_b1_ctx2048_k3": Workload("e2b_bf16_b1_ctx2048_k3", E2B, _drafter(E2B, 4, 256, True),
                                       B=1, ctx=(2048, 2048), k=3, alphas=(0.0, 0.5, 0.8)),
    "e2b_q4_0_b1_ctx4096_k4": Workload("e2b_q4_0_b1_ctx4096_k4", E2B_Q4,
                                       _drafter(E2B_Q4, 4, 256, True), B=1, ctx=(4096, 4096),
                                       k=4, alphas=(0.7,)),
    "e2b_q4_0_b4_ctx4096_k4": Workload("e2b_q4_0_b4_ctx4096_k4", E2B_Q4,
                                       _drafter(E2B_Q4, 4, 256, True), B=4, ctx=(4096, 4096),
                                       k=4, alphas=(0.7,)),
    "e4b_bf16_b8_ragged_k4": Workload("e4b_bf16_b8_ragged_k4", E4B, _drafter(E4B, 4, 256, True),
                                      B=8, ctx=(1024, 8192), k=4, alphas=(0.6,)),
    "dense30b_bf16_b1_ctx8192_k4": Workload("dense30b_bf16_b1_ctx8192_k4", DENSE30B,
                                            _drafter(DENSE30B, 4, 256, True), B=1,
                                            ctx=(8192, 8192), k=4, alphas=(0.5, 0.8)),
    "dense30b_bf16_b8_ctx8192_k4": Workload("dense30b_bf16_b8_ctx8192_k4", DENSE30B,
                                            _drafter(DENSE30B, 4, 256, True), B=8,
                                            ctx=(8192, 8192), k=4, alphas=(0.5, 0.8)),
    "moe_bf16_b8_ctx4096_k4": Workload("moe_bf16_b8_ctx4096_k4", MOE, _drafter(MOE, 4, 256, True), B=8,
                                       ctx=(4096, 4096), k=4, alphas=(0.7,)),
}

BENCH_WORKLOAD = "dense30b_bf16_b8_ctx8192_k4"
