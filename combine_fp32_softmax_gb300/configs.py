"""Named MoE-layer workloads.

Each workload is one MoE layer (UniEP page, section 1.1, Figure 1: gate ->
top-k -> dispatch -> GroupGEMM -> SwiGLU -> GroupGEMM -> combine) with
synthetic, seeded inputs.  ``T`` tokens, model width ``d``, expert hidden
width ``f`` (SwiGLU), ``E`` routed experts, top-``k`` routing, ``S``
always-on shared experts, ``renorm`` (0: routing weight = softmax
probability; 1: probabilities renormalised over the selected k), ``zipf``
(per-expert logit bias 2*ln(Zipf(1.2) rank weight), heavy-tailed load).
"""
from dataclasses import dataclass, replace


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    f: int
    E: int
    k: int
    S: int = 0
    renorm: int = 0
    zipf: bool = False

    @property
    def R(self) -> int:
        """Routed rows: one per (token, slot)."""
        return self.T * self.k

    @property
    def Rs(self) -> int:
        """Rows through the expert GEMMs: routed rows plus S*T shared rows."""
        return self.T * self.k + self.S * self.T

    def fwd_flops(self) -> int:
        """Algorithmic forward GEMM flops: 2*d*f for each of the three
        projections of every expert row."""
        return 6 * self.d * self.f * self.Rs

    def bwd_flops(self) -> int:
        """Backward GEMM flops: dH and dX (6*d*f per row) plus dW1, dW3,
        dW2 (6*d*f per row)."""
        return 12 * self.d * self.f * self.Rs

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# The five workloads: a tiny layer, a DeepSeek-V2-Lite-like layer (64 routed
# experts, top-6, 2 shared), a Mixtral-like layer (8 experts, top-2), a
# skewed-routing layer (128 experts, top-8, Zipf-biased logits) and a
# long-sequence (128k token) layer.
TINY = MoEConfig("tiny_T512_d256_f512_E8_k2", 512, 256, 512, 8, 2)
DSV2_LITE = MoEConfig("dsv2lite_T8192_d2048_f1408_E64_k6_S2", 8192, 2048, 1408, 64, 6, S=2)
MIXTRAL = MoEConfig("mixtral_T16384_d4096_f14336_E8_k2", 16384, 4096, 14336, 8, 2)
SKEWED = MoEConfig("skewed_T32768_d4096_f2048_E128_k8_zipf", 32768, 4096, 2048, 128, 8, zipf=True)
LONG128K = MoEConfig("long_T131072_d2048_f1408_E64_k6_S2", 131072, 2048, 1408, 64, 6, S=2)

ALL = [TINY, DSV2_LITE, MIXTRAL, SKEWED, LONG128K]
BY_NAME = {c.name: c for c in ALL}
