"""Named workloads of the MoE expert layer (shapes of a Qwen3.6-35B-A3B layer).

The five workloads are:
  tiny      T=16,   H=256,  E=16,  top-2, I=128, 1 shared expert, 1 layer
  prefill   T=512,  H=2048, E=256, top-8, I=512, 1 shared expert, 1 layer
  skewed    T=2048, same layer, router logits shifted by a Zipf(s=1.1) bias
  decode    T=1,    same layer, 40 distinct stacked layers
  chunked   T=16384 in chunks of 2048 tokens, 40 stacked layers
"""
from dataclasses import dataclass


@dataclass(frozen=True)
class LayerShape:
    H: int          # hidden size
    E: int          # routed experts
    K: int          # experts selected per token
    I: int          # expert intermediate size (routed and shared)
    n_shared: int   # always-on shared experts (0 or 1)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                  # tokens per layer call
    shape: LayerShape
    layers: int = 1         # distinct stacked layers
    zipf_s: float = 0.0     # >0: per-expert router bias -s*ln(rank)
    chunk: int = 0          # >0: tokens per chunk (bounded-chunk prefill)
    total_tokens: int = 0   # tokens of the whole prompt when chunked
    seed: int = 0


FULL = LayerShape(H=2048, E=256, K=8, I=512, n_shared=1)
TINY = LayerShape(H=256, E=16, K=2, I=128, n_shared=1)

CONFIGS = {
    "tiny": Workload("tiny", T=16, shape=TINY),
    "prefill": Workload("prefill", T=512, shape=FULL),
    "skewed": Workload("skewed", T=2048, shape=FULL, zipf_s=1.1),
    "decode": Workload("decode", T=1, shape=FULL, layers=40),
    "chunked": Workload("chunked", T=2048, shape=FULL, layers=40, chunk=2048,
                        total_tokens=16384),
}


def workload(name: str) -> Workload:
    return CONFIGS[name]
