"""Workload shapes for the wave-index hot path (sizes only; no method arithmetic).

Shapes follow the RetroInfer summaries' workloads: Llama3-8B / Qwen2.5-7B
shaped GQA attention (head_dim 128) at 128K..1M-token contexts, segmented
clustering with 512 clusters per 8192-token segment, a steady zone of 4 sink
plus 64 local tokens, and a retrieval budget of about 1.8% of the clusters
(summary page zh, section 3).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_ctx: int
    seg_len: int
    clusters_per_seg: int
    iters: int
    n_sink: int
    local_window: int
    budget_frac: float
    budget_k: int          # 0: derive from budget_frac
    n_topics: int
    decode_steps: int      # decode steps in the workload
    append: bool           # each decode step appends one token after attending
    seed: int
    # generator distribution
    p_stay: float = 0.95
    sigma_k: float = 0.3
    sink_scale: float = 4.0
    rope_theta: float = 500000.0
    q_scale: float = 1.5
    sigma_q: float = 0.3

    @property
    def units(self) -> int:
        return self.batch * self.layers * self.n_kv_heads

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def n_segments(self) -> int:
        return self.n_ctx // self.seg_len

    @property
    def clusters(self) -> int:
        return self.n_segments * self.clusters_per_seg

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # single unit, one segment: the small case
    "tiny-8k": Workload("tiny-8k", 1, 1, 1, 1, 128, 8192, 8192, 512, 10, 4, 64, 0.018, 10, 64, 1, False, 0),
    # Llama-3-8B-shaped single-layer decode, 131072 tokens
    "llama3-8b-131k": Workload("llama3-8b-131k", 1, 1, 32, 8, 128, 131072, 8192, 512, 10, 4, 64, 0.018, 0, 64,
                               1, False, 1),
    # batch 16 at 120K tokens
    "llama3-8b-b16-120k": Workload("llama3-8b-b16-120k", 16, 1, 32, 8, 128, 122880, 8192, 512, 10, 4, 64, 0.018,
                                   0, 64, 1, False, 2),
    # one million tokens across 32 layers
    "llama3-8b-1m-32l": Workload("llama3-8b-1m-32l", 1, 32, 32, 8, 128, 1048576, 8192, 512, 10, 4, 64, 0.018, 0,
                                 256, 1, False, 3),
    # Qwen2.5-7B-shaped build plus 64 decode steps with append
    "qwen2.5-7b-b8-262k": Workload("qwen2.5-7b-b8-262k", 8, 1, 28, 4, 128, 262144, 8192, 512, 10, 4, 64, 0.018, 0,
                                   64, 64, True, 4),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
