"""The five synthetic workloads of the tree-verify path, as data.

Each workload fixes the shapes, dtypes, tree recipe and value distributions of
one benchmark case.  Nothing here computes any part of the method; the module
only describes inputs.

Shapes follow the pages' own settings:
  * tree recipes (num_steps / topk / num_draft_tokens) -- "Speculative Decoding"
    (SGLang docs), section "EAGLE Decoding" and the EAGLE-2 launch examples;
  * 64-node trees -- "Tech Radar: SGLang EAGLE-2", section 2 (sequence diagram)
    and section 5 (64-bit ancestry bitmask, K <= 64);
  * Llama-family attention shapes (8B: 32/8 heads, 70B: 64/8, Llama-2-7B: 32/32,
    head_dim 128) -- the models named in the same pages' benchmarks.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    cfg_id: int                 # seed namespace: every stream is keyed by it
    batch: int
    prefix_lo: int              # prefix length per sequence, uniform in [lo, hi]
    prefix_hi: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str                  # "f32" or "bf16" (storage of q / K / V / out)
    num_steps: int              # draft depth
    topk: int                   # branching per draft step
    num_nodes: int              # tree nodes N, root included
    vary_tree: bool             # a different tree shape per sequence
    vocab: int
    logit_std: float            # target logits ~ N(0, logit_std^2)
    temperature: float          # 0 => greedy acceptance
    shuffle_pages: bool = True

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def rows_per_kv_head(self) -> int:
        return self.num_nodes * self.group

    @property
    def greedy(self) -> bool:
        return self.temperature == 0.0

    def with_batch(self, batch: int) -> "Workload":
        return replace(self, batch=batch, name=f"{self.name.split('@')[0]}@b{batch}")


# 1: tiny fp32 greedy case the oracle finishes instantly.
C1 = Workload("c1_tiny_f32_greedy", 1, 1, 64, 64, 4, 1, 64, 16, "f32",
              num_steps=3, topk=2, num_nodes=8, vary_tree=False,
              vocab=256, logit_std=3.0, temperature=0.0)
# 2: Llama-3-8B attention shape, greedy.
C2 = Workload("c2_llama3_8b_bf16_greedy", 2, 1, 2048, 2048, 32, 8, 128, 16, "bf16",
              num_steps=5, topk=4, num_nodes=8, vary_tree=False,
              vocab=128256, logit_std=3.0, temperature=0.0)
# 3: Llama-2-7B shape (MHA), stochastic at T = 1.
C3 = Workload("c3_llama2_7b_bf16_stoch", 3, 8, 4096, 4096, 32, 32, 128, 16, "bf16",
              num_steps=3, topk=4, num_nodes=16, vary_tree=False,
              vocab=32000, logit_std=2.0, temperature=1.0)
# 4: Llama-3-70B attention shape with a 64-node tree; greedy and T = 0.7.
C4_GREEDY = Workload("c4_llama3_70b_bf16_greedy", 4, 32, 8192, 8192, 64, 8, 128, 16, "bf16",
                     num_steps=6, topk=8, num_nodes=64, vary_tree=False,
                     vocab=128256, logit_std=3.0, temperature=0.0)
C4_STOCH = replace(C4_GREEDY, name="c4_llama3_70b_bf16_t0.7", temperature=0.7)
# 5: ragged large batch, per-sequence tree shapes, stochastic at T = 1.
C5 = Workload("c5_ragged_b64_bf16_stoch", 5, 64, 512, 32768, 32, 8, 128, 16, "bf16",
              num_steps=4, topk=4, num_nodes=16, vary_tree=True,
              vocab=128256, logit_std=3.0, temperature=1.0)

WORKLOADS = {w.name: w for w in (C1, C2, C3, C4_GREEDY, C4_STOCH, C5)}


def get(name: str) -> Workload:
    """Look up a workload; "<name>@b<B>" selects another batch size."""
    if "@b" in name:
        base, b = name.split("@b")
        return WORKLOADS[base].with_batch(int(b))
    return WORKLOADS[name]
