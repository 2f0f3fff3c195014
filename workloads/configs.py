"""The five synthetic MoE-layer workloads, by name and shape.

Shapes follow the model families the PagedWeight pages evaluate on
(PagedWeight, "Main contributions" item 4 and "Results": Qwen1.5-MoE-A2.7B,
Mixtral-8x7B) plus a Qwen3-30B-A3B-shaped layer; the pages print no layer
sizes, so the sizes below are the public architecture sizes of those models.

Every workload is a single routed-expert layer:
  T tokens, hidden size H, expert intermediate size I, E experts, top-k routing.
  Each expert e owns two linear blocks, block id 2e (gate_up, [2I x H]) and
  2e+1 (down, [H x I]).
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple

BITWIDTHS = (3, 4, 5, 6, 8)


@dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int
    I: int
    E: int
    k: int
    T: Tuple[int, ...]
    # q distribution: "uniform" (draw from BITWIDTHS per block), "hot8_rest34"
    # (experts in `hot` held at 8, others drawn from {3, 4}), "zipf_floor6"
    # (draw from BITWIDTHS, experts with popularity > 1/E floored at 6).
    q_mode: str = "uniform"
    # router logits: "normal" (N(0,1)), "bias2" (+2.0 on experts in `hot`),
    # "zipf" (+log p_e with p_e proportional to (e+1)^-zipf_s).
    logit_mode: str = "normal"
    hot: Tuple[int, ...] = ()
    zipf_s: float = 1.1
    prefill: bool = False
    recommit_frac: float = 0.0
    description: str = field(default="", compare=False)


CONFIGS = (
    LayerConfig("tiny", H=256, I=512, E=8, k=2, T=(16,),
                description="tiny single layer, 16 tokens"),
    LayerConfig("qwen15_decode", H=2048, I=1408, E=60, k=4, T=(1, 4, 8),
                description="Qwen1.5-MoE-A2.7B-shaped routed layer, decode"),
    LayerConfig("mixtral_decode", H=4096, I=14336, E=8, k=2, T=(4,),
                q_mode="hot8_rest34", logit_mode="bias2", hot=(0, 1),
                description="Mixtral-8x7B-shaped layer, decode, 2 hot experts"),
    LayerConfig("qwen3_decode", H=2048, I=768, E=128, k=8, T=(64,),
                q_mode="zipf_floor6", logit_mode="zipf", recommit_frac=0.25,
                description="Qwen3-30B-A3B-shaped layer, decode, Zipf routing, "
                            "recommit of 25% of blocks between steps"),
    LayerConfig("mixtral_prefill", H=4096, I=14336, E=8, k=2, T=(4096,),
                prefill=True,
                description="Mixtral-8x7B-shaped layer, prefill"),
)


def config_by_name(name: str) -> LayerConfig:
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def custom(name: str, H: int, I: int, E: int, k: int, T: int,
           q_mode: str = "uniform", logit_mode: str = "normal",
           hot: Optional[Tuple[int, ...]] = None) -> LayerConfig:
    """A small ad-hoc shape for tests (ragged tails, degenerate cases)."""
    return LayerConfig(name, H=H, I=I, E=E, k=k, T=(T,), q_mode=q_mode,
                       logit_mode=logit_mode, hot=tuple(hot or ()))
