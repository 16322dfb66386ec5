"""The five synthetic workloads of the ZeRO shard step.

Sizes follow the ZeRO memory examples: a tiny ZeRO-2 case, a GPT-2-small-sized
flat buffer, a padding/overflow case, GPT-2 1.5B (the paper's "24 GB of model
states" example, section on quantifying memory consumption) and the 7.5B model of
the Stage-3 memory table.  Inputs are seeded and synthetic; no dataset or
trained weights are involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

ADAMW = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    psi: int                 # flat parameter count
    nd: int                  # data-parallel degree (emulated ranks)
    grad_dtype: str          # "f16" | "bf16"
    loss_scale: float        # static loss scale (fp16: 1024, bf16: 1)
    bucket: int              # fusion-buffer (CB) size in elements
    steps: int
    seed: int
    view: str                # "full": every rank's shard; "shard": one rank
    fresh_grads: bool        # new gradients every step (else fixed)
    m_sigma: float | None    # None -> m = 0
    v_sigma: float | None    # None -> v = 0 ; else v = |N(0, v_sigma)|
    master_sigma: float = 0.02
    grad_sigma: float = 1e-3
    plant: tuple | None = None   # (step, contributor, flat index) of a +inf
    hparams: dict = field(default_factory=lambda: dict(ADAMW))

    @property
    def shard(self) -> int:
        return -(-self.psi // self.nd)

    @property
    def torch_grad_dtype(self) -> torch.dtype:
        return torch.float16 if self.grad_dtype == "f16" else torch.bfloat16

    @property
    def bytes_per_param(self) -> int:
        """Algorithmic HBM bytes per updated parameter: Nd 2-byte gradient
        reads, 12 B of fp32 state read, 12 B written, 2 B cast written."""
        return 2 * self.nd + 26


def _c2_plant():
    psi, nd = 350_000_017, 16
    s = -(-psi // nd)
    return (5, 7, 7 * s + s // 2)


WORKLOADS = {
    "c0": Workload("c0", "tiny ZeRO-2 step", 1_048_576, 4, "f16", 1024.0, 65_536, 3, 0,
                   "full", True, None, None),
    "c1": Workload("c1", "GPT-2-small-sized flat buffer, ZeRO-2", 124_439_808, 8, "bf16",
                   1.0, 50_000_000, 10, 1, "shard", True, 1e-4, 1e-6),
    "c2": Workload("c2", "padding and overflow, ZeRO-2", 350_000_017, 16, "f16", 1024.0,
                   50_000_000, 6, 2, "full", False, None, None, plant=_c2_plant()),
    "c3": Workload("c3", "GPT-2 1.5B, ZeRO-3 shard view", 1_500_000_000, 64, "f16", 1024.0,
                   50_000_000, 20, 3, "shard", False, 1e-4, 1e-6),
    "c4": Workload("c4", "7.5B model, ZeRO-3 shard view", 7_500_000_000, 64, "bf16", 1.0,
                   500_000_000, 20, 4, "shard", False, 1e-4, 1e-6),
}
