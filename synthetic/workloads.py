"""The synthetic workloads: sizes, layouts, input distributions, hyperparameters.

Inputs only; no optimizer arithmetic.  Sizes follow the pages' models
("Grow a Language Model: Checkpoints", section "Total size": ANDREA-12M with
12.8M parameters; "Grow a Language Model: Backprop", section "Where the
gradients live": the per-block tensors of ANDREA-120M), the seed 7 and the
hyperparameters lr = 0.003, wd = 0.01, clip = 1 of "Training as a
Recoverable State Transition" (section "Task and Prerequisites").
"""
from __future__ import annotations

from dataclasses import dataclass, field

SEED = 7
LR = 3e-3
WD = 0.01
CLIP = 1.0
BETA1 = 0.9
BETA2 = 0.999
EPS = 1e-8
W_SIGMA = 0.02


def gpt_110m_tensors():
    """(name, numel) in flat order: embeddings, 12 blocks, final norm.

    Per block: W_Q, W_K, W_V, W_O [768x768] with biases [768], W_1 [768x3072]
    with bias [3072], W_2 [3072x768] with bias [768], LN1 and LN2 gamma/beta
    [768].  The output head is tied to the token embedding (no extra tensor).
    196 tensors, 110,418,432 parameters.
    """
    d, ff, vocab, ctx, layers = 768, 3072, 32000, 1024, 12
    out = [("tok_emb", vocab * d), ("pos_emb", ctx * d)]
    for i in range(layers):
        p = f"h{i}."
        for k in ("q", "k", "v", "o"):
            out.append((p + f"W_{k.upper()}", d * d))
            out.append((p + f"b_{k.upper()}", d))
        out += [(p + "W_1", d * ff), (p + "b_1", ff), (p + "W_2", ff * d),
                (p + "b_2", d), (p + "ln1.gamma", d), (p + "ln1.beta", d),
                (p + "ln2.gamma", d), (p + "ln2.beta", d)]
    out += [("lnf.gamma", d), ("lnf.beta", d)]
    return out


def decay_flags_matrices_only(tensors):
    """The common alternative grouping: weight decay on matrices and
    embeddings, none on biases and normalisation gains/shifts (every 1-D
    tensor of the list).  One flag per tensor, in table order."""
    return [0 if (".b_" in name or "ln" in name) else 1 for name, _ in tensors]


def offset_table(tensors):
    """(offsets, numels) of a contiguous flat layout, in the given order."""
    offsets, numels, off = [], [], 0
    for _, k in tensors:
        offsets.append(off)
        numels.append(k)
        off += k
    return offsets, numels


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    grad_sigma: float
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    steps: int = 1
    ckpt_step: int = 0
    tensors: tuple = field(default=None)  # ((name, numel), ...) or None = flat
    lr: float = LR
    wd: float = WD
    clip: float = CLIP
    seed: int = SEED

    def table(self):
        t = self.tensors if self.tensors is not None else (("flat", self.n),)
        return offset_table(t)


def flat_65k():
    return Workload("flat-65536", 65536, 1e-2, outlier_frac=0.01,
                    outlier_mult=100.0, steps=80, ckpt_step=80)


def flat_12m8():
    return Workload("flat-12.8M", 12_800_000, 1e-3, steps=100, ckpt_step=100)


def gpt_110m(steps=1, ckpt_step=0):
    t = tuple(gpt_110m_tensors())
    return Workload("gpt-110M-list", sum(k for _, k in t), 1e-3, steps=steps,
                    ckpt_step=ckpt_step, tensors=t)


def gpt_110m_resume():
    return gpt_110m(steps=200, ckpt_step=100)


def flat_pow2(log2n: int):
    return Workload(f"flat-2^{log2n}", 1 << log2n, 1e-3, outlier_frac=0.001,
                    outlier_mult=1000.0)


WORKLOADS = {
    "flat-65536": flat_65k,
    "flat-12.8M": flat_12m8,
    "gpt-110M-list": gpt_110m,
    "gpt-110M-resume": gpt_110m_resume,
}
