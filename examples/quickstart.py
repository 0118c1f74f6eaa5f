"""Quick start: the clipped-AdamW step over a flat float32 state, a checkpoint
every 100 steps written in the background, and a resume from the last file.

    python examples/quickstart.py [--n N] [--dir DIR]

The gradient is filled with random numbers where a training loop's backward
pass would write it.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import optimizer_step_resumable_gb300 as osr  # noqa: E402


def main(n=110_418_432, first=24_576_000, directory="ckpt", steps=200):
    """Returns (stored step of the file read back, last norm, last clip factor)."""
    w, g, m, v = (torch.zeros(n, device="cuda") for _ in range(4))  # caller-owned state
    offsets, numels = [0, first], [first, n - first]  # tensor table of the flat layout
    os.makedirs(directory, exist_ok=True)
    with osr.adamw_create(n, offsets, numels) as ctx:  # preallocates all scratch
        side = torch.cuda.Stream()
        for t in range(1, steps + 1):
            g.normal_(0.0, 1e-3)  # the backward pass writes g here
            osr.adamw_clip_step(ctx, w, g, m, v, t, lr=3e-3, wd=0.01, clip=1.0)
            if t % 100 == 0:
                osr.ckpt_pack(ctx, t, w, m, v, side_stream=side)  # device pack + copy to host
                osr.ckpt_write_async(ctx, directory)  # tmp -> fsync -> rename, background
        osr.ckpt_wait(ctx)
        norm, factor = osr.adamw_last_norm(ctx)  # raises NonFiniteGradient on inf/nan
        # validated read; a resumed run continues with t = step + 1
        step = osr.ckpt_read(ctx, os.path.join(directory, f"step_{steps:06d}.bin"), w, m, v)
    return step, norm, factor


if __name__ == "__main__":
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--n", type=int, default=110_418_432)
    p.add_argument("--dir", default="ckpt")
    a = p.parse_args()
    print(main(n=a.n, first=min(24_576_000, a.n // 2), directory=a.dir))
