"""A small training loop for the signal test (run as a child process on the
GPU): clipped-AdamW steps on generator gradients, ckpt_step_end after each
step with checkpoints only on signals.  Prints "step <k>" after each step;
exits 0 after a SIGTERM checkpoint."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import optimizer_step_resumable_gb300 as osr  # noqa: E402
from synthetic import device as synth_dev  # noqa: E402


def main():
    n, ckdir, max_steps = int(sys.argv[1]), sys.argv[2], int(sys.argv[3])
    dev = torch.device("cuda:0")
    w = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, 7)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    g = torch.empty(n, device=dev)
    osr.ckpt_signals_install()
    ctx = osr.adamw_create(n)
    side = torch.cuda.Stream()
    print("ready", flush=True)
    for t in range(1, max_steps + 1):
        synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
        osr.adamw_clip_step(ctx, w, g, m, v, t, 3e-3, 0.01, 1.0)
        action = osr.ckpt_step_end(ctx, t, w, m, v, ckdir, 0, side_stream=side)
        torch.cuda.synchronize()
        print(f"step {t} {action}", flush=True)
        if action == osr.CKPT_ACTION_EXIT:
            ctx.close()
            return 0
        time.sleep(0.002)
    ctx.close()
    return 3


if __name__ == "__main__":
    sys.exit(main())
