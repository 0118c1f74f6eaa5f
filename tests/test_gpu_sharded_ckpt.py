"""GPU sharded checkpoint: R virtual shards (R contexts on one GPU) run the
sharded step, save rank files and a manifest through their contexts, are
resumed into fresh contexts (as after a restart) and continue bit-identically
to the uninterrupted sharded run; the files are the oracle's image of the
state; a different world size is refused before any device memory changes."""
import os

import numpy as np
import pytest

import synthetic
from oracle import sharded as osh
from synthetic import device as synth_dev

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402
from optimizer_step_resumable_gb300.sharded import ordered_sum, shard_range  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def sharded_steps(ctxs, spans, w, m, v, g, t0, t1):
    for t in range(t0, t1 + 1):
        synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
        sl = [slice(o, o + k) for o, k in spans]
        total = ordered_sum(osr.grad_sumsq(c, g[s]) for c, s in zip(ctxs, sl))
        for c, s in zip(ctxs, sl):
            osr.adamw_clip_step_ex(c, w[s], g[s], m[s], v[s], t, 3e-3, 0.01, 1.0,
                                   global_sumsq=total)


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_save_resume(dev, tmp_path, world):
    n = 2_000_003
    spans = [shard_range(n, r, world) for r in range(world)]
    g = torch.empty(n, device=dev)

    def fresh():
        w = torch.empty(n, device=dev)
        synth_dev.fill_weights(w, 7)
        return w, torch.zeros(n, device=dev), torch.zeros(n, device=dev)

    def contexts():
        return [osr.adamw_create(k) for _, k in spans]

    # uninterrupted: 30 steps
    w, m, v = fresh()
    ctxs = contexts()
    sharded_steps(ctxs, spans, w, m, v, g, 1, 30)
    ref = [x.clone() for x in (w, m, v)]
    for c in ctxs:
        c.close()
    # interrupted: 20 steps, sharded checkpoint, restart, 10 more
    w, m, v = fresh()
    ctxs = contexts()
    sharded_steps(ctxs, spans, w, m, v, g, 1, 20)
    digests = []
    for r, (c, (o, k)) in enumerate(zip(ctxs, spans)):
        osr.ckpt_pack(c, 20, w[o:o + k], m[o:o + k], v[o:o + k])
        digests.append(osr.ckpt_shard_write(c, str(tmp_path), r))
    d = osr.ckpt_manifest_commit(str(tmp_path), 20, [s[0] for s in spans],
                                 [s[1] for s in spans], digests)
    snap = [x.cpu().numpy() for x in (w, m, v)]
    for c in ctxs:
        c.close()
    # the files hold exactly the state at step 20 (the oracle re-verifies)
    step, got = osh.load_sharded(d, world)
    assert step == 20
    for (o, k, sw, sm, sv) in got:
        for a, b in zip((sw, sm, sv), snap):
            assert a.tobytes() == b[o:o + k].tobytes()
    with pytest.raises(osr.AdamWError) as e:  # world size changed
        c = osr.adamw_create(spans[0][1])
        try:
            osr.ckpt_shard_read(c, d, 0, w[:spans[0][1]], m[:spans[0][1]], v[:spans[0][1]],
                                expected_world=world + 1)
        finally:
            c.close()
    assert e.value.status == osr.EMISMATCH
    w, m, v = (torch.full((n,), float("nan"), device=dev) for _ in range(3))
    ctxs = contexts()
    for r, (c, (o, k)) in enumerate(zip(ctxs, spans)):
        assert osr.ckpt_shard_read(c, d, r, w[o:o + k], m[o:o + k], v[o:o + k],
                                   expected_world=world) == 20
    sharded_steps(ctxs, spans, w, m, v, g, 21, 30)
    for c in ctxs:
        c.close()
    for a, b in zip((w, m, v), ref):
        assert torch.equal(a, b)
