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
from optimizer_step_resumable_gb300.sharded import shard_range  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def sharded_steps(ctxs, spans, w, m, v, g, t0, t1):
    for t in range(t0, t1 + 1):
        synth_dev.fill_grads(g, 7, t, 1e-2, 0.01, 100.0)
        sl = [slice(o, o + k) for o, k in spans]
        parts = [osr.grad_sumsq(c, g[s]) for c, s in zip(ctxs, sl)]
        for c, s in zip(ctxs, sl):
            osr.adamw_clip_step_ranks(c, w[s], g[s], m[s], v[s], t, 3e-3, 0.01, 1.0, parts)


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


@pytest.mark.parametrize("world_a,world_b", [(4, 3), (2, 5), (3, 1)])
def test_resume_at_another_world_size(dev, tmp_path, world_a, world_b):
    """world_a ranks run 20 steps and save a sharded checkpoint; it is
    consolidated into one flat file, and world_b ranks each read their own
    range of it (ckpt_read_range): the state arrives bit for bit, and 10 more
    world_b steps give the same bits as world_b steps run on the state handed
    over in memory."""
    from optimizer_step_resumable_gb300 import sharded
    n = 2_000_003
    spans_a = [shard_range(n, r, world_a) for r in range(world_a)]
    spans_b = [shard_range(n, r, world_b) for r in range(world_b)]
    g = torch.empty(n, device=dev)
    w = torch.empty(n, device=dev)
    synth_dev.fill_weights(w, 7)
    m, v = torch.zeros(n, device=dev), torch.zeros(n, device=dev)
    ctxs = [osr.adamw_create(k) for _, k in spans_a]
    sharded_steps(ctxs, spans_a, w, m, v, g, 1, 20)
    digests = []
    for r, (c, (o, k)) in enumerate(zip(ctxs, spans_a)):
        osr.ckpt_pack(c, 20, w[o:o + k], m[o:o + k], v[o:o + k])
        digests.append(osr.ckpt_shard_write(c, str(tmp_path), r))
    for c in ctxs:
        c.close()
    d = osr.ckpt_manifest_commit(str(tmp_path), 20, [s[0] for s in spans_a],
                                 [s[1] for s in spans_a], digests)
    flat_dir = tmp_path / "flat"
    flat_dir.mkdir()
    flat = sharded.consolidate(d, str(flat_dir), expected_world=world_a)
    assert os.path.getsize(flat) == osr.ckpt_file_size(n)
    handed = [x.clone() for x in (w, m, v)]
    # the state in memory, continued by world_b ranks
    ctxs = [osr.adamw_create(k) for _, k in spans_b]
    sharded_steps(ctxs, spans_b, *handed, g, 21, 30)
    for c in ctxs:
        c.close()
    # the same from the file
    rw, rm, rv = (torch.full((n,), float("nan"), device=dev) for _ in range(3))
    ctxs = [osr.adamw_create(k) for _, k in spans_b]
    for r, (c, (o, k)) in enumerate(zip(ctxs, spans_b)):
        assert sharded.load_range(c, flat, r, world_b, rw[o:o + k], rm[o:o + k],
                                  rv[o:o + k]) == 20
    for a, b in zip((rw, rm, rv), (w, m, v)):
        assert torch.equal(a, b)
    sharded_steps(ctxs, spans_b, rw, rm, rv, g, 21, 30)
    for c in ctxs:
        c.close()
    for a, b in zip((rw, rm, rv), handed):
        assert torch.equal(a, b)


def test_read_range_bounds_and_full_range(dev, tmp_path):
    n = 1001
    hw, hm, hv = (np.random.default_rng(s).standard_normal(n).astype(np.float32)
                  for s in (1, 2, 3))
    path = osr.ckpt_write_host(str(tmp_path), 5, hw, hm, hv)
    full = osr.adamw_create(n)
    w, m, v = (torch.empty(n, device=dev) for _ in range(3))
    assert osr.ckpt_read_range(full, path, 0, w, m, v) == 5
    assert w.cpu().numpy().tobytes() == hw.tobytes()
    assert v.cpu().numpy().tobytes() == hv.tobytes()
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_read_range(full, path, 1, w, m, v)  # [1, 1002) is past the end
    assert e.value.status == osr.EMISMATCH
    full.close()
    part = osr.adamw_create(10)
    pw, pm, pv = (torch.full((10,), -7.0, device=dev) for _ in range(3))
    for off in (0, 3, 991):
        assert osr.ckpt_read_range(part, path, off, pw, pm, pv) == 5
        assert pw.cpu().numpy().tobytes() == hw[off:off + 10].tobytes()
        assert pm.cpu().numpy().tobytes() == hm[off:off + 10].tobytes()
        assert pv.cpu().numpy().tobytes() == hv[off:off + 10].tobytes()
    before = [x.clone() for x in (pw, pm, pv)]
    for off in (992, -1):
        with pytest.raises(osr.AdamWError):
            osr.ckpt_read_range(part, path, off, pw, pm, pv)
    for a, b in zip((pw, pm, pv), before):  # untouched on failure
        assert torch.equal(a, b)
    part.close()
    nock = osr.adamw_create(10, flags=osr.CREATE_NO_CKPT)  # no staging to read through
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_read_range(nock, path, 0, pw, pm, pv)
    assert e.value.status == osr.ESTATE
    nock.close()
