"""Host logic of the sharded step on CPU ranks (gloo, world sizes 2 and 4):
the partition covers [0, n) exactly, the library's rank-order sum of the
gathered values (adamw_rank_total, host only) gives every rank the same
global sum, and the oracle applied shard by shard with that sum reproduces
the unsharded oracle step."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import optimizer_step_resumable_gb300 as osr
from optimizer_step_resumable_gb300.sharded import shard_range


def test_shard_ranges_cover_exactly():
    for n in (4, 7, 65536, 65537, 110_418_432, 1000003):
        for world in (1, 2, 3, 4, 8):
            if n < world:
                continue
            spans = [shard_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and sum(k for _, k in spans) == n
            assert all(a + k == b for (a, k), (b, _) in zip(spans, spans[1:]))
            assert all(k > 0 for _, k in spans)
            if n // world >= 4:
                assert all(off % 4 == 0 for off, _ in spans)
    with pytest.raises(ValueError):
        shard_range(3, 0, 4)


def test_rank_total_adds_in_rank_order(lib):
    # 1 + 2^-53 rounds to 1 (ties to even), so the order of the additions
    # shows in the last bit: rank order keeps 1, the reverse order gives
    # 1 + 2^-52
    tiny = 2.0 ** -53
    assert osr.adamw_rank_total([1.0, tiny, tiny], 1.0)[0] == 1.0
    assert osr.adamw_rank_total([tiny, tiny, 1.0], 1.0)[0] == 1.0 + 2.0 ** -52


def test_rank_total_norm_and_factor(lib):
    # 3-4-5: the ranks hold 9 and 16, the norm is 5 and the factor c / 5
    s, norm, scale = osr.adamw_rank_total([9.0, 16.0], 1.0)
    assert (s, norm) == (25.0, 5.0)
    assert scale == float(np.float32(0.2))
    # the gradient scale multiplies the norm and the factor applied to g
    s, norm, scale = osr.adamw_rank_total([9.0, 16.0], 1.0, grad_scale=0.5)
    assert norm == 2.5 and scale == float(np.float32(0.5 * (1.0 / 2.5)))
    # at or below the threshold the factor is exactly 1 (strict >)
    assert osr.adamw_rank_total([9.0, 16.0], 5.0)[2] == 1.0
    assert osr.adamw_rank_total([0.0, 0.0], 1.0)[1:] == (0.0, 1.0)
    assert osr.adamw_rank_total([9.0, 16.0], float("inf"))[2] == 1.0


def test_rank_total_refusals(lib):
    for bad in ([float("inf"), 1.0], [1.0, float("nan")]):
        with pytest.raises(osr.NonFiniteGradient) as e:
            osr.adamw_rank_total(bad, 1.0)
        assert not np.isfinite(e.value.values[1])
    for parts, clip, gs in (([1.0, -1.0], 1.0, 1.0), ([1.0], 0.0, 1.0), ([1.0], 1.0, 0.0),
                            ([1.0], 1.0, float("inf"))):
        with pytest.raises(osr.AdamWError) as e:
            osr.adamw_rank_total(parts, clip, grad_scale=gs)
        assert e.value.status == osr.EINVAL
    with pytest.raises(ValueError):
        osr.adamw_rank_total([], 1.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, n, out_dir):
    import torch.distributed as dist

    import oracle
    import synthetic
    import optimizer_step_resumable_gb300 as osr
    from optimizer_step_resumable_gb300.sharded import gather_sumsq, shard_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    o = oracle.load()
    off, k = shard_range(n, rank, world)
    idx = np.arange(off, off + k)
    w = synthetic.weights(7, idx=idx)
    m = np.zeros(k, np.float32)
    v = np.zeros(k, np.float32)
    for t in (1, 2, 3):
        g = synthetic.grads(7, t, 1e-2, idx=idx, outlier_frac=0.01, outlier_mult=100.0)
        parts = gather_sumsq(o.sumsq(g))
        assert len(parts) == world
        total = osr.adamw_rank_total(parts, 1.0)[0]  # the library's rank-order sum
        s = o.clip_scale(np.sqrt(total), 1.0)
        w, m, v = o.adamw_at(np.arange(k), w, g, m, v, s, t, 3e-3, 0.01)
        np.save(os.path.join(out_dir, f"r{rank}_t{t}_total.npy"), np.array([total]))
    np.save(os.path.join(out_dir, f"r{rank}.npy"), np.stack([w, m, v]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_sharded_oracle_matches_unsharded(oracle, lib, tmp_path, world):
    n = 65536 + 37
    mp.start_processes(_rank_main, args=(world, _free_port(), n, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    import synthetic
    w = synthetic.weights(7, n=n)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    for t in (1, 2, 3):
        g = synthetic.grads(7, t, 1e-2, n=n, outlier_frac=0.01, outlier_mult=100.0)
        _, norm = oracle.adamw_clip_step(w, g, m, v, t, 3e-3, 0.01, 1.0)
        totals = {float(np.load(tmp_path / f"r{r}_t{t}_total.npy")[0]) for r in range(world)}
        assert len(totals) == 1  # every rank got the same global sum
        assert abs(np.sqrt(totals.pop()) - norm) <= 1e-12 * norm
    got = np.concatenate([np.load(tmp_path / f"r{r}.npy") for r in range(world)], axis=1)
    for a, b in zip(got, (w, m, v)):
        # the same definition summed in another order: equal up to the last bit
        assert np.all(np.abs(a.astype(np.float64) - b) <= np.abs(b) * 2.0 ** -22 + 1e-30)
