"""GPU per-tensor sums of squares (one pass with the global norm) against
the oracle, on the 110M tensor list and on tables built to stress the
segment bookkeeping; fault localisation; bit stability; and the step with
ADAMW_TENSOR_NORMS giving the same bits as without."""
import numpy as np
import pytest

import synthetic
from synthetic import device as synth_dev
from synthetic import workloads as W
from parity import RTOL_NORM

torch = pytest.importorskip("torch")
import optimizer_step_resumable_gb300 as osr  # noqa: E402

pytestmark = pytest.mark.gpu
TILE = 8192


@pytest.fixture(scope="module")
def dev(lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def table_from_sizes(sizes):
    off = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    return list(off), [int(k) for k in sizes]


def check_against_oracle(oracle, ctx, g, off, num):
    got = osr.grad_tensor_sumsq(ctx, g)
    want = oracle.tensor_sumsq(g.cpu().numpy(), off, num)
    assert got.shape == want.shape
    err = np.abs(got - want)
    assert np.all(err <= RTOL_NORM * want + 1e-300), (np.argmax(err / np.maximum(want, 1e-300)))
    return got


def test_gpt_110m_tensor_norms(dev, oracle):
    wl = W.gpt_110m()
    off, num = wl.table()
    g = torch.empty(wl.n, device=dev)
    synth_dev.fill_grads(g, 7, 1, 1e-3, 0.001, 1000.0)
    with osr.adamw_create(wl.n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        got = check_against_oracle(oracle, ctx, g, off, num)
        total = osr.grad_sumsq(ctx, g)
        # the two differ only on tiles where a tensor starts (exact squares
        # for the split there, float32 runs in the global sum): at most a
        # few float32 roundings of those tiles' share
        assert abs(got.sum() - total) <= 1e-9 * total
        again = osr.grad_tensor_sumsq(ctx, g)
        assert again.tobytes() == got.tobytes()  # bit-stable


SIZES = {
    "tiny_tensors": [1, 1, 2, 3, 5, 7, 100, 8181, 1, 8192, 8192, 1, 3, 40000],
    "on_tile_edges": [8192, 8192, 16384, 8192 * 3, 1, 8191, 8193],
    "one_tile_many": [768] * 40 + [5, 9],
    "ragged_tail": [123457, 3, 9999, 77777, 2],
    "huge_then_tiny": [8192 * 700 + 13] + [1] * 300 + [4096] * 9,
}


@pytest.mark.parametrize("name", sorted(SIZES))
def test_adversarial_tables(dev, oracle, name):
    sizes = SIZES[name]
    off, num = table_from_sizes(sizes)
    n = int(sum(sizes))
    g = torch.from_numpy(synthetic.grads(7, 3, 1e-2, n=n, outlier_frac=0.01,
                                         outlier_mult=100.0)).to(dev)
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        check_against_oracle(oracle, ctx, g, off, num)
        # unaligned copy of the same gradient: scalar kernel, same values
        buf = torch.empty(n + 1, device=dev)
        buf[1:].copy_(g)
        check_against_oracle(oracle, ctx, buf[1:], off, num)


def test_flat_table_is_the_global_sum(dev):
    n = 3 * TILE * 608 + 11  # several tiles per block
    g = torch.empty(n, device=dev)
    synth_dev.fill_grads(g, 7, 2, 1e-3)
    with osr.adamw_create(n, flags=osr.CREATE_NO_CKPT) as ctx:
        (one,) = osr.grad_tensor_sumsq(ctx, g)
        total = osr.grad_sumsq(ctx, g)
        assert abs(one - total) <= 1e-12 * total  # same runs, summed in another order


def test_nonfinite_is_localised(dev):
    sizes = [1000, 2000, 3000, 4000]
    off, num = table_from_sizes(sizes)
    g = torch.ones(10000, device=dev)
    g[off[2] + 17] = float("nan")
    with osr.adamw_create(10000, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        with pytest.raises(osr.NonFiniteGradient) as e:
            osr.grad_tensor_sumsq(ctx, g)
        vals = e.value.values
        assert np.isnan(vals[2]) and list(vals[[0, 1, 3]]) == [1000.0, 2000.0, 4000.0]


def test_step_with_tensor_norms_same_bits(dev, oracle):
    wl = W.gpt_110m()
    off, num = wl.table()
    n = wl.n
    out = []
    for flag in (False, True):
        w = torch.empty(n, device=dev)
        synth_dev.fill_weights(w, 7)
        m = torch.zeros(n, device=dev)
        v = torch.zeros(n, device=dev)
        g = torch.empty(n, device=dev)
        with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
            for t in (1, 2):
                synth_dev.fill_grads(g, 7, t, 1e-3)
                osr.adamw_clip_step_ex(ctx, w, g, m, v, t, wl.lr, wl.wd, wl.clip,
                                       tensor_norms=flag)
            if flag:
                last = osr.adamw_last_tensor_sumsq(ctx)
                assert last.tobytes() == osr.grad_tensor_sumsq(ctx, g).tobytes()
                osr.adamw_clip_step(ctx, w, g, m, v, 3, wl.lr, wl.wd, wl.clip)
                with pytest.raises(osr.AdamWError) as e:
                    osr.adamw_last_tensor_sumsq(ctx)
                assert e.value.status == osr.ESTATE
            else:
                osr.adamw_clip_step(ctx, w, g, m, v, 3, wl.lr, wl.wd, wl.clip)
        out.append(torch.cat([w, m, v]).cpu())
        del w, m, v, g
    assert torch.equal(out[0], out[1])
    torch.cuda.empty_cache()


def test_small_state_steps_do_not_leave_stale_tensor_sums(dev):
    """After a step with per-tensor sums, a one-launch step or a graph step
    (neither computes them) makes adamw_last_tensor_sumsq refuse instead of
    returning the older step's sums."""
    sizes = [300, 7, 4000, 1]
    num = np.array(sizes, np.int64)
    off = np.concatenate([[0], np.cumsum(num)[:-1]]).astype(np.int64)
    n = int(num.sum())
    w = torch.zeros(n, device=dev)
    m = torch.zeros(n, device=dev)
    v = torch.zeros(n, device=dev)
    g = torch.full((n,), 1e-3, device=dev)
    with osr.adamw_create(n, off, num, flags=osr.CREATE_NO_CKPT) as ctx:
        for follow in ("one_launch", "graph"):
            osr.adamw_clip_step_ex(ctx, w, g, m, v, 1, 1e-3, 0.0, 1.0, tensor_norms=True)
            assert osr.adamw_last_tensor_sumsq(ctx).shape == (len(sizes),)
            if follow == "one_launch":
                osr.adamw_clip_step(ctx, w, g, m, v, 2, 1e-3, 0.0, 1.0)
            else:
                osr.adamw_graph_create(ctx, w, g, m, v)
                osr.adamw_graph_step(ctx, 2, 1e-3, 0.0, 1.0)
                osr.adamw_graph_destroy(ctx)
            with pytest.raises(osr.AdamWError) as e:
                osr.adamw_last_tensor_sumsq(ctx)
            assert e.value.status == osr.ESTATE
