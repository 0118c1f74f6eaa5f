"""Sharded checkpoint, host side (no GPU): SHA-256 against the standard's
test vectors, the library's shard files and manifest read back by the oracle
and the oracle's read back by the library, the three refused failure modes,
the commit point, and gloo ranks writing one checkpoint together."""
import hashlib
import json
import os
import shutil
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import optimizer_step_resumable_gb300 as osr
from oracle import sharded as osh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("msg,digest", [
    (b"", "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855"),
    (b"abc", "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"),
    (b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq",
     "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1"),
    (b"a" * 1000000, "cdc76e5c9914fb9281a1c7e284d73e67f1809a48a497200e046d39ccc7112cd0"),
])
def test_sha256_standard_vectors(lib, msg, digest):
    assert osr.ckpt_sha256_hex(msg) == digest


def test_sha256_matches_hashlib(lib):
    rng = np.random.default_rng(0)
    for size in list(range(0, 200)) + [1023, 4096, 65537, 1 << 20]:
        data = rng.integers(0, 256, size, dtype=np.uint8).tobytes()
        assert osr.ckpt_sha256_hex(data) == hashlib.sha256(data).hexdigest(), size


def test_sha256_builtin_backend_matches_hashlib(lib):
    """The library's own SHA-256 (forced with OSR_SHA256=builtin, in a fresh
    process) against the standard's vectors and hashlib on odd lengths --
    the code that runs where libcrypto cannot be loaded."""
    import subprocess
    import sys
    code = (
        "import hashlib, sys, numpy as np\n"
        "sys.path.insert(0, %r)\n"
        "import optimizer_step_resumable_gb300 as osr\n"
        "assert osr.ckpt_sha256_backend() == 'builtin'\n"
        "assert osr.ckpt_sha256_hex(b'abc') == "
        "'ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad'\n"
        "rng = np.random.default_rng(1)\n"
        "for size in list(range(0, 130)) + [1023, 65537, 1 << 20]:\n"
        "    d = rng.integers(0, 256, size, dtype=np.uint8).tobytes()\n"
        "    assert osr.ckpt_sha256_hex(d) == hashlib.sha256(d).hexdigest(), size\n"
        "print('ok')\n") % ROOT
    env = dict(os.environ, OSR_SHA256="builtin")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr[-2000:]


def test_sha256_backend_is_reported(lib):
    assert osr.ckpt_sha256_backend() in ("libcrypto", "builtin")


def _shards(sizes, seed=3):
    rng = np.random.default_rng(seed)
    return [tuple(rng.standard_normal(k).astype(np.float32) for _ in range(3)) for k in sizes]


def _offsets(sizes):
    return [int(x) for x in np.concatenate([[0], np.cumsum(sizes)[:-1]])]


def test_library_writes_oracle_reads(lib, oracle, tmp_path):
    sizes = [1000, 1000, 1000, 997]
    shards = _shards(sizes)
    digests = [osr.ckpt_shard_write_host(str(tmp_path), 42, r, *s) for r, s in enumerate(shards)]
    assert not os.path.exists(tmp_path / "step_000042")  # invisible before the commit
    d = osr.ckpt_manifest_commit(str(tmp_path), 42, _offsets(sizes), sizes, digests, 4521.0)
    assert d == str(tmp_path / "step_000042") and not os.path.exists(d + ".tmp")
    step, got = osh.load_sharded(d, 4)
    assert step == 42
    for (off, k, w, m, v), s, o in zip(got, shards, _offsets(sizes)):
        assert off == o and k == s[0].size
        assert w.tobytes() == s[0].tobytes() and v.tobytes() == s[2].tobytes()
    man = json.load(open(os.path.join(d, "manifest.json")))
    page = json.load(open(os.path.join(ROOT, "tests", "golden", "manifest_example.json")))
    assert list(man) == list(page) and list(man["shards"][0]) == list(page["shards"][0])
    assert man["wall_clock_seconds"] == 4521.0
    assert osr.ckpt_manifest_load(d, 4) == (42, _offsets(sizes), sizes)


def test_oracle_writes_library_reads(lib, oracle, tmp_path):
    sizes = [4096, 4096]
    d = osh.save_sharded(str(tmp_path), 100, _shards(sizes), _offsets(sizes), 12.5)
    assert osr.ckpt_manifest_load(d, 2) == (100, [0, 4096], sizes)


def _copy(d, tmp_path, name):
    bad = str(tmp_path / name)
    shutil.copytree(d, bad)
    return bad


def test_library_refuses_the_three_failure_modes(lib, tmp_path):
    sizes = [500, 500, 500, 500]
    d = osh.save_sharded(str(tmp_path), 9, _shards(sizes), _offsets(sizes))
    with pytest.raises(osr.AdamWError) as e:  # world size changed
        osr.ckpt_manifest_load(d, 2)
    assert e.value.status == osr.EMISMATCH
    bad = _copy(d, tmp_path, "count")
    man = json.load(open(os.path.join(bad, "manifest.json")))
    man["shards"] = man["shards"][:3]
    json.dump(man, open(os.path.join(bad, "manifest.json"), "w"))
    with pytest.raises(osr.AdamWError) as e:  # shard count mismatch
        osr.ckpt_manifest_load(bad, 4)
    assert e.value.status == osr.EMISMATCH
    bad = _copy(d, tmp_path, "trunc")
    p = os.path.join(bad, "rank3.bin")
    open(p, "wb").write(open(p, "rb").read()[:-4])
    with pytest.raises(osr.AdamWError) as e:  # partial write: size
        osr.ckpt_manifest_load(bad, 4)
    assert e.value.status == osr.ESIZE
    bad = _copy(d, tmp_path, "flip")
    p = os.path.join(bad, "rank0.bin")
    data = bytearray(open(p, "rb").read())
    data[-1] ^= 0x40
    open(p, "wb").write(bytes(data))
    with pytest.raises(osr.AdamWError) as e:  # partial write: digest
        osr.ckpt_manifest_load(bad, 4)
    assert e.value.status == osr.EFORMAT
    osr.ckpt_manifest_load(bad, 4, verify=False)  # sizes and headers alone pass
    for mutate in (lambda m: m.update(schema_version=2),
                   lambda m: m["shards"][1].update(path="../rank1.bin"),
                   lambda m: m["shards"][1].update(param_shard_offset=499),
                   lambda m: m["shards"][2].update(rank=1),
                   lambda m: m["shards"][0].update(sha256="xyz")):
        bad = _copy(d, tmp_path, f"m{len(os.listdir(tmp_path))}")
        man = json.load(open(os.path.join(bad, "manifest.json")))
        mutate(man)
        json.dump(man, open(os.path.join(bad, "manifest.json"), "w"))
        with pytest.raises(osr.AdamWError):
            osr.ckpt_manifest_load(bad, 4)
    bad = _copy(d, tmp_path, "json")
    open(os.path.join(bad, "manifest.json"), "w").write('{"world_size": 4,')
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_manifest_load(bad, 4)
    assert e.value.status == osr.EFORMAT


def test_commit_point(lib, tmp_path):
    """Before the commit the step does not exist and the previous one is
    intact; a commit with a missing shard is refused; a stale staging
    directory (more ranks, from a crashed attempt) is cleaned by the commit."""
    sizes = [300, 300]
    old = osh.save_sharded(str(tmp_path), 1, _shards(sizes, 1), _offsets(sizes))
    sh = _shards([200, 200, 200], 2)
    for r in range(3):  # a crashed attempt with 3 ranks
        osr.ckpt_shard_write_host(str(tmp_path), 2, r, *sh[r])
    new = _shards(sizes, 5)
    d0 = osr.ckpt_shard_write_host(str(tmp_path), 2, 0, *new[0])
    with pytest.raises(osr.AdamWError) as e:  # rank 1 still holds the stale 200
        osr.ckpt_manifest_commit(str(tmp_path), 2, _offsets(sizes), sizes, [d0, d0])
    assert e.value.status == osr.ESTATE
    assert not os.path.exists(tmp_path / "step_000002")
    assert osr.ckpt_manifest_load(old, 2)[0] == 1
    d1 = osr.ckpt_shard_write_host(str(tmp_path), 2, 1, *new[1])
    d = osr.ckpt_manifest_commit(str(tmp_path), 2, _offsets(sizes), sizes, [d0, d1])
    assert sorted(os.listdir(d)) == ["manifest.json", "rank0.bin", "rank1.bin"]
    assert osr.ckpt_manifest_load(d, 2)[0] == 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, d):
    import torch.distributed as dist

    import optimizer_step_resumable_gb300 as osr2
    from optimizer_step_resumable_gb300.sharded import _gather_objects, shard_range
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    n = 10_001
    spans = [shard_range(n, r, world) for r in range(world)]
    off, k = spans[rank]
    rng = np.random.default_rng(100 + rank)
    w, m, v = (rng.standard_normal(k).astype(np.float32) for _ in range(3))
    digest = osr2.ckpt_shard_write_host(d, 77, rank, w, m, v)
    digests = _gather_objects(digest)
    if rank == 0:
        osr2.ckpt_manifest_commit(d, 77, [s[0] for s in spans], [s[1] for s in spans], digests)
    dist.barrier()
    step, offs, nums = osr2.ckpt_manifest_load(os.path.join(d, "step_000077"), world)
    assert step == 77 and offs[rank] == off and nums[rank] == k
    np.save(os.path.join(d, f"in{rank}.npy"), np.stack([w, m, v]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_gloo_ranks_write_one_checkpoint(lib, tmp_path, world):
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    step, got = osh.load_sharded(str(tmp_path / "step_000077"), world)
    assert step == 77
    for r, (_, _, w, m, v) in enumerate(got):
        ref = np.load(tmp_path / f"in{r}.npy")
        assert w.tobytes() == ref[0].tobytes() and v.tobytes() == ref[2].tobytes()


# ---------------------------------------------------------------------------
# Consolidation: the shards' ranges put back at their offsets of the flat
# vector, as one step_NNNNNN.bin.
# ---------------------------------------------------------------------------
def _flat(n, seed=11):
    rng = np.random.default_rng(seed)
    return [rng.standard_normal(n).astype(np.float32) for _ in range(3)]


def _split(flat, world):
    from optimizer_step_resumable_gb300 import sharded
    n = flat[0].size
    ranges = [sharded.shard_range(n, r, world) for r in range(world)]
    return ranges, [tuple(a[o:o + k] for a in flat) for o, k in ranges]


def _flat_bytes(step, flat):
    import struct
    return struct.pack("<ii", step, flat[0].size) + b"".join(a.tobytes() for a in flat)


@pytest.mark.parametrize("n,world", [(3997, 4), (4096, 1), (10, 3), (7, 7), (65_537, 5)])
def test_consolidate_puts_shards_at_their_offsets(lib, oracle, tmp_path, n, world):
    flat = _flat(n)
    ranges, shards = _split(flat, world)
    digests = [osr.ckpt_shard_write_host(str(tmp_path), 300, r, *s) for r, s in enumerate(shards)]
    d = osr.ckpt_manifest_commit(str(tmp_path), 300, [o for o, _ in ranges],
                                 [k for _, k in ranges], digests, 1.0)
    out = tmp_path / "flat"
    out.mkdir()
    path = osr.ckpt_consolidate(d, str(out), expected_world=world)
    assert path == str(out / "step_000300.bin")
    assert sorted(os.listdir(out)) == ["step_000300.bin"]  # no .tmp left
    assert open(path, "rb").read() == _flat_bytes(300, flat)
    st, step, ow, om, ov = oracle.ckpt_read(path, n)  # the oracle's reader agrees
    assert st == 0 and step == 300
    assert ow.tobytes() == flat[0].tobytes() and ov.tobytes() == flat[2].tobytes()
    assert osr.ckpt_probe(path) == (300, n)


def test_consolidate_of_oracle_written_shards(lib, tmp_path):
    sizes = [1000, 24, 3]
    shards = _shards(sizes, 5)
    d = osh.save_sharded(str(tmp_path), 7, shards, _offsets(sizes), 2.0)
    path = osr.ckpt_consolidate(d, str(tmp_path))
    flat = [np.concatenate([s[i] for s in shards]) for i in range(3)]
    assert open(path, "rb").read() == _flat_bytes(7, flat)


def test_consolidate_refuses_and_leaves_no_file(lib, tmp_path):
    flat = _flat(2000)
    ranges, shards = _split(flat, 4)
    src = tmp_path / "src"
    src.mkdir()
    digests = [osr.ckpt_shard_write_host(str(src), 12, r, *s) for r, s in enumerate(shards)]
    d = osr.ckpt_manifest_commit(str(src), 12, [o for o, _ in ranges], [k for _, k in ranges],
                                 digests, 0.0)
    out = tmp_path / "out"
    out.mkdir()
    with pytest.raises(osr.AdamWError) as e:  # a different world size
        osr.ckpt_consolidate(d, str(out), expected_world=3)
    assert e.value.status == osr.EMISMATCH
    # one flipped bit in the last shard's v region: found by the digest only
    # after every other byte was streamed; the output never appears
    p = os.path.join(d, "rank3.bin")
    data = bytearray(open(p, "rb").read())
    data[-5] ^= 0x01
    open(p, "wb").write(bytes(data))
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_consolidate(d, str(out), expected_world=4)
    assert e.value.status == osr.EFORMAT
    assert os.listdir(out) == []
    open(p, "wb").write(bytes(data[:-4]))  # truncated: refused before writing
    with pytest.raises(osr.AdamWError) as e:
        osr.ckpt_consolidate(d, str(out))
    assert e.value.status == osr.ESIZE
    assert os.listdir(out) == []
