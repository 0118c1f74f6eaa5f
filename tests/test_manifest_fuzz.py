"""The library's manifest reader on hostile input (no GPU).  manifest.json is
read from disk, so its hand-written JSON parser and validation must refuse
any malformed or inconsistent file with an error status -- never crash, read
out of bounds or accept it.  Seeded mutations of a valid manifest (byte
flips, cuts, insertions, token swaps, deep nesting, huge or fractional
numbers, escapes, duplicate and missing keys) and random bytes; each load
either succeeds with exactly the committed table (only possible if the
mutation kept the meaning, e.g. whitespace) or raises AdamWError."""
import json
import os
import shutil

import numpy as np
import pytest

import optimizer_step_resumable_gb300 as osr

SIZES = [1000, 1000, 997]


@pytest.fixture(scope="module")
def committed(lib, tmp_path_factory):
    root = tmp_path_factory.mktemp("fuzz")
    rng = np.random.default_rng(9)
    digests = []
    for r, k in enumerate(SIZES):
        w, m, v = (rng.standard_normal(k).astype(np.float32) for _ in range(3))
        digests.append(osr.ckpt_shard_write_host(str(root), 7, r, w, m, v))
    offs = [0, 1000, 2000]
    d = osr.ckpt_manifest_commit(str(root), 7, offs, SIZES, digests, 12.5)
    text = open(os.path.join(d, "manifest.json"), "rb").read()
    return d, text, (7, offs, SIZES)


TOKENS = [b"{", b"}", b"[", b"]", b",", b":", b'"', b"\\", b"\\u0041", b"\\u00e9", b"\\q",
          b"null", b"true", b"false", b"-", b"1e309", b"-1", b"0.5", b"99999999999999999999999",
          b"2147483648", b"-2147483649", b" ", b"\n", b"\x00", b"\xff", b'"rank"',
          b'"world_size"', b'"shards"', b"[" * 40, b"]" * 40, b'{"a":' * 20]


def mutate(rng, text):
    b = bytearray(text)
    kind = int(rng.integers(0, 7))
    if kind == 0 and b:                              # flip bytes
        for _ in range(int(rng.integers(1, 4))):
            b[int(rng.integers(0, len(b)))] = int(rng.integers(0, 256))
    elif kind == 1:                                  # cut
        b = b[:int(rng.integers(0, len(b) + 1))]
    elif kind == 2:                                  # insert a token
        i = int(rng.integers(0, len(b) + 1))
        b[i:i] = TOKENS[int(rng.integers(0, len(TOKENS)))]
    elif kind == 3 and b:                            # delete a span
        i = int(rng.integers(0, len(b)))
        del b[i:i + int(rng.integers(1, 16))]
    elif kind == 4:                                  # replace a value in the parsed object
        man = json.loads(text)
        shard = man["shards"][int(rng.integers(0, len(man["shards"])))]
        key = ["rank", "param_shard_offset", "param_shard_numel", "path", "sha256"][
            int(rng.integers(0, 5))]
        val = [None, True, -1, 0, 1, 2, 3, 2 ** 31, 2 ** 63, 1.5, "x", "../x", "/etc/passwd",
               "rank0.bin", "0" * 64, "g" * 64, [], {}][int(rng.integers(0, 18))]
        if rng.integers(0, 4) == 0:
            shard.pop(key)
        else:
            shard[key] = val
        b = bytearray(json.dumps(man).encode())
    elif kind == 5:                                  # top-level fields
        man = json.loads(text)
        key = ["schema_version", "world_size", "step", "wall_clock_seconds", "shards"][
            int(rng.integers(0, 5))]
        val = [None, 0, 1, 2, 3, 4, -1, 2 ** 31, 1e300, "1", [], {}, [1, 2, 3]][
            int(rng.integers(0, 13))]
        if rng.integers(0, 4) == 0:
            man.pop(key)
        else:
            man[key] = val
        b = bytearray(json.dumps(man).encode())
    else:                                            # random bytes
        b = bytearray(rng.integers(0, 256, int(rng.integers(0, 300)), dtype=np.uint8).tobytes())
    return bytes(b)


def test_mutated_manifests_are_refused_or_unchanged(committed, tmp_path):
    d, text, want = committed
    rng = np.random.default_rng(2024)
    work = tmp_path / "step_000007"
    shutil.copytree(d, work)
    accepted = refused = 0
    for _ in range(1500):
        data = mutate(rng, text)
        with open(work / "manifest.json", "wb") as f:
            f.write(data)
        try:
            got = osr.ckpt_manifest_load(str(work), 3, verify=False)
        except osr.AdamWError:
            refused += 1
            continue
        accepted += 1
        assert got == want, data  # accepted only if the table is the committed one
    assert refused > 1000, (accepted, refused)


def test_deep_nesting_and_long_strings_are_refused(committed, tmp_path):
    d, _, _ = committed
    work = tmp_path / "step_000007"
    shutil.copytree(d, work)
    for data in (b"[" * 100000, b'{"a":' * 50000 + b"1" + b"}" * 50000,
                 b'"' + b"a" * (1 << 22), b"{" + b" " * (1 << 22), b"",
                 b'{"schema_version": 1' + b", \"x\": 0" * 100000 + b"}"):
        with open(work / "manifest.json", "wb") as f:
            f.write(data)
        with pytest.raises(osr.AdamWError):
            osr.ckpt_manifest_load(str(work), 3, verify=False)
