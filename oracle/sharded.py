"""Oracle of the sharded checkpoint: per-rank shard files and a manifest.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Plain Python,
restating "Checkpoint and Sharded Resume" (AI Engineering from Scratch,
phase 19 lesson 80): each rank's state goes to its own file, a manifest
records world_size, step, wall_clock_seconds, per shard {rank, path,
sha256, param_shard_offset, param_shard_numel} and schema_version 1 (section
"Manifest schema"); files are written to temporary names, fsynced, then
renamed (section "Atomic write"); the loader verifies every shard's sha256
and refuses a different world size, a shard count that does not match it,
and partial writes (section "Three failure modes").  Each shard file holds
the rank's range in the step_NNNNNN.bin layout (the oracle's own pack).
The whole step directory is staged as step_NNNNNN.tmp and renamed last.
"""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np

from . import load

SCHEMA_VERSION = 1


class ShardedCheckpointError(RuntimeError):
    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind  # "world_size", "shard_count", "partial_write", "format"


def _fsync_dir(path):
    fd = os.open(path, os.O_RDONLY)
    try:
        os.fsync(fd)
    finally:
        os.close(fd)


def _write(path, data: bytes):
    with open(path + ".tmp", "wb") as f:
        f.write(data)
        f.flush()
        os.fsync(f.fileno())
    os.replace(path + ".tmp", path)


def manifest(world, step, wall, offsets, numels, digests):
    return {"world_size": world, "step": step, "wall_clock_seconds": wall,
            "shards": [{"rank": r, "path": f"rank{r}.bin", "sha256": digests[r],
                        "param_shard_offset": offsets[r], "param_shard_numel": numels[r]}
                       for r in range(world)],
            "schema_version": SCHEMA_VERSION}


def save_sharded(directory, step, shards, offsets, wall_clock_seconds=0.0):
    """shards: per rank (w, m, v) float32 arrays.  Returns the step dir."""
    o = load()
    world = len(shards)
    final = os.path.join(directory, f"step_{step:06d}")
    staging = final + ".tmp"
    os.makedirs(staging, exist_ok=True)
    digests, numels = [], []
    for r, (w, m, v) in enumerate(shards):
        data = o.pack(step, w, m, v).tobytes()
        _write(os.path.join(staging, f"rank{r}.bin"), data)
        digests.append(hashlib.sha256(data).hexdigest())
        numels.append(int(w.size))
    man = manifest(world, step, float(wall_clock_seconds), list(offsets), numels, digests)
    _write(os.path.join(staging, "manifest.json"), json.dumps(man, indent=2).encode())
    _fsync_dir(staging)
    os.rename(staging, final)
    _fsync_dir(directory)
    return final


def load_sharded(step_dir, expected_world):
    """Returns (step, [(offset, numel, w, m, v) per rank]) after checking
    the manifest and every shard; raises ShardedCheckpointError."""
    with open(os.path.join(step_dir, "manifest.json")) as f:
        man = json.load(f)
    if man.get("schema_version") != SCHEMA_VERSION:
        raise ShardedCheckpointError("format", "schema_version")
    world = man["world_size"]
    if world != expected_world:
        raise ShardedCheckpointError("world_size", f"saved {world}, loading {expected_world}")
    shards = man["shards"]
    if len(shards) != world or sorted(s["rank"] for s in shards) != list(range(world)):
        raise ShardedCheckpointError("shard_count", f"{len(shards)} shards for world {world}")
    o = load()
    out, expect = [], 0
    for s in sorted(shards, key=lambda s: s["rank"]):
        if s["param_shard_offset"] != expect:
            raise ShardedCheckpointError("format", "ranges not contiguous")
        expect += s["param_shard_numel"]
        path = os.path.join(step_dir, s["path"])
        data = open(path, "rb").read()
        if hashlib.sha256(data).hexdigest() != s["sha256"]:
            raise ShardedCheckpointError("partial_write", f"sha256 of {s['path']}")
        st, step, w, m, v = o.ckpt_read(path, s["param_shard_numel"])
        if st != 0 or step != man["step"]:
            raise ShardedCheckpointError("partial_write", f"{s['path']} status {st}")
        out.append((s["param_shard_offset"], s["param_shard_numel"], w, m, v))
    return man["step"], out
