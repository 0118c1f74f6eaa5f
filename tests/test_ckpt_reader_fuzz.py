"""The step_NNNNNN.bin reader on hostile files (no GPU): random headers,
sizes and truncations.  ckpt_probe accepts a file only when its header is a
non-negative step and n and its size is exactly 8 + 12 n (and n matches the
expected one when given); everything else raises AdamWError.  The rule is
checked against the file's own bytes, never by crashing."""
import struct

import numpy as np
import pytest

import optimizer_step_resumable_gb300 as osr


def consistent(data, n_expected):
    if len(data) < 8:
        return False
    step, n = struct.unpack("<ii", data[:8])
    if step < 0 or n < 0 or len(data) != 8 + 12 * n:
        return False
    return n_expected < 0 or n == n_expected


def test_random_files(lib, tmp_path):
    rng = np.random.default_rng(77)
    path = tmp_path / "step_000001.bin"
    accepted = 0
    for i in range(600):
        kind = i % 4
        n = int(rng.integers(0, 64))
        step = int(rng.integers(-3, 1 << 20))
        if kind == 0:      # consistent header, then a random size change
            body = rng.integers(0, 256, 12 * n, dtype=np.uint8).tobytes()
            data = struct.pack("<ii", step, n) + body
            cut = int(rng.integers(-3, 4))
            data = data[:len(data) + cut] if cut < 0 else data + b"\0" * cut
        elif kind == 1:    # random header over a plausible body
            data = rng.integers(0, 256, 8 + 12 * n, dtype=np.uint8).tobytes()
        elif kind == 2:    # extreme header values
            hn = int(rng.choice([0, 1, n, -1, 2 ** 31 - 1, -2 ** 31]))
            data = struct.pack("<ii", step, hn) + b"\0" * (12 * max(n, 0))
        else:              # short files
            data = rng.integers(0, 256, int(rng.integers(0, 9)), dtype=np.uint8).tobytes()
        path.write_bytes(data)
        n_expected = -1 if rng.integers(0, 2) else n
        ok = consistent(data, n_expected)
        try:
            got = osr.ckpt_probe(str(path), n_expected)
        except osr.AdamWError:
            assert not ok, (kind, data[:16])
            continue
        assert ok, (kind, data[:16])
        assert got == struct.unpack("<ii", data[:8])
        accepted += 1
    assert accepted > 20  # the accepting branch is exercised too
