"""Pins of the oracle's counter-based uniform generator.

The oracle restates Philox4x64-10 from Salmon et al., "Parallel random
numbers: as easy as 1, 2, 3" (SC 2011).  numpy ships an independent
implementation of the same generator (numpy.random.Philox, whose default is
the 4x64, 10-round variant); it advances its 256-bit counter by one before
each block, so its first block after ``counter=C`` is the block at C + 1.
"""
import numpy as np
import pytest

import oracle

MASK64 = (1 << 64) - 1


def _words(c: int):
    return [(c >> (64 * j)) & MASK64 for j in range(4)]


def _numpy_blocks(key, counter_int: int, nblocks: int) -> np.ndarray:
    """Blocks counter_int, counter_int + 1, ... from numpy's own Philox."""
    start = (counter_int - 1) % (1 << 256)
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array(_words(start), dtype=np.uint64))
    return bg.random_raw(4 * nblocks).astype(np.uint64).reshape(nblocks, 4)


@pytest.mark.parametrize("seed", [0, 1, 0x5EED, 2**64 - 1])
def test_block_function_matches_numpy(seed):
    rng = np.random.default_rng(seed & 0xFFFF)
    keys = [(0, 0), (seed & MASK64, 0), (int(rng.integers(0, 2**63)), int(rng.integers(0, 2**63)))]
    counters = [0, 1, MASK64, (1 << 64), (1 << 128) - 1,
                int.from_bytes(rng.bytes(32), "little")]
    for key in keys:
        for c in counters:
            want = _numpy_blocks(key, c, 1)[0]
            got = oracle.philox4x64(np.array(_words(c), dtype=np.uint64),
                                    np.array(key, dtype=np.uint64))
            np.testing.assert_array_equal(got, want, err_msg=f"key={key} counter={c:#x}")


@pytest.mark.parametrize("n,base", [(1, 0), (7, 3), (480, 1000), (1027, 2**40 + 5)])
def test_uniform_mapping(n, base):
    seed = 0xABCDEF
    got = oracle.philox_uniforms(seed, base, n)
    words = _numpy_blocks((seed, 0), base, (n + 3) // 4).reshape(-1)[:n]
    want = ((words >> np.uint64(40)).astype(np.float64) * 2.0 ** -24).astype(np.float32)
    np.testing.assert_array_equal(got, want)


def test_range_and_streams():
    u = oracle.philox_uniforms(11, 0, 40000)
    assert u.min() >= 0.0 and u.max() < 1.0
    scaled = u.astype(np.float64) * 2.0 ** 24
    assert np.all(scaled == np.floor(scaled))            # multiples of 2^-24
    assert abs(u.mean() - 0.5) < 0.01                    # 40k draws: sd of the mean ~0.0014
    # a different seed or a shifted counter gives a different stream; a shift by
    # one block is the same stream moved by four uniforms
    assert not np.array_equal(u[:100], oracle.philox_uniforms(12, 0, 100))
    np.testing.assert_array_equal(oracle.philox_uniforms(11, 1, 96), u[4:100])
