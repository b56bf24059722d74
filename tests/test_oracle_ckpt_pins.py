"""Pins of the oracle's checkpoint flush and load (no GPU): they are element
copies through the address function (ROCm/ATOM pull request 2945, Changes:
under ReplaySSM the checkpoint load and the flush go through state_at), so they
must equal NumPy's fancy-index assignment, round-trip exactly, and skip
negative indices."""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.usefixtures("oracle_mod")


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
def test_flush_and_load_are_fancy_index_copies(dtype):
    rng = np.random.default_rng(3)
    pool = rng.integers(0, 60000, size=(10, 3, 16, 32)).astype(dtype)
    plane = rng.integers(0, 60000, size=(6, 3, 16, 32)).astype(dtype)
    slots, entries = np.array([4, 0, 9], np.int32), np.array([5, 2, 0], np.int32)
    ref_plane = plane.copy()
    ref_plane[entries] = pool[slots]
    oracle.ckpt_transfer(pool, plane, slots, entries, load=False)
    assert np.array_equal(plane, ref_plane)
    pool2 = rng.integers(0, 60000, size=pool.shape).astype(dtype)
    ref_pool = pool2.copy()
    ref_pool[slots] = plane[entries]
    oracle.ckpt_transfer(pool2, plane, slots, entries, load=True)
    assert np.array_equal(pool2, ref_pool)
    # round trip: what was flushed comes back bit for bit
    assert np.array_equal(pool2[slots], pool[slots])


def test_negative_indices_skip_and_range_is_checked():
    pool = np.arange(4 * 2 * 16 * 16, dtype=np.float32).reshape(4, 2, 16, 16)
    plane = np.zeros((3, 2, 16, 16), np.float32)
    oracle.ckpt_transfer(pool, plane, np.array([1, -1, 2], np.int32), np.array([0, 1, -1], np.int32), load=False)
    assert np.array_equal(plane[0], pool[1]) and not plane[1:].any()
    with pytest.raises(ValueError):
        oracle.ckpt_transfer(pool, plane, np.array([4], np.int32), np.array([0], np.int32), load=False)
    with pytest.raises(ValueError):
        oracle.ckpt_transfer(pool, plane, np.array([0], np.int32), np.array([3], np.int32), load=True)
