"""Pins for the per-step top-k block signal oracle (CPU only)."""
import numpy as np

from oracle import block_signal as bs
from oracle.attention import decode_attention


def test_masses_of_a_step_add_up_to_the_q_heads():
    # every head's softmax row sums to 1, whatever the partial last block
    rng = np.random.default_rng(1)
    q = rng.standard_normal((8, 16))
    K, V = rng.standard_normal((2, 70, 16)), rng.standard_normal((2, 70, 16))
    _, p = decode_attention(q, K, V, 0.25)
    m = bs.block_masses(p)
    assert m.shape == (5,)
    assert abs(m.sum() - 8) < 1e-12


def test_masses_by_hand():
    # 2 heads, 5 keys, block size 2: blocks {0,1}, {2,3}, {4}
    p = np.array([[0.125, 0.25, 0.375, 0.125, 0.0],
                  [0.5, 0.0, 0.0, 0.25, 0.25]])
    assert bs.block_masses(p, page=2).tolist() == [0.875, 0.75, 0.25]


def test_top_blocks_ties_and_short_rows():
    m = np.array([0.5, 0.9, 0.5, 0.9, 0.1])
    assert bs.top_blocks(m, 2).tolist() == [1, 3]
    assert bs.top_blocks(m, 3).tolist() == [0, 1, 3]          # tie at 0.5: the lower block
    assert bs.top_blocks(m, 9).tolist() == [0, 1, 2, 3, 4]


def test_signal_updates_only_the_chosen_physical_blocks():
    acc = np.zeros(10)
    last = np.full(10, -1, dtype=np.int64)
    bt = np.array([7, 2, 9])                                  # logical block -> physical
    mass = np.array([0.25, 1.5, 0.75])
    acc, last = bs.apply_signal(acc, last, bt, np.array([1, 2]), mass, step=4)
    assert acc.tolist() == [0, 0, 1.5, 0, 0, 0, 0, 0, 0, 0.75]
    assert last.tolist() == [-1, -1, 4, -1, -1, -1, -1, -1, -1, 4]
    acc, last = bs.apply_signal(acc, last, bt, np.array([0, 1]), mass, step=5)
    assert acc[2] == 3.0 and acc[7] == 0.25 and last[9] == 4 and last[2] == 5


def test_metadata_sizes_match_the_page(golden):
    from oracle import costs
    rows = {r[0]: r[1:] for r in golden("block_metadata_bytes.txt")}
    req, per, val, unit = rows["metadata"]
    got = costs.block_metadata_bytes(int(req), int(per))
    assert got == 256 * 2000 * 8
    assert abs(got / 1e6 - float(val)) / float(val) < 0.05        # "about 4 MB" (4.1 MB)
    req, k, val, unit = rows["update"]
    assert costs.signal_update_bytes(int(req), int(k)) == int(val) * 1024   # 512 KiB exactly
