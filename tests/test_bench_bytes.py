"""The bench's algorithmic bytes (the roofline numerator), from routing and masks, against
counts worked out by hand.  FloE's kernel reads, per routed expert, the packed INT2 up
projection whole and only the threshold-kept columns of the gate and down projections
(FloE, section 3, Algorithm 1 and the kernel optimisation list); a column kept for
several tokens of one expert is read once."""
import numpy as np

import bench


def words_of(cols_per_slot, nwords):
    """uint32 mask words of one (token, slot): bit c of word c // 32 for each kept column c."""
    w = np.zeros(nwords, dtype=np.uint32)
    for c in cols_per_slot:
        w[c // 32] |= np.uint32(1) << np.uint32(c % 32)
    return w


def test_one_token_two_experts():
    d, f, E, k, B, up = 256, 64, 8, 2, 1, 1000
    idx = np.array([[3, 5]])
    words = np.stack([np.stack([words_of([0, 1, 33], 2), words_of([2], 2)])])
    r = bench.count_bytes(idx, words, d, f, E, k, B, up)
    # 4 kept columns x 4 d bytes; 2 up projections; router 2 d E; x and y 2 B d each
    assert r["gather"] == 4 * 4 * 256 == 4096
    assert r["total"] == 2 * 1000 + 4096 + 2 * 256 * 8 + 2 * 256 * 2 == 11216
    assert r["up"] == 2000 + 512
    assert r["route"] == 4096 + 512
    assert r["kept_frac"] == 4 / 128
    assert r["pairs"] == 2


def test_shared_expert_reads_the_union_once():
    d, f, E, k, B, up = 256, 64, 8, 2, 2, 1000
    # token 0 -> experts 3, 5; token 1 -> experts 5, 7: three distinct experts
    idx = np.array([[3, 5], [5, 7]])
    words = np.stack([
        np.stack([words_of([0], 2), words_of([2, 40], 2)]),
        np.stack([words_of([2, 63], 2), words_of([], 2)]),
    ])
    r = bench.count_bytes(idx, words, d, f, E, k, B, up)
    # expert 3: {0}; expert 5: {2, 40} | {2, 63} = {2, 40, 63}; expert 7: {}  -> 4 columns
    assert r["gather"] == 4 * 256 * 4
    assert r["total"] == 3 * 1000 + 4 * 256 * 4 + 2 * 256 * 8 + 2 * 2 * 256 * 2 == 13240
    assert r["kept_frac"] == 4 / (64 * 3)
    assert r["pairs"] == 4


def test_bits_past_f_are_not_columns():
    d, f, E, k, B, up = 256, 40, 8, 1, 1, 0
    idx = np.array([[1]])
    words = np.stack([np.stack([words_of([39, 40, 50, 63], 2)])])
    r = bench.count_bytes(idx, words, d, f, E, k, B, up)
    assert r["gather"] == 4 * 256 * 1  # only column 39 exists
