"""The 1-byte V tile layout the library's header states, as the tests'
helper restates it: a bijection of each tile's 16 * D bytes, hand-worked
positions, and the INT8 offset, checked without a GPU."""
import numpy as np

from gpu_helpers import v_pool_logical, v_pool_stored, v_tile_positions


def test_positions_are_a_permutation_of_the_tile():
    for d in (64, 128):
        pos = v_tile_positions(d)
        assert pos.shape == (16, d)
        assert np.array_equal(np.sort(pos.reshape(-1)), np.arange(16 * d))


def test_hand_worked_positions_d128():
    pos = v_tile_positions(128)
    # dim 0: tokens 0, 1, 8, 9 are bytes 0..3 of lane 0's first word
    assert [pos[0, 0], pos[1, 0], pos[8, 0], pos[9, 0]] == [0, 1, 2, 3]
    # tokens 2, 3, 10, 11 belong to lane 1 (its 64-byte region starts at 64)
    assert [pos[2, 0], pos[3, 0], pos[10, 0], pos[11, 0]] == [64, 65, 66, 67]
    # dim 8 is the lane's second word, dim 16 its third, dim 32 its fifth
    # (chunk 1; lane 0's chunks are not permuted)
    assert pos[0, 8] == 4 and pos[0, 16] == 8 and pos[0, 32] == 16
    # lane 2 (tokens 4, 5, 12, 13 of dim 0): chunk 0 stored at chunk 0 ^ 1
    assert pos[4, 0] == 2 * 64 + 16
    # dim 1 goes to lane 4 (gid 1), whose chunk permutation is 2
    assert pos[0, 1] == 4 * 64 + 32


def test_hand_worked_positions_d64():
    pos = v_tile_positions(64)
    assert [pos[0, 0], pos[1, 0], pos[8, 0], pos[9, 0]] == [0, 1, 2, 3]
    assert pos[2, 0] == 32          # lane 1
    assert pos[0, 1] == 4 * 32 + 16  # lane 4: chunk 0 stored at chunk 1


def test_stored_and_logical_are_inverse_and_offset():
    rng = np.random.default_rng(1)
    for d in (64, 128):
        codes = rng.integers(-127, 128, size=(3, 2, 16, d)).astype(np.int8)
        st = v_pool_stored(codes, fp8=False)
        assert st.dtype == np.int8
        back = v_pool_logical(st, fp8=False)
        assert np.array_equal(back, codes)
        # offset binary: the stored byte of code c is c + 128
        pos = v_tile_positions(d)
        assert int(st[1, 1].reshape(-1).view(np.uint8)[pos[5, 7]]) == int(codes[1, 1, 5, 7]) + 128
        e4 = rng.integers(0, 255, size=(2, 2, 16, d)).astype(np.uint8)
        assert np.array_equal(v_pool_logical(v_pool_stored(e4, fp8=True), fp8=True), e4)
        assert v_pool_stored(e4, fp8=True)[0, 0].reshape(-1)[pos[3, 9]] == e4[0, 0, 3, 9]
