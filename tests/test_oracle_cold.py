"""Pins of the oracle's cold-page block functions ("KV Cache Compression in TensorRT LLM",
NVIDIA: "NVFP4 Cold-Page Compression", Figure 6 and Figure 7) against facts fixed outside
the functions themselves: the storage size of 4.5 bits per value, bytes worked out by hand from
the E2M1 / E4M3 definitions at hand-computed offsets, exact round trips of values on the
NVFP4 grid, untouched slots and lossless bytes."""
import numpy as np
import pytest

import oracle


def _bf16_bits(x):
    """BF16 patterns of float values that are exactly representable in BF16."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32)
    assert not np.any(b & 0xFFFF), "value not exact in BF16"
    return (b >> 16).astype(np.uint16)


@pytest.mark.parametrize("H,T,D", [(8, 32, 128), (8, 64, 128), (2, 16, 64), (4, 64, 256)])
def test_cold_block_is_4_5_bits_per_value(H, T, D):
    """Figure 6: the cold page of K and V holds 4-bit data plus one 8-bit scale per 16 values,
    i.e. 4.5 bits per value: 9/32 of the 16-bit hot page, with no padding at these shapes."""
    lay = oracle.cold_block_layout(H, D, T)
    hot_bytes = 2 * H * T * D * 2
    assert lay["bytes"] * 32 == hot_bytes * 9
    assert (lay["k_data"], lay["k_scales"], lay["v_data"], lay["v_scales"]) == (
        0, H * T * D // 2, H * T * D * 9 // 16, H * T * D * 9 // 16 + H * T * D // 2)
    assert oracle.cold_block_layout(H, D, T, 4096)["bytes"] == lay["bytes"] + 4096


def test_cold_block_pads_each_part_to_16_bytes():
    """One token of one head with 16 dims: 8 code bytes and 1 scale byte per tensor, each part
    rounded up to 16 bytes."""
    lay = oracle.cold_block_layout(1, 16, 1, 32)
    assert [lay[k] for k in ("k_data", "k_scales", "v_data", "v_scales", "extra", "bytes")] == \
        [0, 16, 32, 48, 64, 96]


def test_cold_block_bytes_by_hand():
    """A page that is zero except one block of K at (head 1, token 2, block 3) holding the whole
    E2M1 grid with both signs, and the same values doubled in V at (head 0, token 5, block 0),
    g = 1. By the format definitions: K scale E4M3(6 / 6) = 1.0 = 0x38, V scale 2.0 = 0x40; the
    codes are 0..15 in order, packed low nibble first; every other block has scale 0 and code 0."""
    H, T, D = 2, 8, 64
    grid = [0.0, 0.5, 1, 1.5, 2, 3, 4, 6]
    vals = np.array(grid + [-x for x in grid], dtype=np.float32)
    vals[8] = -0.0
    k = np.zeros((1, H, T, D), dtype=np.uint16)
    v = np.zeros((1, H, T, D), dtype=np.uint16)
    k[0, 1, 2, 48:64] = _bf16_bits(vals)
    v[0, 0, 5, 0:16] = _bf16_bits(2 * vals)
    blocks = oracle.cold_offload(k, v, oracle.BF16, H, D, T, 1.0, 1.0, num_slots=1)
    lay = oracle.cold_block_layout(H, D, T)
    want = np.zeros(lay["bytes"], dtype=np.uint8)
    codes = bytes([0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE])
    nb = D // 16
    kblk = (1 * T + 2) * nb + 3       # block index of (head 1, token 2, block 3)
    vblk = (0 * T + 5) * nb + 0
    want[lay["k_data"] + kblk * 8:lay["k_data"] + kblk * 8 + 8] = list(codes)
    want[lay["k_scales"] + kblk] = 0x38
    want[lay["v_data"] + vblk * 8:lay["v_data"] + vblk * 8 + 8] = list(codes)
    want[lay["v_scales"] + vblk] = 0x40
    assert np.array_equal(blocks[0], want)


def _grid_pages(rng, P, H, T, D):
    """BF16 pages whose every block is s * (E2M1 grid values) for a normal E4M3 s, so that the
    NVFP4 encoding with g = 1 is exact."""
    grid = np.array([0.0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    e = grid[rng.integers(0, 8, size=(P, H, T, D))] * rng.choice([-1.0, 1.0], size=(P, H, T, D))
    e[..., ::16] = 6.0                                     # every block reaches the top code
    s = 2.0 ** rng.integers(-6, 7, size=(P, H, T, D // 16, 1)) * rng.choice(
        [1.0, 1.125, 1.25, 1.5, 1.75], size=(P, H, T, D // 16, 1))
    x = (e.reshape(P, H, T, D // 16, 16) * s).reshape(P, H, T, D)
    return _bf16_bits(x.astype(np.float32)), x


def test_cold_round_trip_is_exact_on_the_grid():
    """Offload then onboard returns every value of grid-valued pages exactly (BF16 and FP16
    hot pools), through scattered hot pages and slots, with the lossless bytes unchanged."""
    rng = np.random.default_rng(11)
    P, H, T, D = 5, 2, 8, 32
    kb, kx = _grid_pages(rng, P, H, T, D)
    vb, vx = _grid_pages(rng, P, H, T, D)
    extra = rng.integers(0, 256, size=(P, 48), dtype=np.uint8)
    hot = np.array([4, 1, 3], dtype=np.int32)
    slots = np.array([2, 0, 5], dtype=np.int32)
    blocks = oracle.cold_offload(kb, vb, oracle.BF16, H, D, T, 1.0, 1.0, num_slots=6,
                                 hot_page_ids=hot, cold_slot_ids=slots, extra=extra,
                                 extra_bytes=32)
    back_hot = np.array([0, 2, 1], dtype=np.int32)
    for odt, value in ((oracle.BF16, oracle.bf16_value), (oracle.FP16, oracle.fp16_value)):
        k, v, ex = oracle.cold_onboard(blocks, H, D, T, 1.0, 1.0, odt, num_hot_pages=3,
                                       cold_slot_ids=slots, hot_page_ids=back_hot,
                                       extra_bytes=32)
        for i in range(3):
            got_k = np.vectorize(value)(k[back_hot[i]]).astype(np.float64)
            got_v = np.vectorize(value)(v[back_hot[i]]).astype(np.float64)
            assert np.array_equal(got_k, kx[hot[i]])
            assert np.array_equal(got_v, vx[hot[i]])
            assert np.array_equal(ex[back_hot[i]], extra[hot[i], :32])


def test_cold_offload_leaves_other_slots_untouched():
    """Slots that no page maps to stay zero; a slot holds the block of the page mapped to it."""
    rng = np.random.default_rng(12)
    P, H, T, D = 3, 1, 4, 16
    kb, _ = _grid_pages(rng, P, H, T, D)
    vb, _ = _grid_pages(rng, P, H, T, D)
    all_blocks = oracle.cold_offload(kb, vb, oracle.BF16, H, D, T, 1.0, 1.0, num_slots=3)
    some = oracle.cold_offload(kb, vb, oracle.BF16, H, D, T, 1.0, 1.0, num_slots=4,
                               hot_page_ids=[2, 0], cold_slot_ids=[3, 0])
    assert not some[1].any() and not some[2].any()
    assert np.array_equal(some[3], all_blocks[2]) and np.array_equal(some[0], all_blocks[0])
