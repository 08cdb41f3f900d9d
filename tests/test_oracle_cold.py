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


# ---------------------------------------------------------------- the RoPE part of K

def _codes_values(codes, scales):
    """Exact block values e2m1(c) * e4m3(s) of packed codes [n, 8] and scales [n]: [n, 16]."""
    lo = (codes & 15).astype(int)
    hi = (codes >> 4).astype(int)
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], 16)
    e = np.vectorize(oracle.e2m1_value)(c)
    s = np.vectorize(oracle.e4m3_value)(scales.astype(int))
    return e * s[:, None]


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def test_2fp4_is_exact_on_the_grid():
    """Blocks s * (E2M1 grid) with g = 1: the first component is exact, so the residual is 0,
    the second component is all +0 codes with scale 0, and decoding returns x (a -0 comes back
    as +0: the decode sums -0 and +0)."""
    rng = np.random.default_rng(21)
    bits, x = _grid_pages(rng, 2, 1, 4, 32)
    c1, s1, c2, s2 = oracle.encode_2fp4_blocks(bits, oracle.BF16, 1.0)
    assert not c2.any() and not s2.any()
    y = oracle.decode_2fp4_blocks(c1, s1, c2, s2, 1.0, oracle.BF16)
    plus_zero = np.where(bits == 0x8000, 0, bits)
    assert np.array_equal(y.reshape(-1), plus_zero.reshape(-1))
    assert np.array_equal(_codes_values(c1, s1).reshape(-1), x.reshape(-1))


@pytest.mark.parametrize("g", [1.0, 0.0123])
def test_2fp4_second_component_encodes_the_first_ones_error(g):
    """Random BF16 blocks: the residual is r = fp32(x - fp32(v1 g)); the second component is the
    plain encoding of r (scale E4M3(amax(r) / fp32(6 g)), each code the nearest E2M1 value of
    fp32(r / fp32(s2 g)) by brute force), and the two-component value is never farther from x
    than the first component alone (0 is on the E2M1 grid)."""
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((64, 16)) * rng.choice([1e-2, 1.0, 40.0], (64, 1))).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # truncate to BF16
    xv = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    c1, s1, c2, s2 = oracle.encode_2fp4_blocks(bits, oracle.BF16, g)
    gf = float(np.float32(g))
    y1 = _f32(_codes_values(c1, s1) * gf)
    r = _f32(xv - y1)
    d = float(np.float32(6.0 * gf))
    grid = [oracle.e2m1_value(c) for c in range(16)]
    for b in range(64):
        s_expect = oracle.e4m3_encode(float(np.float32(np.abs(r[b]).max() / d)))
        assert s2[b] == s_expect
        sg = float(np.float32(oracle.e4m3_value(int(s2[b])) * gf))
        rcp = 0.0 if sg == 0.0 else float(np.float32(1.0 / sg))
        for k in range(16):
            q = float(np.float32(r[b, k] * rcp))
            code = (c2[b, k // 2] >> (4 * (k & 1))) & 15
            best = min(abs(q - e) for e in grid[:8]) if q >= 0 else min(abs(q - e) for e in grid[8:])
            assert abs(q - grid[code]) == best or abs(q) > 6
    y2 = _f32(y1 + _f32(_codes_values(c2, s2) * gf))
    assert np.all(np.abs(xv - y2) <= np.abs(xv - y1) * (1 + 2 ** -20) + 1e-30)
    assert np.abs(xv - y2).mean() < 0.25 * np.abs(xv - y1).mean()


def test_skip_rope_block_bytes_by_hand():
    """SKIP keeps the RoPE dims as 16-bit values at k_rope + (row R + d - first) * 2: a page that
    is zero except one BF16 value 1.5 (0x3FC0) at (head 1, token 3, dim first + 5) shows exactly
    there; the other dims' codes and scales are all zero."""
    H, T, D, first, R = 2, 4, 64, 32, 16
    k = np.zeros((1, H, T, D), np.uint16)
    v = np.zeros((1, H, T, D), np.uint16)
    k[0, 1, 3, first + 5] = 0x3FC0
    rope = (oracle.ROPE_SKIP, first, R)
    blocks = oracle.cold_offload(k, v, oracle.BF16, H, D, T, 1.0, 1.0, 1, rope=rope)
    lay = oracle.cold_block_layout(H, D, T, 0, rope)
    want = np.zeros(lay["bytes"], np.uint8)
    off = lay["k_rope"] + ((1 * T + 3) * R + 5) * 2
    want[off], want[off + 1] = 0xC0, 0x3F
    assert np.array_equal(blocks[0], want)


@pytest.mark.parametrize("mode", [1, 2])
def test_rope_round_trip(mode):
    """SKIP returns the RoPE dims bit for bit; 2FP4 returns decode_2fp4 of them; the other dims
    are what a plain NVFP4 round trip of those dims gives, whatever the RoPE mode."""
    rng = np.random.default_rng(23)
    P, H, T, D, first, R = 3, 2, 8, 64, 16, 32
    k = (rng.standard_normal((P, H, T, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    v = (rng.standard_normal((P, H, T, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rope = (mode, first, R)
    g = 0.01
    blocks = oracle.cold_offload(k, v, oracle.BF16, H, D, T, g, g, P, rope=rope)
    kk, vv, _ = oracle.cold_onboard(blocks, H, D, T, g, g, oracle.BF16, P, rope=rope)
    rc = np.arange(first, first + R)
    oc = np.setdiff1d(np.arange(D), rc)
    if mode == 1:
        assert np.array_equal(kk[..., rc], k[..., rc])
    else:
        c1, s1, c2, s2 = oracle.encode_2fp4_blocks(np.ascontiguousarray(k[..., rc]), oracle.BF16, g)
        assert np.array_equal(kk[..., rc].reshape(-1),
                              oracle.decode_2fp4_blocks(c1, s1, c2, s2, g).reshape(-1))
    kd, ks = oracle.quantize_pages(np.ascontiguousarray(k[..., oc]), oracle.BF16, H, D - R, T, g)
    assert np.array_equal(kk[..., oc], oracle.dequantize_pages(kd, ks, H, D - R, T, g))
    vd, vs = oracle.quantize_pages(v, oracle.BF16, H, D, T, g)
    assert np.array_equal(vv, oracle.dequantize_pages(vd, vs, H, D, T, g))
