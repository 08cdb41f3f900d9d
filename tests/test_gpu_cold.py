"""GPU parity of the cold-page codec (offload = encode fused with the write of the cold block,
onboard = decode fused with the read of it) against the oracle, through the C ABI: cold blocks
byte for byte, hot pages bit for bit, for device and pinned host cold pools, separate and
combined K/V hot pools, scattered pages and slots, shapes that span several work items with a
ragged tail or need padding, lossless bytes, and out-of-range ids."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv(cuda):
    from nvfp4_paged_kv_gb300 import build
    build.build()
    import nvfp4_paged_kv_gb300 as m
    m.load()
    return m


def _bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _pages(kind, P, H, T, D, seed):
    g = synthetic.gen(seed)
    x = synthetic.outlier_blocks_bf16(P, H, T, D, g)
    return x if kind == "bf16" else synthetic.outlier_blocks_bf16(
        P, H, T, D, g, big=30.0, small=1e-2).to(torch.float16)


def _scalar(x, dev):
    return torch.tensor([x], dtype=torch.float32, device=dev)


# (H, T, D): small; 2304 blocks per tensor (two work items, ragged second); 15 blocks per
# tensor (every part padded to 16 bytes)
SHAPES = [(2, 16, 64), (4, 64, 144), (1, 3, 80), (8, 32, 128)]


@pytest.mark.parametrize("kind", ["bf16", "fp16"])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("host", [False, True])
def test_offload_onboard_parity(kv, cuda, kind, shape, host):
    H, T, D = shape
    P, slots, n = 11, 13, 9
    k = _pages(kind, P, H, T, D, seed=60).to(cuda)
    v = _pages(kind, P, H, T, D, seed=61).to(cuda)
    odt = oracle.BF16 if kind == "bf16" else oracle.FP16
    g_k = oracle.global_scale(_bits(k), odt, H, D, T)
    g_v = oracle.global_scale(_bits(v), odt, H, D, T)
    rng = np.random.default_rng(3)
    hot = rng.permutation(P)[:n].astype(np.int32)
    slot = rng.permutation(slots)[:n].astype(np.int32)
    extra_bytes = 32
    extra = torch.from_numpy(rng.integers(0, 256, size=(P, 64), dtype=np.uint8)).to(cuda)
    lay = kv.Layout(H, D, T)
    bl = kv.nvfp4_kv_cold_block_layout(lay, extra_bytes)
    ref = oracle.cold_block_layout(H, D, T, extra_bytes)
    assert [getattr(bl, f) for f in ("k_data", "k_scales", "v_data", "v_scales", "extra",
                                     "bytes")] == \
        [ref[f] for f in ("k_data", "k_scales", "v_data", "v_scales", "extra", "bytes")]
    if host:
        cold = torch.zeros((slots, bl.bytes), dtype=torch.uint8).pin_memory()
    else:
        cold = torch.zeros((slots, bl.bytes), dtype=torch.uint8, device=cuda)
    t = lambda a: torch.from_numpy(a).to(cuda)  # noqa: E731
    gk, gv = _scalar(g_k, cuda), _scalar(g_v, cuda)
    kv.nvfp4_kv_offload_pages(lay, k, v, cold, k_global_scale=gk, v_global_scale=gv,
                              hot_page_ids=t(hot), cold_slot_ids=t(slot), extra=extra,
                              extra_bytes=extra_bytes)
    torch.cuda.synchronize()
    want = oracle.cold_offload(_bits(k), _bits(v), odt, H, D, T, g_k, g_v, slots,
                               hot_page_ids=hot, cold_slot_ids=slot,
                               extra=extra.cpu().numpy(), extra_bytes=extra_bytes)
    assert np.array_equal(cold.cpu().numpy(), want)
    # onboard into other hot pages of fresh pools
    back = rng.permutation(P)[:n].astype(np.int32)
    k2, v2 = torch.zeros_like(k), torch.zeros_like(v)
    ex2 = torch.zeros((P, 48), dtype=torch.uint8, device=cuda)
    kv.nvfp4_kv_onboard_pages(lay, cold, k2, v2, k_global_scale=gk, v_global_scale=gv,
                              cold_slot_ids=t(slot), hot_page_ids=t(back), extra=ex2,
                              extra_bytes=extra_bytes)
    torch.cuda.synchronize()
    wk, wv, wex = oracle.cold_onboard(want, H, D, T, g_k, g_v, odt, P, cold_slot_ids=slot,
                                      hot_page_ids=back, extra_bytes=extra_bytes)
    assert np.array_equal(_bits(k2), wk)
    assert np.array_equal(_bits(v2), wv)
    got_ex = ex2.cpu().numpy()
    assert np.array_equal(got_ex[:, :extra_bytes], wex) and not got_ex[:, extra_bytes:].any()


def test_cold_codec_matches_the_page_codec(kv, cuda):
    """Offload's codes and scales are those of nvfp4_kv_quantize_pages, onboard's values those
    of nvfp4_kv_dequantize_pages (one combined K/V hot pool [pages, 2, H, T, D], g = 1 by
    default)."""
    P, H, T, D = 6, 8, 32, 128
    pool = torch.stack([_pages("bf16", P, H, T, D, seed=70), _pages("bf16", P, H, T, D, 71)],
                       dim=1).to(cuda)
    lay = kv.Layout(H, D, T)
    bl = kv.nvfp4_kv_cold_block_layout(lay)
    cold = torch.zeros((P, bl.bytes), dtype=torch.uint8, device=cuda)
    kv.nvfp4_kv_offload_pages(lay, pool[:, 0], pool[:, 1], cold)
    one = torch.ones(1, dtype=torch.float32, device=cuda)
    n = H * T * D
    for tix, (od, osc) in enumerate(((bl.k_data, bl.k_scales), (bl.v_data, bl.v_scales))):
        d = torch.zeros((P, H, T, D // 2), dtype=torch.uint8, device=cuda)
        s = torch.zeros((P, H, T, D // 16), dtype=torch.uint8, device=cuda)
        kv.nvfp4_kv_quantize_pages(lay, pool[:, tix].contiguous(), one, d, s)
        assert torch.equal(cold[:, od:od + n // 2], d.reshape(P, -1))
        assert torch.equal(cold[:, osc:osc + n // 16], s.reshape(P, -1))
    back = torch.zeros_like(pool)
    kv.nvfp4_kv_onboard_pages(lay, cold, back[:, 0], back[:, 1])
    for tix, (od, osc) in enumerate(((bl.k_data, bl.k_scales), (bl.v_data, bl.v_scales))):
        d = cold[:, od:od + n // 2].reshape(P, H, T, D // 2).contiguous()
        s = cold[:, osc:osc + n // 16].reshape(P, H, T, D // 16).contiguous()
        ref = torch.zeros((P, H, T, D), dtype=torch.bfloat16, device=cuda)
        kv.nvfp4_kv_dequantize_pages(lay, d, s, one, ref)
        assert torch.equal(back[:, tix], ref)


def test_cold_codec_flags_out_of_range_ids(kv, cuda):
    """A hot page id or slot outside its pool sets PAGE_OOB and that page is skipped."""
    P, H, T, D = 4, 2, 16, 64
    k = _pages("bf16", P, H, T, D, seed=80).to(cuda)
    v = _pages("bf16", P, H, T, D, seed=81).to(cuda)
    lay = kv.Layout(H, D, T)
    bl = kv.nvfp4_kv_cold_block_layout(lay)
    cold = torch.zeros((P, bl.bytes), dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    hot = torch.tensor([0, 9, 2, 3], dtype=torch.int32, device=cuda)
    slot = torch.tensor([0, 1, -1, 3], dtype=torch.int32, device=cuda)
    kv.nvfp4_kv_offload_pages(lay, k, v, cold, hot_page_ids=hot, cold_slot_ids=slot,
                              status=status)
    assert int(status.item()) & kv.STATUS_PAGE_OOB
    c = cold.cpu()
    assert c[0].any() and c[3].any() and not c[1].any() and not c[2].any()
    status.zero_()
    k2, v2 = torch.zeros_like(k), torch.zeros_like(v)
    kv.nvfp4_kv_onboard_pages(lay, cold, k2, v2, cold_slot_ids=slot, hot_page_ids=hot,
                              status=status)
    assert int(status.item()) & kv.STATUS_PAGE_OOB
    assert k2[0].ne(0).any() and not k2[1].ne(0).any() and not k2[2].ne(0).any()


def test_cold_codec_rejects_bad_arguments(kv, cuda):
    lay = kv.Layout(2, 64, 16)
    k = torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16, device=cuda)
    bl = kv.nvfp4_kv_cold_block_layout(lay)
    with pytest.raises(ValueError):      # pageable host memory
        kv.nvfp4_kv_offload_pages(lay, k, k, torch.zeros((2, bl.bytes), dtype=torch.uint8))
    with pytest.raises(kv.NVFP4KVError):  # extra bytes not a multiple of 16
        kv.nvfp4_kv_cold_block_layout(lay, 8)
    cold = torch.zeros((2, bl.bytes), dtype=torch.uint8, device=cuda)
    with pytest.raises(kv.NVFP4KVError):  # FP8 hot pool
        kv.nvfp4_kv_offload_pages(lay, k, k, cold, hot_dtype=kv.FP8_E4M3)


# (H, T, D, first_dim, dims): RoPE dims in the middle, two row items with a ragged second, the
# whole head, a three-row page
ROPE_CASES = [(2, 16, 128, 64, 64), (4, 64, 144, 16, 32), (2, 8, 64, 0, 64), (1, 3, 80, 32, 16)]


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("case", ROPE_CASES)
@pytest.mark.parametrize("kind", ["bf16", "fp16"])
def test_rope_modes_parity(kv, cuda, mode, case, kind):
    """The RoPE part of K kept at 16 bits (SKIP) or as two NVFP4 components (2FP4): cold blocks
    byte for byte and onboarded pages bit for bit against the oracle, through pinned host
    memory, scattered pages and slots."""
    H, T, D, first, dims = case
    P, slots, n = 7, 9, 5
    k = _pages(kind, P, H, T, D, seed=90).to(cuda)
    v = _pages(kind, P, H, T, D, seed=91).to(cuda)
    odt = oracle.BF16 if kind == "bf16" else oracle.FP16
    g_k = oracle.global_scale(_bits(k), odt, H, D, T)
    g_v = oracle.global_scale(_bits(v), odt, H, D, T)
    rng = np.random.default_rng(5)
    hot = rng.permutation(P)[:n].astype(np.int32)
    slot = rng.permutation(slots)[:n].astype(np.int32)
    lay = kv.Layout(H, D, T)
    rope = kv.ColdRope(mode, first, dims)
    bl = kv.nvfp4_kv_cold_block_layout(lay, 0, rope)
    cold = torch.zeros((slots, bl.bytes), dtype=torch.uint8).pin_memory()
    t = lambda a: torch.from_numpy(a).to(cuda)  # noqa: E731
    gk, gv = _scalar(g_k, cuda), _scalar(g_v, cuda)
    kv.nvfp4_kv_offload_pages(lay, k, v, cold, k_global_scale=gk, v_global_scale=gv,
                              hot_page_ids=t(hot), cold_slot_ids=t(slot), rope=rope)
    torch.cuda.synchronize()
    want = oracle.cold_offload(_bits(k), _bits(v), odt, H, D, T, g_k, g_v, slots,
                               hot_page_ids=hot, cold_slot_ids=slot, rope=(mode, first, dims))
    assert np.array_equal(cold.numpy(), want)
    k2, v2 = torch.zeros_like(k), torch.zeros_like(v)
    kv.nvfp4_kv_onboard_pages(lay, cold, k2, v2, k_global_scale=gk, v_global_scale=gv,
                              cold_slot_ids=t(slot), hot_page_ids=t(hot), rope=rope)
    torch.cuda.synchronize()
    wk, wv, _ = oracle.cold_onboard(want, H, D, T, g_k, g_v, odt, P, cold_slot_ids=slot,
                                    hot_page_ids=hot, rope=(mode, first, dims))
    assert np.array_equal(_bits(k2), wk)
    assert np.array_equal(_bits(v2), wv)
    if mode == 1:
        rc = slice(first, first + dims)
        assert torch.equal(k2[t(hot).long()][..., rc], k[t(hot).long()][..., rc])
