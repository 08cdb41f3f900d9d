"""GPU parity of the NVFP4 codec against the CPU oracle: bit-exact codes, scales, decoded
values and global scales, through the C ABI.

Cases span several CUDA work items and ragged tails (page counts and block counts that are not
multiples of the kernels' item sizes), every source / output dtype, page-id gathers and
scatters, the full page round-trip workload (4096 pages x 32 tokens x 8 heads x 128) and the
extend workload (a 1024-page prefix gathered into an FP8 workspace plus a 512-token chunk per
sequence quantized into new pages)."""
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


def _src_bits(t: torch.Tensor):
    if t.dtype == torch.bfloat16 or t.dtype == torch.float16:
        return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().contiguous().view(torch.uint8).numpy()


def _odt(t: torch.Tensor):
    return {torch.bfloat16: oracle.BF16, torch.float16: oracle.FP16}.get(t.dtype,
                                                                        oracle.FP8_E4M3)


def _make_src(kind, P, H, T, D, seed):
    g = synthetic.gen(seed)
    if kind == "bf16":
        return synthetic.outlier_blocks_bf16(P, H, T, D, g)
    if kind == "fp16":
        return synthetic.outlier_blocks_bf16(P, H, T, D, g, big=30.0, small=1e-2).to(
            torch.float16)
    return synthetic.random_fp8_bytes((P, H, T, D), g)


def _scalar(x, dev):
    return torch.tensor([x], dtype=torch.float32, device=dev)


# ------------------------------------------------------------------------------ roundings

@pytest.mark.slow
@pytest.mark.parametrize("target", [0, 1])
def test_rounding_exhaustive_fp32(kv, cuda, target):
    """Every finite fp32 bit pattern through the encoder's E2M1 (target 0) and E4M3 (target 1)
    rounding, GPU against the oracle, bit for bit."""
    chunk = 1 << 28
    x_dev = torch.empty(chunk, dtype=torch.int32, device=cuda)
    out_dev = torch.empty(chunk, dtype=torch.uint8, device=cuda)
    base = np.arange(chunk, dtype=np.uint32)
    for k in range(1 << 4):
        start = k * chunk
        pat = torch.arange(start, start + chunk, dtype=torch.int64, device=cuda)
        x_dev.copy_(torch.where(pat >= 2 ** 31, pat - 2 ** 32, pat))
        kv.nvfp4_kv_round_f32(x_dev.view(torch.float32), target, out_dev)
        got = out_dev.cpu().numpy()
        xs = (base + np.uint32(start)).view(np.float32)
        fin = np.isfinite(xs)
        want = (oracle.e2m1_encode_f32 if target == 0 else oracle.e4m3_encode_f32)(
            np.where(fin, xs, np.float32(0)))
        bad = np.nonzero((got != want) & fin)[0]
        assert bad.size == 0, [(hex(int(base[i]) + start), got[i], want[i]) for i in bad[:8]]


# ------------------------------------------------------------------------------ encode

@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp8"])
@pytest.mark.parametrize("shape", [(7, 3, 5, 48), (33, 8, 32, 128), (5, 2, 64, 256),
                                   (1, 1, 1, 16), (300, 2, 16, 64), (6, 3, 6, 48),
                                   (9, 2, 256, 128)])
@pytest.mark.parametrize("ids", [False, True])
@pytest.mark.parametrize("pack", [0, 1])
def test_quantize_parity(kv, cuda, kind, shape, ids, pack):
    P, H, T, D = shape
    if pack == 1 and T % 2:
        pytest.skip("token-pair packing needs an even page size")
    src = _make_src(kind, P, H, T, D, seed=P + D)
    lay = kv.Layout(H, D, T)
    rng = np.random.default_rng(P * 7 + D)
    src_scale = float(np.float32(0.37)) if kind == "fp8" else 1.0
    sbits = _src_bits(src)
    if ids:
        n = max(1, P - 2)
        sid = rng.permutation(P)[:n].astype(np.int32)
        did = rng.permutation(P + 3)[:n].astype(np.int32)
        npool = P + 3
    else:
        n, sid, did, npool = P, None, None, P
    g = oracle.global_scale(sbits, _odt(src), H, D, T, src_page_ids=sid, src_scale=src_scale)
    want_d, want_s = oracle.quantize_pages(sbits, _odt(src), H, D, T, g, num_dst_pages=npool,
                                           src_page_ids=sid, dst_page_ids=did,
                                           src_scale=src_scale, packing=pack)
    lay = kv.Layout(H, D, T, pack)
    src_dev = src.to(cuda)
    gs = torch.empty(1, dtype=torch.float32, device=cuda)
    ss = _scalar(src_scale, cuda) if kind == "fp8" else None
    sid_t = None if sid is None else torch.from_numpy(sid).to(cuda)
    did_t = None if did is None else torch.from_numpy(did).to(cuda)
    kv.nvfp4_kv_compute_global_scale(lay, src_dev, gs, src_page_ids=sid_t, src_scale=ss,
                                     src_dtype=kv.FP8_E4M3 if kind == "fp8" else None)
    assert gs.item() == np.float32(g)
    dshape, sshape = oracle.pool_shapes(npool, H, T, D, pack)
    data = torch.zeros(dshape, dtype=torch.uint8, device=cuda)
    scales = torch.zeros(sshape, dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kv.nvfp4_kv_quantize_pages(lay, src_dev, gs, data, scales, src_page_ids=sid_t,
                               dst_page_ids=did_t, src_scale=ss, status=status,
                               src_dtype=kv.FP8_E4M3 if kind == "fp8" else None)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(data.cpu().numpy(), want_d)


# ------------------------------------------------------------------------------ decode

@pytest.mark.parametrize("out_kind", ["bf16", "fp16", "fp8"])
@pytest.mark.parametrize("shape", [(9, 3, 16, 48), (40, 8, 32, 128), (1, 1, 1, 16),
                                   (3, 2, 2, 256), (5, 1, 3, 80), (9, 2, 256, 128)])
@pytest.mark.parametrize("pack", [0, 1])
def test_dequantize_parity(kv, cuda, out_kind, shape, pack):
    P, H, T, D = shape
    if pack == 1 and T % 2:
        pytest.skip("token-pair packing needs an even page size")
    rng = np.random.default_rng(P + H + D)
    ds, ss = oracle.pool_shapes(P, H, T, D, pack)
    data = rng.integers(0, 256, ds, dtype=np.uint8)
    scales = rng.integers(0, 0x7F, ss, dtype=np.uint8)  # every finite scale
    g = float(np.float32(0.0731))
    out_scale = float(np.float32(0.25)) if out_kind == "fp8" else 1.0
    odt = {"bf16": oracle.BF16, "fp16": oracle.FP16, "fp8": oracle.FP8_E4M3}[out_kind]
    sid = rng.permutation(P).astype(np.int32)
    did = rng.permutation(P + 2)[:P].astype(np.int32)
    want = oracle.dequantize_pages(data, scales, H, D, T, g, odt, num_dst_pages=P + 2,
                                   src_page_ids=sid, dst_page_ids=did, out_scale=out_scale,
                                   packing=pack)
    lay = kv.Layout(H, D, T, pack)
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp8": torch.uint8}[out_kind]
    dst = torch.zeros((P + 2, H, T, D), dtype=tdt, device=cuda)
    kv.nvfp4_kv_dequantize_pages(
        lay, torch.from_numpy(data).to(cuda), torch.from_numpy(scales).to(cuda),
        _scalar(g, cuda), dst, src_page_ids=torch.from_numpy(sid).to(cuda),
        dst_page_ids=torch.from_numpy(did).to(cuda),
        dst_scale=_scalar(out_scale, cuda) if out_kind == "fp8" else None,
        dst_dtype=odt)
    got = dst.cpu().contiguous()
    got = got.view(torch.int16).numpy().view(np.uint16) if out_kind != "fp8" else got.numpy()
    assert np.array_equal(got, want)


def test_page_roundtrip_workload_full_size(kv, cuda):
    """4096 pages x 32 tokens x 8 KV heads x 128, K and V ~ N(0,1) BF16 with 1% of blocks x1e3
    and 1% x1e-3; g = amax/(448*6) per tensor; encode, decode to BF16 and to FP8 E4M3 (output
    scale amax/448). Every byte against the oracle."""
    wl = synthetic.RoundTripWorkload()
    k, v = wl.make(device=cuda)
    for t, pack in ((k, 0), (v, 1)):       # K dim-pair packed, V token-pair packed
        lay = kv.Layout(wl.H, wl.D, wl.T, pack)
        bits = _src_bits(t)
        g = oracle.global_scale(bits, oracle.BF16, wl.H, wl.D, wl.T)
        amax = oracle.tensor_amax(bits, oracle.BF16, wl.H, wl.D, wl.T)
        out_scale = float(np.float32(amax) / np.float32(448.0))
        wd, wsc = oracle.quantize_pages(bits, oracle.BF16, wl.H, wl.D, wl.T, g, packing=pack)
        gs = torch.empty(1, dtype=torch.float32, device=cuda)
        kv.nvfp4_kv_compute_global_scale(lay, t, gs)
        assert gs.item() == np.float32(g)
        ds, ss = oracle.pool_shapes(wl.P, wl.H, wl.T, wl.D, pack)
        data = torch.empty(ds, dtype=torch.uint8, device=cuda)
        scales = torch.empty(ss, dtype=torch.uint8, device=cuda)
        kv.nvfp4_kv_quantize_pages(lay, t, gs, data, scales)
        assert np.array_equal(scales.cpu().numpy(), wsc)
        assert np.array_equal(data.cpu().numpy(), wd)
        back = torch.empty_like(t)
        kv.nvfp4_kv_dequantize_pages(lay, data, scales, gs, back)
        want_b = oracle.dequantize_pages(wd, wsc, wl.H, wl.D, wl.T, g, oracle.BF16,
                                         packing=pack)
        assert np.array_equal(_src_bits(back), want_b)
        f8 = torch.empty(t.shape, dtype=torch.uint8, device=cuda)
        kv.nvfp4_kv_dequantize_pages(lay, data, scales, gs, f8, dst_dtype=kv.FP8_E4M3,
                                     dst_scale=_scalar(out_scale, cuda))
        want_f = oracle.dequantize_pages(wd, wsc, wl.H, wl.D, wl.T, g, oracle.FP8_E4M3,
                                         out_scale=out_scale, packing=pack)
        assert np.array_equal(f8.cpu().numpy(), want_f)
        del data, scales, back, f8


def test_extend_workload(kv, cuda):
    """16 sequences: a 4096-token NVFP4 prefix each, gathered by page table and dequantized into
    a contiguous FP8 E4M3 workspace, and a 512-token BF16 chunk each quantized into new pages of
    the same pool."""
    wl = synthetic.ExtendWorkload()
    prefix, pt, chunk, chunk_dst = wl.make(device=cuda)
    lay = kv.Layout(wl.H, wl.D, wl.T)
    pool = prefix.shape[0]
    pbits = _src_bits(prefix)
    g = oracle.global_scale(pbits, oracle.BF16, wl.H, wl.D, wl.T)
    pool_d, pool_s = oracle.quantize_pages(pbits, oracle.BF16, wl.H, wl.D, wl.T, g)
    gs = _scalar(g, cuda)
    data = torch.from_numpy(pool_d).to(cuda)
    scales = torch.from_numpy(pool_s).to(cuda)
    ids = pt.reshape(-1).contiguous()
    ws = torch.empty((ids.numel(), wl.H, wl.T, wl.D), dtype=torch.uint8, device=cuda)
    kv.nvfp4_kv_dequantize_pages(lay, data, scales, gs, ws, dst_dtype=kv.FP8_E4M3,
                                 src_page_ids=ids)
    want = oracle.dequantize_pages(pool_d, pool_s, wl.H, wl.D, wl.T, g, oracle.FP8_E4M3,
                                   src_page_ids=ids.cpu().numpy())
    assert np.array_equal(ws.cpu().numpy(), want)
    # the current chunk goes into the free pages of the pool (same tensor scale)
    kv.nvfp4_kv_quantize_pages(lay, chunk, gs, data, scales, dst_page_ids=chunk_dst)
    cd = chunk_dst.cpu().numpy()
    wd, wsc = oracle.quantize_pages(_src_bits(chunk), oracle.BF16, wl.H, wl.D, wl.T, g,
                                    num_dst_pages=pool, dst_page_ids=cd)
    got_d, got_s = data.cpu().numpy(), scales.cpu().numpy()
    assert np.array_equal(got_d[cd], wd[cd]) and np.array_equal(got_s[cd], wsc[cd])
    untouched = np.setdiff1d(np.arange(pool), cd)
    assert np.array_equal(got_d[untouched], pool_d[untouched])


# ------------------------------------------------------------------------------ extend write

@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp8"])
@pytest.mark.parametrize("pack", [oracle.DIM_PAIRS, oracle.TOKEN_PAIRS])
@pytest.mark.parametrize("ws_scale", [1.0, 0.375])
def test_extend_write_parity(kv, cuda, kind, pack, ws_scale):
    """One pass over a chunk's pages (scattered sources, destinations and workspace slots, a
    ragged page count): the NVFP4 pages equal both the oracle and the plain quantize call, the
    FP8 workspace copy equals the oracle's E4M3(fp32(x * fp32(1 / ws_scale))), x read from FP8
    sources as fp32(e4m3 * src_scale)."""
    P, H, T, D = 37, 2, 32, 128
    src = _make_src(kind, P, H, T, D, seed=40 + pack).to(cuda)
    bits = _src_bits(src)
    odt = _odt(src)
    lay = kv.Layout(H, D, T).with_packing(pack)
    src_scale = float(np.float32(0.375)) if kind == "fp8" else 1.0
    sst = _scalar(src_scale, cuda) if kind == "fp8" else None
    sdt = kv.FP8_E4M3 if kind == "fp8" else None
    g = oracle.global_scale(bits, odt, H, D, T, src_scale=src_scale)
    gs = _scalar(g, cuda)
    rng = np.random.default_rng(7)
    n = 29
    sid = rng.permutation(P)[:n].astype(np.int32)
    did = rng.permutation(48)[:n].astype(np.int32)
    wid = rng.permutation(33)[:n].astype(np.int32)
    ds, ss = oracle.pool_shapes(48, H, T, D, pack)
    data = torch.zeros(ds, dtype=torch.uint8, device=cuda)
    scales = torch.zeros(ss, dtype=torch.uint8, device=cuda)
    ws = torch.zeros((33, H, T, D), dtype=torch.uint8, device=cuda)
    t = lambda a: torch.from_numpy(a).to(cuda)  # noqa: E731
    kv.nvfp4_kv_extend_write(lay, src, gs, data, scales, ws, src_page_ids=t(sid),
                             dst_page_ids=t(did), ws_page_ids=t(wid), src_scale=sst,
                             ws_scale=_scalar(ws_scale, cuda), src_dtype=sdt)
    want_d, want_s = oracle.quantize_pages(bits, odt, H, D, T, g, num_dst_pages=48,
                                           src_page_ids=sid, dst_page_ids=did,
                                           src_scale=src_scale, packing=pack)
    want_ws = oracle.cast_fp8_pages(bits, odt, H, D, T, ws_scale=ws_scale, num_dst_pages=33,
                                    src_page_ids=sid, dst_page_ids=wid, src_scale=src_scale)
    assert np.array_equal(data.cpu().numpy(), want_d)
    assert np.array_equal(scales.cpu().numpy(), want_s)
    assert np.array_equal(ws.cpu().numpy(), want_ws)
    # the NVFP4 half is exactly the plain quantize call
    d2, s2 = torch.zeros_like(data), torch.zeros_like(scales)
    kv.nvfp4_kv_quantize_pages(lay, src, gs, d2, s2, src_page_ids=t(sid), dst_page_ids=t(did),
                               src_scale=sst, src_dtype=sdt)
    assert torch.equal(d2, data) and torch.equal(s2, scales)
    if kind == "fp8" and ws_scale == src_scale:
        # an FP8 chunk written at its own scale is copied byte for byte
        assert torch.equal(ws[t(wid).long()], src[t(sid).long()])


def test_extend_write_flags_out_of_range_workspace_pages(kv, cuda):
    """A workspace page id outside its pool skips that page in all three pools."""
    P, H, T, D = 4, 2, 16, 64
    src = _make_src("bf16", P, H, T, D, seed=9).to(cuda)
    lay = kv.Layout(H, D, T)
    gs = _scalar(0.25, cuda)
    data = torch.zeros((P, H, T, D // 2), dtype=torch.uint8, device=cuda)
    scales = torch.zeros((P, H, T, D // 16), dtype=torch.uint8, device=cuda)
    ws = torch.zeros((P, H, T, D), dtype=torch.uint8, device=cuda)
    wid = torch.tensor([0, 7, 2, 3], dtype=torch.int32, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kv.nvfp4_kv_extend_write(lay, src, gs, data, scales, ws, ws_page_ids=wid, status=status)
    assert int(status.item()) & kv.STATUS_PAGE_OOB
    assert int(data[1].abs().sum()) == 0 and int(ws[1].abs().sum()) == 0
    assert int(data[0].ne(0).sum()) > 0 and int(ws[0].ne(0).sum()) > 0


# ------------------------------------------------------------------------------ faults

def test_out_of_range_page_ids_are_flagged_and_skipped(kv, cuda):
    P, H, T, D = 6, 2, 16, 64
    src = _make_src("bf16", P, H, T, D, seed=3).to(cuda)
    lay = kv.Layout(H, D, T)
    gs = _scalar(0.5, cuda)
    sid = torch.tensor([0, 1, 99, 3, -1, 5], dtype=torch.int32, device=cuda)
    data = torch.zeros((P, H, T, D // 2), dtype=torch.uint8, device=cuda)
    scales = torch.zeros((P, H, T, D // 16), dtype=torch.uint8, device=cuda)
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    kv.nvfp4_kv_quantize_pages(lay, src, gs, data, scales, src_page_ids=sid, status=status)
    torch.cuda.synchronize()
    assert status.item() & kv.STATUS_PAGE_OOB
    wd, wsc = oracle.quantize_pages(_src_bits(src), oracle.BF16, H, D, T, 0.5)
    got = data.cpu().numpy()
    for i in (0, 1, 3, 5):
        assert np.array_equal(got[i], wd[i])
    assert not got[2].any() and not got[4].any()
    status.zero_()
    dst = torch.zeros_like(src)
    kv.nvfp4_kv_dequantize_pages(lay, data, scales, gs, dst, dst_page_ids=sid, status=status)
    torch.cuda.synchronize()
    assert status.item() & kv.STATUS_PAGE_OOB
    status.zero_()
    kv.nvfp4_kv_compute_global_scale(lay, src, gs, src_page_ids=sid, status=status)
    torch.cuda.synchronize()
    assert status.item() & kv.STATUS_PAGE_OOB


def test_zero_pages_and_zero_tensor(kv, cuda):
    lay = kv.Layout(2, 32, 16)
    gs = torch.zeros(1, dtype=torch.float32, device=cuda)
    empty = torch.zeros((0, 2, 16, 32), dtype=torch.bfloat16, device=cuda)
    kv.nvfp4_kv_compute_global_scale(lay, empty, gs)
    assert gs.item() == 1.0
    z = torch.zeros((3, 2, 16, 32), dtype=torch.bfloat16, device=cuda)
    gs.zero_()
    kv.nvfp4_kv_compute_global_scale(lay, z, gs)
    assert gs.item() == 1.0


# ------------------------------------------------------------------------------ scale study

@pytest.mark.parametrize("calibrated", [False, True])
def test_global_scale_study_counts_match_the_oracle(kv, cuda, calibrated):
    """The benchmark's global-scale study (error and scale-range counts of g = 1 against
    g = amax / 2688) computed through the library equals the same statistics of the oracle's
    codes and decoded values on a sample with x1e3 and x1e-3 blocks."""
    import bench
    P, H, T, D = 16, 2, 16, 64
    x = synthetic.outlier_blocks_bf16(P, H, T, D, synthetic.gen(33), frac_big=0.02,
                                      frac_small=0.05).to(cuda)
    lay = kv.Layout(H, D, T)
    bits = _src_bits(x)
    g = oracle.global_scale(bits, oracle.BF16, H, D, T) if calibrated else 1.0
    st = bench.scale_stats(kv, lay, x, _scalar(g, cuda))
    d, s = oracle.quantize_pages(bits, oracle.BF16, H, D, T, g)
    y = oracle.dequantize_pages(d, s, H, D, T, g)
    xs = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(-1, 16)
    ys = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(-1, 16)
    sb = s.reshape(-1).astype(int)
    amax = np.abs(xs).max(1)
    nz = amax > 0
    assert st["blocks_zero_scale"] == int(((sb == 0) & nz).sum())
    assert st["blocks_subnormal_scale"] == int((((sb & 0x78) == 0) & (sb != 0)).sum())
    assert st["blocks_saturated_scale"] == int((amax / (6 * g) > 464).sum())
    assert st["values_clipped"] == int((np.abs(xs) > 7 * 448 * g).sum())
    err = xs - ys
    want = np.sqrt((err ** 2).sum()) / np.sqrt((xs ** 2).sum())
    assert abs(st["rel_rmse"] - want) <= 1e-5 * want + 1e-12
    if calibrated:
        assert st["blocks_saturated_scale"] == 0 and st["values_clipped"] == 0
    else:
        assert st["blocks_saturated_scale"] > 0 and st["blocks_zero_scale"] > 0


def test_global_scale_workspace_needs_no_clearing(kv, cuda):
    """One launch computes g through a tagged maximum and a tagged count in the workspace: g is
    right whatever the workspace holds (all ones, random bytes, the previous call's words), for
    calls that alternate between tensors of different maxima."""
    H, T, D = 2, 16, 64
    xs = [synthetic.outlier_blocks_bf16(9, H, T, D, synthetic.gen(s), big=b).to(cuda)
          for s, b in ((41, 1e3), (42, 3.0), (43, 50.0))]
    lay = kv.Layout(H, D, T)
    want = [oracle.global_scale(_src_bits(x), oracle.BF16, H, D, T) for x in xs]
    ws = torch.empty(kv.nvfp4_kv_global_scale_workspace_size(), dtype=torch.uint8, device=cuda)
    out = torch.empty(1, dtype=torch.float32, device=cuda)
    gen = torch.Generator(device="cpu").manual_seed(5)
    for trial in range(12):
        if trial == 0:
            ws.fill_(0xFF)
        elif trial % 4 == 1:
            ws.copy_(torch.randint(0, 256, ws.shape, generator=gen, dtype=torch.uint8))
        i = trial % 3
        kv.nvfp4_kv_compute_global_scale(lay, xs[i], out, workspace=ws)
        assert out.item() == want[i], (trial, out.item(), want[i])


# ------------------------------------------------------------------------------ round trips

@pytest.mark.parametrize("pack", [0, 1])
def test_round_trips_back_to_back_do_not_accumulate_error(kv, cuda, pack):
    """Encode -> decode to BF16 -> encode ... four times on one stream with no host
    synchronisation between the launches (each launch reads the previous one's output; the
    kernels are launched with programmatic dependent launch). "KV Cache Compression in TensorRT
    LLM", "Evaluation -> Accuracy", Figure 15: repeated round trips add no error. Under the
    encoder's arithmetic this holds exactly for every block whose E4M3 scale is zero or normal;
    a block whose scale is subnormal may move once more on trip 2, and nothing moves from trip 3
    on. The first trip's codes and scales are checked against the oracle's encoding."""
    P, H, T, D = 37, 3, 32, 96
    NB = D // 16
    x = _make_src("bf16", P, H, T, D, seed=41).to(cuda)
    lay = kv.Layout(H, D, T, pack)
    g = torch.empty(1, device=cuda)
    kv.nvfp4_kv_compute_global_scale(lay, x, g)
    dsh, ssh = oracle.pool_shapes(P, H, T, D, pack)
    trips = []
    cur = x
    for _ in range(4):
        data = torch.empty(dsh, dtype=torch.uint8, device=cuda)
        sc = torch.empty(ssh, dtype=torch.uint8, device=cuda)
        kv.nvfp4_kv_quantize_pages(lay, cur, g, data, sc)
        back = torch.empty_like(x)
        kv.nvfp4_kv_dequantize_pages(lay, data, sc, g, back)
        trips.append((data, sc, back))
        cur = back
    torch.cuda.synchronize()
    ref_d, ref_s = oracle.quantize_pages(_src_bits(x), oracle.BF16, H, D, T, float(g.item()),
                                         packing=pack)
    assert np.array_equal(trips[0][0].cpu().numpy(), ref_d)
    assert np.array_equal(trips[0][1].cpu().numpy(), ref_s)
    # trip-1 scale of every (page, head, token, block)
    s1 = trips[0][1].cpu().numpy()
    if pack == 1:
        s1 = s1.reshape(P, H, T // 2, NB, 2).transpose(0, 1, 2, 4, 3).reshape(P, H, T, NB)
    s1 = s1.astype(np.int32)
    settled = (s1 == 0) | (((s1 >> 3) & 0xF) != 0)        # zero or normal E4M3 scale
    backs = [_src_bits(t[2]).reshape(P, H, T, NB, 16) for t in trips]
    assert np.array_equal(backs[1][settled], backs[0][settled]), "a settled block moved on trip 2"
    for k in (2, 3):
        assert np.array_equal(backs[k], backs[1]), f"values moved on trip {k + 1}"
        assert torch.equal(trips[k][0], trips[1][0]) and torch.equal(trips[k][1], trips[1][1])


@pytest.mark.parametrize("kind", ["bf16", "fp16", "fp8"])
def test_extend_step_equals_the_separate_calls(kv, cuda, kind):
    """The extend step of K (dim pairs) and V (token pairs) in one launch: scattered prefix
    pages gathered to FP8 workspace slots and a ragged chunk written as NVFP4 pages and FP8
    slots, with a workspace scale. Bit-identical to the two separate calls per tensor, and the
    gathered prefix and the chunk's pages equal the oracle's."""
    H, T, D = 2, 32, 128
    P_pool, n_prefix, n_chunk, n_ws = 60, 23, 9, 40
    ws_scale = float(np.float32(1.5))
    src_scale = float(np.float32(0.375)) if kind == "fp8" else 1.0
    rng = np.random.default_rng(11)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda)  # noqa: E731
    perm = rng.permutation(P_pool).astype(np.int32)
    prefix_ids, chunk_dst = perm[:n_prefix], perm[n_prefix:n_prefix + n_chunk]
    wperm = rng.permutation(n_ws).astype(np.int32)
    ws_prefix, ws_chunk = wperm[:n_prefix], wperm[n_prefix:n_prefix + n_chunk]
    parts, sep, want = [], [], []
    for ti, pack in enumerate((oracle.DIM_PAIRS, oracle.TOKEN_PAIRS)):
        lay = kv.Layout(H, D, T).with_packing(pack)
        pool_src = _make_src("bf16", P_pool, H, T, D, seed=60 + ti).to(cuda)
        pbits = _src_bits(pool_src)
        g = oracle.global_scale(pbits, oracle.BF16, H, D, T)
        gs = _scalar(g, cuda)
        ds, ss = oracle.pool_shapes(P_pool, H, T, D, pack)
        data = torch.zeros(ds, dtype=torch.uint8, device=cuda)
        scales = torch.zeros(ss, dtype=torch.uint8, device=cuda)
        kv.nvfp4_kv_quantize_pages(lay, pool_src, gs, data, scales)
        chunk = _make_src(kind, 12, H, T, D, seed=70 + ti).to(cuda)
        chunk_ids = rng.permutation(12)[:n_chunk].astype(np.int32)
        sst = _scalar(src_scale, cuda) if kind == "fp8" else None
        sdt = kv.FP8_E4M3 if kind == "fp8" else None
        ws = torch.zeros((n_ws, H, T, D), dtype=torch.uint8, device=cuda)
        part = dict(layout=lay, global_scale=gs, data=data.clone(), scales=scales.clone(),
                    prefix_page_ids=t(prefix_ids), ws=ws.clone(), ws_prefix_ids=t(ws_prefix),
                    ws_chunk_ids=t(ws_chunk), ws_scale=_scalar(ws_scale, cuda), chunk=chunk,
                    chunk_page_ids=t(chunk_ids), chunk_src_scale=sst, chunk_dst_ids=t(chunk_dst),
                    chunk_dtype=sdt)
        parts.append(part)
        # the separate calls on their own copies
        d2, s2, w2 = data.clone(), scales.clone(), ws.clone()
        kv.nvfp4_kv_dequantize_pages(lay, d2, s2, gs, w2, dst_dtype=kv.FP8_E4M3,
                                     src_page_ids=t(prefix_ids), dst_page_ids=t(ws_prefix),
                                     dst_scale=_scalar(ws_scale, cuda))
        kv.nvfp4_kv_extend_write(lay, chunk, gs, d2, s2, w2, src_page_ids=t(chunk_ids),
                                 dst_page_ids=t(chunk_dst), ws_page_ids=t(ws_chunk),
                                 ws_scale=_scalar(ws_scale, cuda), src_scale=sst, src_dtype=sdt)
        sep.append((d2, s2, w2))
        # the oracle: the prefix pages' FP8 values and the chunk's NVFP4 pages
        hd, hs = data.cpu().numpy(), scales.cpu().numpy()
        want_prefix = oracle.dequantize_pages(hd, hs, H, D, T, g, oracle.FP8_E4M3,
                                              out_scale=ws_scale, src_page_ids=prefix_ids,
                                              packing=pack)
        cbits = _src_bits(chunk)
        want_d, want_s = oracle.quantize_pages(cbits, _odt(chunk), H, D, T, g,
                                               num_dst_pages=P_pool, src_page_ids=chunk_ids,
                                               dst_page_ids=chunk_dst, src_scale=src_scale,
                                               packing=pack)
        want.append((want_prefix, want_d, want_s))
    kv.nvfp4_kv_extend_step(parts)
    torch.cuda.synchronize()
    for part, (d2, s2, w2), (want_prefix, want_d, want_s) in zip(parts, sep, want):
        assert torch.equal(part["data"], d2) and torch.equal(part["scales"], s2)
        assert torch.equal(part["ws"], w2)
        got_ws = part["ws"].cpu().numpy()
        assert np.array_equal(got_ws[ws_prefix], want_prefix.reshape(got_ws[ws_prefix].shape))
        gd, gsc = part["data"].cpu().numpy(), part["scales"].cpu().numpy()
        assert np.array_equal(gd[chunk_dst], want_d[chunk_dst])
        assert np.array_equal(gsc[chunk_dst], want_s[chunk_dst])
    # one tensor alone, and an empty call
    solo = dict(parts[1])
    solo["data"], solo["scales"], solo["ws"] = (torch.zeros_like(solo["data"]),
                                                torch.zeros_like(solo["scales"]),
                                                torch.zeros_like(solo["ws"]))
    kv.nvfp4_kv_extend_step([solo])
    assert torch.equal(solo["ws"][t(ws_chunk).long()], sep[1][2][t(ws_chunk).long()])
