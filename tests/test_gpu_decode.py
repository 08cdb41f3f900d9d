"""GPU parity of NVFP4 paged decode attention against the fp64 CPU oracle, through the C ABI.

Tolerance on the BF16 outputs: max |gpu - oracle| <= 1e-2 and mean |gpu - oracle| <= 1e-3 (BF16
rounding of outputs of magnitude up to a few units, plus FP16 rounding of the softmax weights);
LSE within 1e-3. The error of NVFP4 attention against
attention over the unquantized BF16 K/V is printed, not asserted.

The NVFP4 pages every case decodes are produced by the GPU quantizer and checked byte for byte
against the oracle's encoding of the same BF16 pages first, so the oracle and the kernel see
the same cache."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = pytest.mark.gpu

# Attention tolerance on BF16 outputs against the fp64 oracle: max-abs 1e-2 on top of the output's
# own rounding to BF16 (half an ulp of the exact value: 2^-6 for |x| in [4, 8), where no BF16 value
# lies within 1e-2 of every real number), mean-abs 1e-3; LSE (fp32) within 1e-3.
MAX_ABS, MEAN_ABS, LSE_ABS = 1e-2, 1e-3, 1e-3


def bf16_half_ulp(x):
    """Half the spacing of BF16 values around |x| (0 at 0): the rounding error of a correctly
    rounded BF16 output."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (np.maximum(e, -126.0) - 8), 0.0)


@pytest.fixture(scope="module")
def kv(cuda):
    from nvfp4_paged_kv_gb300 import build
    build.build()
    import nvfp4_paged_kv_gb300 as m
    m.load()
    return m


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Cache:
    """NVFP4 K/V pool quantized on the GPU, verified against the oracle's bytes."""

    def __init__(self, kv, dev, k, v, H, D, T, verify=True):
        self.lay = kv.Layout(H, D, T)
        self.H, self.D, self.T = H, D, T
        P = k.shape[0]
        kd, vd = k.to(dev), v.to(dev)
        self.gk = torch.empty(1, dtype=torch.float32, device=dev)
        self.gv = torch.empty(1, dtype=torch.float32, device=dev)
        kv.nvfp4_kv_compute_global_scale(self.lay, kd, self.gk)
        kv.nvfp4_kv_compute_global_scale(self.lay, vd, self.gv)
        mk = lambda w: torch.empty((P, H, T, w), dtype=torch.uint8, device=dev)  # noqa: E731
        self.kd, self.ks, self.vd, self.vs = mk(D // 2), mk(D // 16), mk(D // 2), mk(D // 16)
        kv.nvfp4_kv_quantize_pages(self.lay, kd, self.gk, self.kd, self.ks)  # K: dim pairs
        kv.nvfp4_kv_quantize_pages(self.lay.with_packing(kv.PACK_TOKEN_PAIRS), vd, self.gv,
                                   self.vd, self.vs)                        # V: token pairs
        torch.cuda.synchronize()
        self.g_k, self.g_v = self.gk.item(), self.gv.item()
        self.host = [t.cpu().numpy() for t in (self.kd, self.ks, self.vd, self.vs)]
        if verify:
            kb, vb = bits(k), bits(v)
            assert self.g_k == oracle.global_scale(kb, oracle.BF16, H, D, T)
            assert self.g_v == oracle.global_scale(vb, oracle.BF16, H, D, T)
            wkd, wks = oracle.quantize_pages(kb, oracle.BF16, H, D, T, self.g_k)
            wvd, wvs = oracle.quantize_pages(vb, oracle.BF16, H, D, T, self.g_v,
                                             packing=oracle.TOKEN_PAIRS)
            for got, want in zip(self.host, (wkd, wks, wvd, wvs)):
                assert np.array_equal(got.reshape(want.shape), want)


def run_decode(kv, dev, cache, q, pt, sl, sm_scale, splits=0, status=None, workspace=None):
    B, Hq, D = q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    kv.nvfp4_paged_decode_attention(cache.lay, q.to(dev), cache.kd, cache.ks, cache.gk,
                                    cache.vd, cache.vs, cache.gv, pt.to(dev), sl.to(dev),
                                    sm_scale, out, lse=lse, max_num_splits=splits,
                                    status=status, workspace=workspace)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def oracle_decode(cache, q, pt, sl, sm_scale, want=None):
    kd, ks, vd, vs = cache.host
    return oracle.paged_decode_attention(bits(q), kd, ks, cache.g_k, vd, vs, cache.g_v,
                                         pt.numpy(), sl.numpy(), sm_scale, cache.H, cache.T,
                                         want=want, v_packing=oracle.TOKEN_PAIRS)


def check(out, lse, ref, ref_lse, mask=None, tag=""):
    if mask is not None:
        out, ref, lse, ref_lse = out[mask], ref[mask], lse[mask], ref_lse[mask]
    assert np.all(np.isfinite(out)), tag
    err = np.abs(out - ref)
    over = err - (MAX_ABS + bf16_half_ulp(ref))
    worst = np.unravel_index(np.argmax(over), over.shape)
    assert over.max() <= 0 and err.mean() <= MEAN_ABS, (tag, err.max(), err.mean(), float(ref[worst]),
                                                         float(err[worst]))
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), tag
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= LSE_ABS, tag
    return err


def test_tiny_decode_workload(kv, cuda):
    """1 sequence of 256 tokens, 8 query / 2 KV heads, head_dim 128, 16-token pages, K with
    four x20 outlier channels; also reports the error against BF16 attention."""
    wl = synthetic.tiny_decode()
    q, k, v, pt, sl = wl.make()
    cache = Cache(kv, cuda, k, v, wl.H, wl.D, wl.T)
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, wl.sm_scale)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, wl.sm_scale)
    err = check(out, lse, ref, ref_lse)
    ref_bf16 = oracle.paged_decode_attention_bf16(bits(q), bits(k), bits(v), pt.numpy(),
                                                  sl.numpy(), wl.sm_scale, wl.H, wl.T)
    qerr = np.abs(out - ref_bf16)
    print(f"tiny decode: |gpu-oracle| max {err.max():.2e} mean {err.mean():.2e}; "
          f"|gpu-bf16 attention| max {qerr.max():.2e} mean {qerr.mean():.2e}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("T,G", [(16, 1), (32, 4), (64, 8), (48, 2), (128, 4), (256, 3)])
def test_decode_shapes(kv, cuda, D, T, G):
    """Ragged lengths (partial pages, partial 64-token stages, 1 token, 0 tokens), a shuffled
    pool, several splits."""
    H, B = 2, 5
    lens = [1, 0, 3 * T + 5, 200, 64 * 3]
    maxp = max(-(-L // T) for L in lens)
    pool = B * maxp + 3
    g = synthetic.gen(D * 100 + T * 10 + G)
    q = synthetic.randn_bf16((B, H * G, D), g)
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g)
    perm = torch.randperm(pool, generator=g)[:B * maxp].view(B, maxp).to(torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    cache = Cache(kv, cuda, k, v, H, D, T)
    sm = 1.0 / math.sqrt(D)
    ref, ref_lse = oracle_decode(cache, q, perm, sl, sm)
    for splits in (0, 1, 3):
        out, lse = run_decode(kv, cuda, cache, q, perm, sl, sm, splits=splits)
        check(out, lse, ref, ref_lse, tag=f"splits={splits}")
        assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_split_count_invariance(kv, cuda):
    """The same sequences under 1 .. 64 splits agree with the oracle and with each other."""
    H, G, D, T, B = 2, 4, 128, 64, 3
    lens = [4096, 2500, 64 * 64]
    maxp = max(-(-L // T) for L in lens)
    g = synthetic.gen(77)
    q = synthetic.randn_bf16((B, H * G, D), g)
    pool = B * maxp
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g)
    pt = torch.randperm(pool, generator=g).view(B, maxp).to(torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    cache = Cache(kv, cuda, k, v, H, D, T)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, 1 / math.sqrt(D))
    outs = []
    for splits in (1, 2, 5, 16, 63, 64):
        out, lse = run_decode(kv, cuda, cache, q, pt, sl, 1 / math.sqrt(D), splits=splits)
        check(out, lse, ref, ref_lse, tag=f"splits={splits}")
        outs.append(out)
    # Split counts differ in fp32 summation order and in the running maximum each chunk uses,
    # so P (rounded to FP16, 2^-11 relative) rounds differently: the outputs may differ by one
    # BF16 ulp (2^-7 relative) plus 2^-10 of the largest |v| (two FP16 roundings of P).
    vmax = float(v.float().abs().max())
    bound = np.abs(outs[0]) * 2.0 ** -7 + vmax * 2.0 ** -10
    for o in outs[1:]:
        d = np.abs(o - outs[0])
        assert np.all(d <= bound), (d.max(), float((d - bound).max()))


def test_mha_and_dominant_key(kv, cuda):
    """Group size 1 (MHA) with one key aligned to the query far above the rest: the output is
    that token's decoded value. Outputs here are O(1), where rounding to BF16 alone moves them by
    up to 2^-9 relative, so the check is: within one BF16 ulp of the oracle."""
    H, D, T, B = 4, 128, 16, 1
    L = 50
    g = synthetic.gen(5)
    q = synthetic.randn_bf16((B, H, D), g)
    k = synthetic.kv_pages_bf16(4, H, T, D, g) * 0.05
    v = synthetic.kv_pages_bf16(4, H, T, D, g)
    k[1, :, 7] = q[0].float().mul(4.0).to(torch.bfloat16)   # token 23 of every head
    pt = torch.arange(4, dtype=torch.int32).view(1, 4)
    sl = torch.tensor([L], dtype=torch.int32)
    cache = Cache(kv, cuda, k.to(torch.bfloat16), v, H, D, T)
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, 1.0)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, 1.0)
    assert np.all(np.abs(out - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)
    assert np.abs(lse - ref_lse).max() <= LSE_ABS


def test_decode_batch_workload_sampled(kv, cuda):
    """32 sequences x 8192 tokens, 32 query / 8 KV heads, page 64, pool of 4096 pages under a
    random permutation, in the split configuration the benchmark uses; 96 sampled (sequence,
    head) pairs against the oracle plus properties on every output."""
    wl = synthetic.decode_batch()
    q, k, v, pt, sl = wl.make(device=cuda)
    cache = Cache(kv, cuda, k, v, wl.H, wl.D, wl.T)
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, wl.sm_scale)
    rng = np.random.default_rng(3)
    want = np.zeros((wl.B, wl.Hq), bool)
    want.reshape(-1)[rng.permutation(wl.B * wl.Hq)[:96]] = True
    ref, ref_lse = oracle_decode(cache, q.cpu(), pt.cpu(), sl.cpu(), wl.sm_scale, want=want)
    check(out, lse, ref, ref_lse, mask=want)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    # every output is a convex combination of decoded values: bounded by the V extremes
    vmax = float(v.abs().max()) * 1.1
    assert np.abs(out).max() <= vmax


def test_long_context_workload_sampled(kv, cuda):
    """8 sequences of 32K-128K tokens, 64 query / 8 KV heads, up to 64 splits; 48 sampled
    (sequence, head) pairs against the oracle."""
    wl = synthetic.long_context()
    q, k, v, pt, sl = wl.make(device=cuda)
    cache = Cache(kv, cuda, k, v, wl.H, wl.D, wl.T, verify=False)
    # verify the cache on a sample of pages (the full pool is 2.7 GB of BF16)
    kb = bits(k[:256])
    wkd, wks = oracle.quantize_pages(kb, oracle.BF16, wl.H, wl.D, wl.T, cache.g_k)
    assert np.array_equal(cache.host[0][:256], wkd) and np.array_equal(cache.host[1][:256], wks)
    del k, v
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, wl.sm_scale)
    rng = np.random.default_rng(4)
    want = np.zeros((wl.B, wl.Hq), bool)
    want.reshape(-1)[rng.permutation(wl.B * wl.Hq)[:48]] = True
    ref, ref_lse = oracle_decode(cache, q.cpu(), pt.cpu(), sl.cpu(), wl.sm_scale, want=want)
    check(out, lse, ref, ref_lse, mask=want)
    assert np.all(np.isfinite(out))


def test_bad_page_ids_and_lengths_are_flagged(kv, cuda):
    H, G, D, T, B = 2, 4, 128, 16, 3
    g = synthetic.gen(9)
    q = synthetic.randn_bf16((B, H * G, D), g)
    k = synthetic.kv_pages_bf16(8, H, T, D, g)
    v = synthetic.kv_pages_bf16(8, H, T, D, g)
    cache = Cache(kv, cuda, k, v, H, D, T)
    pt = torch.tensor([[0, 1, 2], [3, 1000, 4], [5, 6, 7]], dtype=torch.int32)
    sl = torch.tensor([40, 40, 49], dtype=torch.int32)   # 49 > 3 pages * 16
    status = torch.zeros(1, dtype=torch.int32, device=cuda)
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, 0.1, status=status)
    st = status.item()
    assert st & kv.STATUS_PAGE_OOB and st & kv.STATUS_BAD_SEQ_LEN
    ref, ref_lse = oracle_decode(cache, q[:1], pt[:1], sl[:1], 0.1)
    check(out[:1], lse[:1], ref, ref_lse)
    assert np.all(np.isfinite(out[1]))                    # the bad page is skipped
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))


@pytest.mark.parametrize("fill", ["0xff", "random"])
def test_workspace_needs_no_clearing(kv, cuda, fill):
    """The decode workspace holds per-pair counters tagged with the call and the split records;
    a workspace full of 0xFF bytes (every counter's tag above any call's) or of random bytes gives
    the oracle's result, bit-identical to a call on a zeroed workspace, for the automatic split
    and for 1, 5 and 64 forced splits. Only host-side writes to the buffer; nothing faults."""
    H, G, D, T, B = 2, 4, 128, 64, 3
    lens = [4096, 2500, 777]
    maxp = max(-(-L // T) for L in lens)
    g = synthetic.gen(31)
    q = synthetic.randn_bf16((B, H * G, D), g)
    pool = B * maxp
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g)
    pt = torch.randperm(pool, generator=g).view(B, maxp).to(torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    cache = Cache(kv, cuda, k, v, H, D, T)
    sm = 1 / math.sqrt(D)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, sm)
    for splits in (0, 1, 5, 64):
        need = kv.nvfp4_paged_decode_workspace_size(cache.lay, B, H * G, maxp, splits)
        ws = torch.empty(need, dtype=torch.uint8, device=cuda)
        if fill == "0xff":
            ws.fill_(0xFF)
        else:
            ws.copy_(torch.randint(0, 256, (need,), dtype=torch.uint8,
                                   generator=synthetic.gen(1000 + splits)))
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        out, lse = run_decode(kv, cuda, cache, q, pt, sl, sm, splits=splits, status=status,
                              workspace=ws)
        check(out, lse, ref, ref_lse, tag=f"{fill} splits={splits}")
        assert status.item() == 0
        ws.zero_()
        out0, lse0 = run_decode(kv, cuda, cache, q, pt, sl, sm, splits=splits, workspace=ws)
        assert np.array_equal(out, out0) and np.array_equal(lse, lse0), (fill, splits)


@pytest.mark.parametrize("H,G", [(8, 4), (4, 1), (2, 3), (3, 4), (1, 2), (2, 8)])
def test_head_dim_64_heads_and_groups(kv, cuda, H, G):
    """Head_dim 64 over even and odd KV-head counts and query groups 1 to 8, against the oracle
    on ragged lengths and a shuffled pool, with the automatic split and with 1 and 7 forced
    splits, and once more with a workspace full of 0xFF bytes."""
    D, T, B = 64, 64, 4
    lens = [3000, 1, 640, 2049]
    maxp = max(-(-L // T) for L in lens)
    pool = B * maxp + 2
    g = synthetic.gen(640 + 10 * H + G)
    q = synthetic.randn_bf16((B, H * G, D), g)
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g)
    pt = torch.randperm(pool, generator=g)[:B * maxp].view(B, maxp).to(torch.int32)
    sl = torch.tensor(lens, dtype=torch.int32)
    cache = Cache(kv, cuda, k, v, H, D, T)
    sm = 1 / math.sqrt(D)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, sm)
    for splits in (0, 1, 7):
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        out, lse = run_decode(kv, cuda, cache, q, pt, sl, sm, splits=splits, status=status)
        check(out, lse, ref, ref_lse, tag=f"H={H} G={G} splits={splits}")
        assert status.item() == 0
    need = kv.nvfp4_paged_decode_workspace_size(cache.lay, B, H * G, maxp, 0)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device=cuda)
    out, lse = run_decode(kv, cuda, cache, q, pt, sl, sm, workspace=ws)
    check(out, lse, ref, ref_lse, tag=f"H={H} G={G} 0xff workspace")


@pytest.mark.parametrize("D", [64, 128, 256])
def test_many_short_sequences(kv, cuda, D):
    """A batch larger than the CTA's threads (each thread of the stage prefix then owns several
    sequences), lengths from 0 to 300 with runs of empty sequences, one KV head: every sequence
    against the oracle, with the automatic split and with 1 and 3 forced splits."""
    H, G, T, B = 1, 2, 16, 1500
    g = synthetic.gen(4000 + D)
    lens = torch.randint(0, 301, (B,), generator=g)
    lens[100:140] = 0                                     # a run of empty sequences
    lens[-7:] = 0                                         # ... and at the end of the batch
    lens = lens.tolist()
    maxp = max(1, max(-(-L // T) for L in lens))
    need = sum(-(-L // T) for L in lens)
    pool = need + 5
    q = synthetic.randn_bf16((B, H * G, D), g)
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g)
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    pt = torch.zeros((B, maxp), dtype=torch.int32)
    off = 0
    for b, L in enumerate(lens):
        n = -(-L // T)
        pt[b, :n] = perm[off:off + n]
        off += n
    sl = torch.tensor(lens, dtype=torch.int32)
    cache = Cache(kv, cuda, k, v, H, D, T)
    sm = 1 / math.sqrt(D)
    ref, ref_lse = oracle_decode(cache, q, pt, sl, sm)
    empty = np.array(lens) == 0
    for splits in (0, 1, 3):
        status = torch.zeros(1, dtype=torch.int32, device=cuda)
        out, lse = run_decode(kv, cuda, cache, q, pt, sl, sm, splits=splits, status=status)
        check(out, lse, ref, ref_lse, tag=f"D={D} splits={splits}")
        assert status.item() == 0
        assert np.all(out[empty] == 0) and np.all(np.isneginf(lse[empty]))
