"""The decode entry point for callers that cannot allocate device memory.

nvfp4_paged_decode_attention_noalloc keeps its split-KV scratch in a fixed array inside the
library instead of a caller workspace, for callers that cannot allocate (a plugin whose host
framework owns every allocation, a server whose free HBM all belongs to its KV pool, a hot path
that must not call cudaMalloc). This file is collected last so that a run stopping at its first
failure has run every other test already; it also passes alone in a fresh process."""
import math

import numpy as np
import pytest
import torch

import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv(cuda):
    from nvfp4_paged_kv_gb300 import build
    build.build()
    import nvfp4_paged_kv_gb300 as m
    m.load()
    return m


def _workload(kv, dev, seed, lens, G=4, H=2, D=128, T=64):
    g = synthetic.gen(seed)
    B = len(lens)
    maxp = max(-(-L // T) for L in lens)
    pool = B * maxp
    q = synthetic.randn_bf16((B, H * G, D), g).to(dev)
    k = synthetic.kv_pages_bf16(pool, H, T, D, g, k_outliers=True).to(dev)
    v = synthetic.kv_pages_bf16(pool, H, T, D, g).to(dev)
    pt = torch.randperm(pool, generator=g).view(B, maxp).to(torch.int32).to(dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    lay = kv.Layout(H, D, T)
    gk = torch.empty(1, dtype=torch.float32, device=dev)
    gv = torch.empty(1, dtype=torch.float32, device=dev)
    kv.nvfp4_kv_compute_global_scale(lay, k, gk)
    kv.nvfp4_kv_compute_global_scale(lay, v, gv)
    mk = lambda w: torch.empty((pool, H, T, w), dtype=torch.uint8, device=dev)  # noqa: E731
    kd, ks, vd, vs = mk(D // 2), mk(D // 16), mk(D // 2), mk(D // 16)
    kv.nvfp4_kv_quantize_pages(lay, k, gk, kd, ks)
    kv.nvfp4_kv_quantize_pages(lay.with_packing(kv.PACK_TOKEN_PAIRS), v, gv, vd, vs)
    return dict(lay=lay, q=q, kd=kd, ks=ks, gk=gk, vd=vd, vs=vs, gv=gv, pt=pt, sl=sl,
                sm=1.0 / math.sqrt(D))


def _run(kv, w, noalloc):
    B, Hq, D = w["q"].shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=w["q"].device)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=w["q"].device)
    fn = kv.nvfp4_paged_decode_attention_noalloc if noalloc else \
        kv.nvfp4_paged_decode_attention
    fn(w["lay"], w["q"], w["kd"], w["ks"], w["gk"], w["vd"], w["vs"], w["gv"], w["pt"],
       w["sl"], w["sm"], out, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_noalloc_decode_matches_workspace_entry_point(kv, cuda):
    """Two calls in a row (different sequences, so the second finds the first's partials in the
    shared scratch) against the workspace entry point on the same inputs. Both run the same
    kernel with the same split plan and merge order, so the outputs and LSEs must be identical
    bit for bit; a stale partial of the first call leaking into the second would show."""
    first = _workload(kv, cuda, seed=21, lens=[5000, 64, 1, 3000])
    second = _workload(kv, cuda, seed=22, lens=[200, 7777, 0])
    for w in (first, second):
        want, want_lse = _run(kv, w, noalloc=False)
        got, got_lse = _run(kv, w, noalloc=True)
        assert np.all(np.isfinite(got))
        assert np.array_equal(got, want)
        assert np.array_equal(got_lse, want_lse)


def test_noalloc_rejects_work_beyond_its_scratch(kv, cuda):
    """A call whose split partials would not fit the fixed scratch is refused before any launch."""
    lay = kv.Layout(8, 128, 64)
    need = kv.nvfp4_paged_decode_workspace_size(lay, 256, 64, 2048, 64)
    assert need > kv.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((256, 64, 128), dtype=torch.bfloat16, device=cuda)
    pages = torch.zeros((1, 8, 64, 64), dtype=torch.uint8, device=cuda)
    scales = torch.zeros((1, 8, 64, 8), dtype=torch.uint8, device=cuda)
    one = torch.ones(1, dtype=torch.float32, device=cuda)
    pt = torch.zeros((256, 2048), dtype=torch.int32, device=cuda)
    sl = torch.zeros(256, dtype=torch.int32, device=cuda)
    out = torch.zeros_like(q)
    with pytest.raises(kv.NVFP4KVError) as e:
        kv.nvfp4_paged_decode_attention_noalloc(lay, q, pages, scales, one, pages, scales, one,
                                                pt, sl, 0.1, out, max_num_splits=64)
    assert e.value.code == 3
