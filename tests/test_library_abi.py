"""The C ABI library on the host: it builds, loads, exports every function the header declares,
and rejects invalid arguments before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4_kv.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_paged_kv_gb300 import build
    build.build()
    import nvfp4_paged_kv_gb300 as kv
    return kv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(nvfp4\w*)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("nvfp4_kv_quantize_pages", "nvfp4_kv_dequantize_pages", "nvfp4_kv_extend_write",
                 "nvfp4_kv_cold_block_layout", "nvfp4_kv_offload_pages", "nvfp4_kv_onboard_pages",
                 "nvfp4_kv_host_device_pointer",
                 "nvfp4_paged_decode_attention", "nvfp4_paged_decode_workspace_size",
                 "nvfp4_kv_compute_global_scale", "nvfp4_kv_global_scale_workspace_size",
                 "nvfp4_kv_round_f32", "nvfp4kv_status_string", "nvfp4kv_version",
                 "nvfp4_kv_extend_step", "nvfp4_paged_decode_attention_noalloc"):
        assert want in names


def test_library_exports_every_declared_function(lib):
    import subprocess
    from nvfp4_paged_kv_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings_and_version(lib):
    for code in range(5):
        assert lib.nvfp4kv_status_string(code).decode().startswith("NVFP4KV_")
    assert lib.nvfp4kv_version() >= 100


def test_host_validation_rejects_bad_arguments(lib):
    import nvfp4_paged_kv_gb300 as kv
    good = kv.Layout(8, 128, 64)
    bad_d = kv.Layout(8, 120, 64)
    fake = ctypes.c_void_p(4096)       # never dereferenced: validation fails first
    mis = ctypes.c_void_p(4096 + 8)    # misaligned
    q = lib.nvfp4_kv_quantize_pages
    # head_dim not a multiple of 16
    assert q(ctypes.byref(bad_d), 0, fake, 1, None, None, fake, fake, fake, 1, None, 1, None,
             None) == 1
    # null destination
    assert q(ctypes.byref(good), 0, fake, 1, None, None, fake, None, fake, 1, None, 1, None,
             None) == 1
    # misaligned source
    assert q(ctypes.byref(good), 0, mis, 1, None, None, fake, fake, fake, 1, None, 1, None,
             None) == 1
    # pool smaller than the page count without id lists
    assert q(ctypes.byref(good), 0, fake, 1, None, None, fake, fake, fake, 1, None, 2, None,
             None) == 1
    # bad dtype
    assert q(ctypes.byref(good), 7, fake, 1, None, None, fake, fake, fake, 1, None, 1, None,
             None) == 1
    # zero pages is a no-op
    assert q(ctypes.byref(good), 0, None, 0, None, None, None, None, None, 0, None, 0, None,
             None) == 0
    dq = lib.nvfp4_kv_dequantize_pages
    assert dq(ctypes.byref(good), fake, fake, 1, None, fake, 9, fake, 1, None, None, 1, None,
              None) == 1
    xw = lib.nvfp4_kv_extend_write
    # unknown source dtype
    assert xw(ctypes.byref(good), 7, fake, 1, None, None, fake, fake, fake, 1, None, fake, 1,
              None, None, 1, None, None) == 2
    # missing workspace; misaligned workspace; zero pages is a no-op
    assert xw(ctypes.byref(good), 0, fake, 1, None, None, fake, fake, fake, 1, None, None, 1,
              None, None, 1, None, None) == 1
    assert xw(ctypes.byref(good), 2, fake, 1, None, None, fake, fake, fake, 1, None, mis, 1,
              None, None, 1, None, None) == 1
    assert xw(ctypes.byref(good), 0, None, 0, None, None, None, None, None, 0, None, None, 0,
              None, None, 0, None, None) == 0
    off = lib.nvfp4_kv_offload_pages
    hot_stride = 8 * 64 * 128
    # FP8 hot pool: unsupported; null cold pool; misaligned hot pool; page stride below a page;
    # extra bytes without an extra pointer; a malformed RoPE option; zero pages is a no-op
    assert off(ctypes.byref(good), 2, fake, fake, hot_stride, 1, None, None, None, None, None, 0,
               0, fake, 1, None, 1, None, None) == 2
    assert off(ctypes.byref(good), 0, fake, fake, hot_stride, 1, None, None, None, None, None, 0,
               0, None, 1, None, 1, None, None) == 1
    assert off(ctypes.byref(good), 0, mis, fake, hot_stride, 1, None, None, None, None, None, 0,
               0, fake, 1, None, 1, None, None) == 1
    assert off(ctypes.byref(good), 0, fake, fake, hot_stride - 8, 1, None, None, None, None,
               None, 0, 0, fake, 1, None, 1, None, None) == 1
    assert off(ctypes.byref(good), 0, fake, fake, hot_stride, 1, None, None, None, None, None,
               16, 16, fake, 1, None, 1, None, None) == 1
    for bad in (kv.ColdRope(kv.ROPE_SKIP, 8, 64), kv.ColdRope(kv.ROPE_2FP4, 96, 64),
                kv.ColdRope(kv.ROPE_SKIP, 0, 0), kv.ColdRope(7, 0, 16)):
        assert off(ctypes.byref(good), 0, fake, fake, hot_stride, 1, None, None, None,
                   ctypes.byref(bad), None, 0, 0, fake, 1, None, 1, None, None) == 1
    assert off(ctypes.byref(good), 0, None, None, 0, 0, None, None, None, None, None, 0, 0,
               None, 0, None, 0, None, None) == 0
    on = lib.nvfp4_kv_onboard_pages
    assert on(ctypes.byref(good), None, 1, None, None, None, None, 0, fake, fake, hot_stride, 1,
              None, None, 0, 0, 1, None, None) == 1
    assert on(ctypes.byref(good), fake, 1, None, None, None, None, 2, fake, fake, hot_stride, 1,
              None, None, 0, 0, 1, None, None) == 2
    att = lib.nvfp4_paged_decode_attention
    args = [ctypes.byref(good), 2, 32, fake, fake, fake, fake, fake, fake, fake, 10, fake, 4,
            fake, 0.1, 0, fake, 1 << 20, fake, None, None, None]
    # unsupported head_dim for decode (96), GQA group > 8, split count > 64
    a = list(args)
    a[0] = ctypes.byref(kv.Layout(8, 96, 64))
    assert att(*a) == 2
    a = list(args)
    a[2] = 8 * 16
    assert att(*a) == 2
    a = list(args)
    a[15] = 65
    assert att(*a) == 1
    # workspace too small
    a = list(args)
    a[17] = 16
    assert att(*a) == 3


def test_workspace_sizes(lib):
    import nvfp4_paged_kv_gb300 as kv
    lay = kv.Layout(8, 128, 64)
    assert kv.nvfp4_kv_global_scale_workspace_size() >= 4
    # one split: B * Hq * (D + 2) floats, each region 256-byte aligned
    n1 = kv.nvfp4_paged_decode_workspace_size(lay, 4, 32, 1, 1)
    assert n1 >= 4 * 32 * (128 + 2) * 4
    n64 = kv.nvfp4_paged_decode_workspace_size(lay, 4, 32, 4096, 64)
    assert n64 >= 64 * 4 * 32 * (128 + 2) * 4
    assert kv.nvfp4_paged_decode_workspace_size(lay, 4, 32, 4096, 65) == 0


def test_cold_block_layout_matches_its_definition(lib):
    """The library's cold block offsets equal the oracle's, written from the same definition
    (K codes, K scales, the RoPE part as its mode keeps it, V codes, V scales, extra, each part
    at the previous end rounded up to 16), including shapes that need padding; a bad extra size
    or RoPE option is rejected."""
    import nvfp4_paged_kv_gb300 as kv
    import oracle
    fields = ("k_data", "k_scales", "k_rope", "k_rope_scales", "k_rope2", "k_rope2_scales",
              "v_data", "v_scales", "extra", "bytes")
    for H, D, T, extra in ((8, 128, 32, 0), (8, 128, 64, 4096), (1, 16, 1, 32), (3, 80, 5, 16)):
        for rope in (None, (kv.ROPE_SKIP, 0, 16), (kv.ROPE_2FP4, D - 16, 16),
                     (kv.ROPE_2FP4, 0, D), (kv.ROPE_QUANTIZE, 0, 0)):
            cr = None if rope is None else kv.ColdRope(*rope)
            bl = kv.nvfp4_kv_cold_block_layout(kv.Layout(H, D, T), extra, cr)
            ref = oracle.cold_block_layout(H, D, T, extra, rope)
            assert [getattr(bl, f) for f in fields] == [ref[f] for f in fields], (H, D, T, rope)
    out = kv.ColdBlockLayout()
    assert lib.nvfp4_kv_cold_block_layout(ctypes.byref(kv.Layout(8, 128, 32)), None, 8,
                                          ctypes.byref(out)) == 1
    assert lib.nvfp4_kv_cold_block_layout(ctypes.byref(kv.Layout(8, 120, 32)), None, 0,
                                          ctypes.byref(out)) == 1
    bad = kv.ColdRope(kv.ROPE_SKIP, 120, 16)
    assert lib.nvfp4_kv_cold_block_layout(ctypes.byref(kv.Layout(8, 128, 32)),
                                          ctypes.byref(bad), 0, ctypes.byref(out)) == 1


def test_extend_step_host_validation(lib):
    """The one-launch extend step checks every tensor as the separate calls do, on the host,
    before any launch: no tensor list, a tensor count other than 1 or 2, a missing pool or
    workspace, chunks of different dtypes. The pointers below are never dereferenced."""
    import nvfp4_paged_kv_gb300 as kv
    fake = ctypes.c_void_p(1 << 20)   # 16-byte aligned address, never touched
    def tensor(**kw):
        x = kv.ExtendTensor()
        x.layout = kv.Layout(8, 128, 64)
        x.global_scale = fake
        x.data = x.scales = x.ws = x.chunk = fake
        x.pool_pages = x.ws_pages = x.chunk_pool_pages = 4
        x.prefix_pages = 2
        x.chunk_pages = 1
        x.chunk_dtype = kv.BF16
        for k, v in kw.items():
            setattr(x, k, v)
        return x
    call = lib.nvfp4_kv_extend_step
    arr = (kv.ExtendTensor * 2)(tensor(), tensor())
    assert call(None, 1, None, None) == 1
    assert call(arr, 0, None, None) == 1
    assert call(arr, 3, None, None) == 1
    assert call((kv.ExtendTensor * 1)(tensor(data=None)), 1, None, None) == 1
    assert call((kv.ExtendTensor * 1)(tensor(ws=None)), 1, None, None) == 1
    assert call((kv.ExtendTensor * 1)(tensor(layout=kv.Layout(8, 120, 64))), 1, None, None) == 1
    assert call((kv.ExtendTensor * 1)(tensor(chunk_dtype=7)), 1, None, None) == 2
    mixed = (kv.ExtendTensor * 2)(tensor(), tensor(chunk_dtype=kv.FP16))
    assert call(mixed, 2, None, None) == 2
    empty = (kv.ExtendTensor * 1)(tensor(prefix_pages=0, chunk_pages=0))
    assert call(empty, 1, None, None) == 0
