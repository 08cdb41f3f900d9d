"""NVFP4 paged KV cache for GB300: Python binding of ``libnvfp4kv.so``.

Every call here is argument marshalling around the C ABI declared in ``include/nvfp4_kv.h``:
tensors become device pointers, the current torch stream becomes the stream argument, and a
non-OK status becomes an exception. All arithmetic runs in the library's CUDA kernels; there is
no CPU path, and importing a function whose library is not built raises.

PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "Layout", "BF16", "FP16", "FP8_E4M3", "PACK_DIM_PAIRS", "PACK_TOKEN_PAIRS",
    "STATUS_PAGE_OOB", "STATUS_BAD_SEQ_LEN",
    "STATUS_TIMEOUT", "NVFP4KVError", "load", "lib_path", "version",
    "nvfp4_kv_global_scale_workspace_size", "nvfp4_kv_compute_global_scale",
    "nvfp4_kv_quantize_pages", "nvfp4_kv_dequantize_pages", "nvfp4_kv_extend_write",
    "ExtendTensor", "nvfp4_kv_extend_step",
    "nvfp4_paged_decode_workspace_size", "nvfp4_paged_decode_attention", "nvfp4_kv_round_f32",
    "nvfp4_paged_decode_attention_noalloc", "NOALLOC_SCRATCH_BYTES",
    "ColdBlockLayout", "ColdRope", "ROPE_QUANTIZE", "ROPE_SKIP", "ROPE_2FP4",
    "nvfp4_kv_cold_block_layout", "nvfp4_kv_offload_pages",
    "nvfp4_kv_onboard_pages",
]
NOALLOC_SCRATCH_BYTES = 32 << 20   # NVFP4KV_NOALLOC_SCRATCH_BYTES

BF16, FP16, FP8_E4M3 = 0, 1, 2
PACK_DIM_PAIRS, PACK_TOKEN_PAIRS = 0, 1   # nvfp4kv_packing: K pools, V pools of the decode call
STATUS_PAGE_OOB, STATUS_BAD_SEQ_LEN, STATUS_TIMEOUT = 0x1, 0x2, 0x4
_STATUS_NAMES = {1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA"}


class Layout(ctypes.Structure):
    """Geometry and byte packing of one paged K or V tensor (``nvfp4kv_layout``)."""
    _fields_ = [("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("packing", ctypes.c_int32)]

    def __init__(self, num_kv_heads: int, head_dim: int, page_size: int,
                 packing: int = PACK_DIM_PAIRS):
        super().__init__(int(num_kv_heads), int(head_dim), int(page_size), int(packing))

    def with_packing(self, packing: int) -> "Layout":
        return Layout(self.num_kv_heads, self.head_dim, self.page_size, packing)

    def __repr__(self):
        return (f"Layout(num_kv_heads={self.num_kv_heads}, head_dim={self.head_dim}, "
                f"page_size={self.page_size}, packing={self.packing})")


ROPE_QUANTIZE, ROPE_SKIP, ROPE_2FP4 = 0, 1, 2   # nvfp4kv_rope_mode


class ColdRope(ctypes.Structure):
    """The RoPE part of K (head dims [first_dim, first_dim + dims)) and how a cold block keeps
    it (``nvfp4kv_cold_rope``)."""
    _fields_ = [("mode", ctypes.c_int32), ("first_dim", ctypes.c_int32), ("dims", ctypes.c_int32)]

    def __init__(self, mode: int = ROPE_QUANTIZE, first_dim: int = 0, dims: int = 0):
        super().__init__(int(mode), int(first_dim), int(dims))


class ColdBlockLayout(ctypes.Structure):
    """Byte offsets of the parts of one cold block and its size (``nvfp4kv_cold_block_layout``)."""
    _fields_ = [(n, ctypes.c_int64) for n in
                ("k_data", "k_scales", "k_rope", "k_rope_scales", "k_rope2", "k_rope2_scales",
                 "v_data", "v_scales", "extra", "bytes")]

    def __repr__(self):
        return "ColdBlockLayout(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in
                                              self._fields_) + ")"


class ExtendTensor(ctypes.Structure):
    """One tensor (K or V) of an extend step (``nvfp4kv_extend_tensor``)."""
    _fields_ = [("layout", Layout), ("global_scale", ctypes.c_void_p), ("data", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("pool_pages", ctypes.c_int32),
                ("prefix_page_ids", ctypes.c_void_p), ("prefix_pages", ctypes.c_int32),
                ("ws", ctypes.c_void_p), ("ws_pages", ctypes.c_int32),
                ("ws_prefix_ids", ctypes.c_void_p), ("ws_chunk_ids", ctypes.c_void_p),
                ("ws_scale", ctypes.c_void_p), ("chunk_dtype", ctypes.c_int32),
                ("chunk", ctypes.c_void_p), ("chunk_pool_pages", ctypes.c_int32),
                ("chunk_page_ids", ctypes.c_void_p), ("chunk_src_scale", ctypes.c_void_p),
                ("chunk_dst_ids", ctypes.c_void_p), ("chunk_pages", ctypes.c_int32)]


class NVFP4KVError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {code})")
        self.code = code


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load():
    """Load libnvfp4kv.so; raise if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_build.LIB)
        P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        I64 = ctypes.c_int64
        LP = ctypes.POINTER(Layout)
        sigs = {
            "nvfp4kv_status_string": (ctypes.c_char_p, [I32]),
            "nvfp4kv_version": (I32, []),
            "nvfp4_kv_global_scale_workspace_size": (SZ, []),
            "nvfp4_kv_compute_global_scale": (I32, [LP, I32, P, I32, P, I32, P, P, P, SZ, P, P]),
            "nvfp4_kv_quantize_pages": (I32, [LP, I32, P, I32, P, P, P, P, P, I32, P, I32, P, P]),
            "nvfp4_kv_extend_write": (I32, [LP, I32, P, I32, P, P, P, P, P, I32, P, P, I32, P,
                                            P, I32, P, P]),
            "nvfp4_kv_dequantize_pages": (I32, [LP, P, P, I32, P, P, I32, P, I32, P, P, I32, P,
                                                P]),
            "nvfp4_kv_extend_step": (I32, [ctypes.POINTER(ExtendTensor), I32, P, P]),
            "nvfp4_paged_decode_workspace_size": (SZ, [LP, I32, I32, I32, I32]),
            "nvfp4_paged_decode_attention": (I32, [LP, I32, I32, P, P, P, P, P, P, P, I32, P,
                                                   I32, P, F, I32, P, SZ, P, P, P, P]),
            "nvfp4_kv_round_f32": (I32, [P, SZ, I32, P, P]),
            "nvfp4_kv_cold_block_layout": (I32, [LP, P, I32, ctypes.POINTER(ColdBlockLayout)]),
            "nvfp4_kv_offload_pages": (I32, [LP, I32, P, P, I64, I32, P, P, P, P, P, I64, I32,
                                             P, I32, P, I32, P, P]),
            "nvfp4_kv_onboard_pages": (I32, [LP, P, I32, P, P, P, P, I32, P, P, I64, I32, P, P,
                                             I64, I32, I32, P, P]),
            "nvfp4_kv_host_device_pointer": (I32, [P, ctypes.POINTER(ctypes.c_void_p)]),
            "nvfp4_paged_decode_attention_noalloc": (I32, [LP, I32, I32, P, P, P, P, P, P, P,
                                                           I32, P, I32, P, F, I32, P, P, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def version() -> int:
    return load().nvfp4kv_version()


# ------------------------------------------------------------------------------ marshalling

def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t)}")
    if not t.is_cuda:
        raise ValueError("tensors passed to the NVFP4 KV library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the NVFP4 KV library must be contiguous")
    return t.data_ptr()


@contextlib.contextmanager
def _on_device(tensors, stream):
    """Make the device of the call's CUDA tensors current for the library call and yield the
    stream handle to pass: `stream` if given (it must be a stream of that device), else that
    device's current torch stream. The library sizes grids for the current device and launches on
    the given stream, so a call whose tensors live on another GPU than the current one must not
    go out on the current device's stream."""
    devs = {t.device for t in tensors if isinstance(t, torch.Tensor) and t.is_cuda}
    if len(devs) > 1:
        raise ValueError("all CUDA tensors of one call must be on one device, got "
                         + ", ".join(sorted(str(d) for d in devs)))
    dev = devs.pop() if devs else torch.device("cuda", torch.cuda.current_device())
    if isinstance(stream, torch.cuda.Stream) and stream.device != dev:
        raise ValueError(f"stream is on {stream.device} but the tensors are on {dev}")
    with torch.cuda.device(dev):
        if stream is None:
            yield torch.cuda.current_stream(dev).cuda_stream
        elif isinstance(stream, torch.cuda.Stream):
            yield stream.cuda_stream
        else:
            yield int(stream)


def _check(fn: str, code: int):
    if code != 0:
        msg = load().nvfp4kv_status_string(code).decode()
        raise NVFP4KVError(fn, code, msg)


def _dtype_code(t: torch.Tensor, explicit: Optional[int]) -> int:
    if explicit is not None:
        return int(explicit)
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return FP8_E4M3
    raise TypeError(f"unsupported page dtype {t.dtype}")


def _ids(t: Optional[torch.Tensor]):
    if t is not None and t.dtype != torch.int32:
        raise TypeError("page id lists must be int32")
    return _ptr(t)


# ------------------------------------------------------------------------------ entry points

def nvfp4_kv_global_scale_workspace_size() -> int:
    return int(load().nvfp4_kv_global_scale_workspace_size())


def nvfp4_kv_compute_global_scale(layout: Layout, src: torch.Tensor, out: torch.Tensor, *,
                                  src_dtype=None, src_page_ids=None, num_pages=None,
                                  src_scale=None, workspace=None, status=None, stream=None):
    """out[0] = fp32(amax / 2688) over the listed pages of `src` ([pool, H, T, D])."""
    lib = load()
    if num_pages is None:
        num_pages = src_page_ids.numel() if src_page_ids is not None else src.shape[0]
    if workspace is None:
        workspace = torch.empty(nvfp4_kv_global_scale_workspace_size(), dtype=torch.uint8,
                                device=src.device)
    with _on_device((src, out, src_page_ids, src_scale, workspace, status), stream) as s:
        code = lib.nvfp4_kv_compute_global_scale(
            ctypes.byref(layout), _dtype_code(src, src_dtype), _ptr(src), src.shape[0],
            _ids(src_page_ids), int(num_pages), _ptr(src_scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(status), s)
    _check("nvfp4_kv_compute_global_scale", code)
    return out


def nvfp4_kv_quantize_pages(layout: Layout, src: torch.Tensor, global_scale: torch.Tensor,
                            dst_data: torch.Tensor, dst_scales: torch.Tensor, *,
                            src_dtype=None, src_page_ids=None, dst_page_ids=None,
                            num_pages=None, src_scale=None, status=None, stream=None):
    """Encode pages of `src` into the NVFP4 pools (dst_data [pool,H,T,D/2] u8,
    dst_scales [pool,H,T,D/16] u8)."""
    lib = load()
    if num_pages is None:
        num_pages = src_page_ids.numel() if src_page_ids is not None else src.shape[0]
    with _on_device((src, global_scale, dst_data, dst_scales, src_page_ids, dst_page_ids,
                     src_scale, status), stream) as s:
        code = lib.nvfp4_kv_quantize_pages(
            ctypes.byref(layout), _dtype_code(src, src_dtype), _ptr(src), src.shape[0],
            _ids(src_page_ids), _ptr(src_scale), _ptr(global_scale), _ptr(dst_data),
            _ptr(dst_scales), dst_data.shape[0], _ids(dst_page_ids), int(num_pages), _ptr(status),
            s)
    _check("nvfp4_kv_quantize_pages", code)


def nvfp4_kv_extend_write(layout: Layout, src: torch.Tensor, global_scale: torch.Tensor,
                          dst_data: torch.Tensor, dst_scales: torch.Tensor, ws_fp8: torch.Tensor,
                          *, src_dtype=None, src_page_ids=None, src_scale=None,
                          dst_page_ids=None, ws_page_ids=None, ws_scale=None, num_pages=None,
                          status=None, stream=None):
    """One pass over the chunk's pages `src` (BF16 / FP16, or FP8 E4M3 bytes read as
    e4m3 * src_scale): NVFP4 pages into (dst_data, dst_scales) and the FP8 E4M3 workspace copy
    into `ws_fp8` ([pool, H, T, D] uint8)."""
    lib = load()
    if num_pages is None:
        num_pages = src_page_ids.numel() if src_page_ids is not None else src.shape[0]
    with _on_device((src, global_scale, dst_data, dst_scales, ws_fp8, src_page_ids, dst_page_ids,
                     ws_page_ids, src_scale, ws_scale, status), stream) as s:
        code = lib.nvfp4_kv_extend_write(
            ctypes.byref(layout), _dtype_code(src, src_dtype), _ptr(src), src.shape[0],
            _ids(src_page_ids), _ptr(src_scale), _ptr(global_scale), _ptr(dst_data),
            _ptr(dst_scales), dst_data.shape[0], _ids(dst_page_ids), _ptr(ws_fp8), ws_fp8.shape[0],
            _ids(ws_page_ids), _ptr(ws_scale), int(num_pages), _ptr(status), s)
    _check("nvfp4_kv_extend_write", code)


def nvfp4_kv_extend_step(parts, *, status=None, stream=None):
    """The extend step of one or two tensors (K, V) in one launch. Each part is a dict with
    layout, global_scale, data, scales (the NVFP4 pool), prefix_page_ids, ws (FP8 workspace
    [pages, H, T, D] uint8), ws_prefix_ids, ws_chunk_ids, chunk (chunk pages), chunk_dst_ids,
    and optionally ws_scale, chunk_page_ids, chunk_src_scale, chunk_dtype. Equals
    nvfp4_kv_dequantize_pages (prefix -> FP8 workspace) plus nvfp4_kv_extend_write (chunk) for
    every part, byte for byte."""
    lib = load()
    arr = (ExtendTensor * len(parts))()
    tensors = []
    for x, d in zip(arr, parts):
        chunk = d["chunk"]
        x.layout = d["layout"]
        x.global_scale = _ptr(d["global_scale"])
        x.data, x.scales = _ptr(d["data"]), _ptr(d["scales"])
        x.pool_pages = d["data"].shape[0]
        x.prefix_page_ids = _ids(d.get("prefix_page_ids"))
        x.prefix_pages = (d["prefix_page_ids"].numel() if d.get("prefix_page_ids") is not None
                          else int(d.get("prefix_pages", 0)))
        x.ws, x.ws_pages = _ptr(d["ws"]), d["ws"].shape[0]
        x.ws_prefix_ids = _ids(d.get("ws_prefix_ids"))
        x.ws_chunk_ids = _ids(d.get("ws_chunk_ids"))
        x.ws_scale = _ptr(d.get("ws_scale"))
        x.chunk_dtype = _dtype_code(chunk, d.get("chunk_dtype"))
        x.chunk, x.chunk_pool_pages = _ptr(chunk), chunk.shape[0]
        x.chunk_page_ids = _ids(d.get("chunk_page_ids"))
        x.chunk_src_scale = _ptr(d.get("chunk_src_scale"))
        x.chunk_dst_ids = _ids(d.get("chunk_dst_ids"))
        x.chunk_pages = (d["chunk_dst_ids"].numel() if d.get("chunk_dst_ids") is not None
                         else chunk.shape[0])
        tensors += [d[k] for k in ("global_scale", "data", "scales", "ws", "chunk")
                    if d.get(k) is not None]
        tensors += [d[k] for k in ("prefix_page_ids", "ws_prefix_ids", "ws_chunk_ids",
                                   "ws_scale", "chunk_page_ids", "chunk_src_scale",
                                   "chunk_dst_ids") if d.get(k) is not None]
    with _on_device(tensors + [status], stream) as s:
        code = lib.nvfp4_kv_extend_step(arr, len(parts), _ptr(status), s)
    _check("nvfp4_kv_extend_step", code)


def nvfp4_kv_dequantize_pages(layout: Layout, src_data: torch.Tensor, src_scales: torch.Tensor,
                              global_scale: torch.Tensor, dst: torch.Tensor, *, dst_dtype=None,
                              src_page_ids=None, dst_page_ids=None, num_pages=None,
                              dst_scale=None, status=None, stream=None):
    """Decode NVFP4 pages into `dst` ([pool, H, T, D] of BF16 / FP16 / FP8 E4M3)."""
    lib = load()
    if num_pages is None:
        num_pages = src_page_ids.numel() if src_page_ids is not None else src_data.shape[0]
    with _on_device((src_data, src_scales, global_scale, dst, src_page_ids, dst_page_ids,
                     dst_scale, status), stream) as s:
        code = lib.nvfp4_kv_dequantize_pages(
            ctypes.byref(layout), _ptr(src_data), _ptr(src_scales), src_data.shape[0],
            _ids(src_page_ids), _ptr(global_scale), _dtype_code(dst, dst_dtype), _ptr(dst),
            dst.shape[0], _ids(dst_page_ids), _ptr(dst_scale), int(num_pages), _ptr(status),
            s)
    _check("nvfp4_kv_dequantize_pages", code)


def nvfp4_paged_decode_workspace_size(layout: Layout, batch: int, num_q_heads: int,
                                      max_pages_per_seq: int, max_num_splits: int = 0) -> int:
    return int(load().nvfp4_paged_decode_workspace_size(
        ctypes.byref(layout), int(batch), int(num_q_heads), int(max_pages_per_seq),
        int(max_num_splits)))


def nvfp4_paged_decode_attention(layout: Layout, q: torch.Tensor, k_data, k_scales,
                                 k_global_scale, v_data, v_scales, v_global_scale,
                                 page_table: torch.Tensor, seq_lens: torch.Tensor,
                                 sm_scale: float, out: torch.Tensor, *, lse=None,
                                 max_num_splits: int = 0, workspace=None, status=None,
                                 stream=None):
    """out[b, qh] = softmax(sm_scale q.K^T) V over the sequence's NVFP4 pages (BF16)."""
    lib = load()
    B, Hq, _ = q.shape
    maxp = page_table.shape[1]
    if workspace is None:
        need = nvfp4_paged_decode_workspace_size(layout, B, Hq, maxp, max_num_splits)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("page_table and seq_lens must be int32")
    with _on_device((q, k_data, k_scales, k_global_scale, v_data, v_scales, v_global_scale,
                     page_table, seq_lens, out, lse, workspace, status), stream) as s:
        code = lib.nvfp4_paged_decode_attention(
            ctypes.byref(layout), B, Hq, _ptr(q), _ptr(k_data), _ptr(k_scales),
            _ptr(k_global_scale), _ptr(v_data), _ptr(v_scales), _ptr(v_global_scale),
            k_data.shape[0], _ptr(page_table), maxp, _ptr(seq_lens), float(sm_scale),
            int(max_num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(out), _ptr(lse), _ptr(status), s)
    _check("nvfp4_paged_decode_attention", code)
    return out


def nvfp4_paged_decode_attention_noalloc(layout: Layout, q: torch.Tensor, k_data, k_scales,
                                         k_global_scale, v_data, v_scales, v_global_scale,
                                         page_table: torch.Tensor, seq_lens: torch.Tensor,
                                         sm_scale: float, out: torch.Tensor, *, lse=None,
                                         max_num_splits: int = 0, status=None, stream=None):
    """The decode attention for callers that cannot allocate: no workspace argument, the split
    partials use the library's fixed NOALLOC_SCRATCH_BYTES device array. Calls that overlap on
    the GPU race on that array; the first call on a device must precede any stream capture."""
    lib = load()
    B, Hq, _ = q.shape
    if page_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("page_table and seq_lens must be int32")
    with _on_device((q, k_data, k_scales, k_global_scale, v_data, v_scales, v_global_scale,
                     page_table, seq_lens, out, lse, status), stream) as s:
        code = lib.nvfp4_paged_decode_attention_noalloc(
            ctypes.byref(layout), B, Hq, _ptr(q), _ptr(k_data), _ptr(k_scales),
            _ptr(k_global_scale), _ptr(v_data), _ptr(v_scales), _ptr(v_global_scale),
            k_data.shape[0], _ptr(page_table), page_table.shape[1], _ptr(seq_lens),
            float(sm_scale), int(max_num_splits), _ptr(out), _ptr(lse), _ptr(status),
            s)
    _check("nvfp4_paged_decode_attention_noalloc", code)
    return out


def nvfp4_kv_round_f32(x: torch.Tensor, target: int, out: torch.Tensor, stream=None):
    """target 0: E2M1 codes, target 1: E4M3 bytes, of fp32 inputs (one byte each)."""
    with _on_device((x, out), stream) as s:
        code = load().nvfp4_kv_round_f32(_ptr(x), x.numel(), int(target), _ptr(out),
                                         s)
    _check("nvfp4_kv_round_f32", code)


# ------------------------------------------------------------------------------ cold pages

def _rope_ref(rope):
    return None if rope is None else ctypes.byref(rope)


def nvfp4_kv_cold_block_layout(layout: Layout, extra_bytes: int = 0,
                               rope: Optional[ColdRope] = None) -> ColdBlockLayout:
    """Offsets and size of one cold block for `layout` with `extra_bytes` lossless bytes and
    the RoPE option `rope` (None: the RoPE part is quantized like the rest)."""
    out = ColdBlockLayout()
    _check("nvfp4_kv_cold_block_layout",
           load().nvfp4_kv_cold_block_layout(ctypes.byref(layout), _rope_ref(rope),
                                             int(extra_bytes), ctypes.byref(out)))
    return out


def _paged_ptr(t: torch.Tensor):
    """Pointer and page stride (elements) of a [pages, ...] CUDA tensor whose pages are each
    contiguous (pages may be strided, e.g. the K or V half of one combined pool)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("hot pools must be CUDA tensors")
    if not t[0].is_contiguous():
        raise ValueError("each page of a hot pool must be contiguous")
    return t.data_ptr(), t.stride(0)


def _cold_ptr(t: torch.Tensor):
    """Device address of a cold pool: a CUDA tensor, or pinned host memory (its device alias)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"expected a torch.Tensor, got {type(t)}")
    if not t.is_contiguous():
        raise ValueError("the cold pool must be contiguous")
    if t.is_cuda:
        return t.data_ptr()
    if not t.is_pinned():
        raise ValueError("a host cold pool must be pinned memory")
    dev = ctypes.c_void_p()
    _check("nvfp4_kv_host_device_pointer",
           load().nvfp4_kv_host_device_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(dev)))
    return dev.value


def _extra_args(extra, extra_bytes):
    if extra is None or extra_bytes == 0:
        return None, 0, 0
    if not extra.is_cuda or not extra[0].is_contiguous():
        raise ValueError("extra must be a CUDA tensor [pages, bytes] with contiguous rows")
    return extra.data_ptr(), extra.stride(0) * extra.element_size(), int(extra_bytes)


def nvfp4_kv_offload_pages(layout: Layout, hot_k: torch.Tensor, hot_v: torch.Tensor,
                           cold: torch.Tensor, *, k_global_scale=None, v_global_scale=None,
                           hot_page_ids=None, cold_slot_ids=None, extra=None, extra_bytes=0,
                           rope: Optional[ColdRope] = None, num_pages=None, hot_dtype=None,
                           status=None, stream=None):
    """Quantize hot pages (BF16 / FP16 [pages, H, T, D]) into cold blocks of `cold`
    ([slots, block bytes] uint8, device or pinned host memory) in one pass."""
    lib = load()
    bl = nvfp4_kv_cold_block_layout(layout, extra_bytes, rope)
    kp, ks = _paged_ptr(hot_k)
    vp, vs = _paged_ptr(hot_v)
    if ks != vs:
        raise ValueError("hot_k and hot_v must have the same page stride")
    if num_pages is None:
        num_pages = hot_page_ids.numel() if hot_page_ids is not None else hot_k.shape[0]
    ep, es, eb = _extra_args(extra, extra_bytes)
    with _on_device((hot_k, hot_v, cold, k_global_scale, v_global_scale, hot_page_ids,
                     cold_slot_ids, extra, status), stream) as s:
        code = lib.nvfp4_kv_offload_pages(
            ctypes.byref(layout), _dtype_code(hot_k, hot_dtype), kp, vp, ks, hot_k.shape[0],
            _ids(hot_page_ids), _ptr(k_global_scale), _ptr(v_global_scale), _rope_ref(rope), ep, es,
            eb, _cold_ptr(cold), cold.numel() // bl.bytes, _ids(cold_slot_ids), int(num_pages),
            _ptr(status), s)
    _check("nvfp4_kv_offload_pages", code)


def nvfp4_kv_onboard_pages(layout: Layout, cold: torch.Tensor, hot_k: torch.Tensor,
                           hot_v: torch.Tensor, *, k_global_scale=None, v_global_scale=None,
                           cold_slot_ids=None, hot_page_ids=None, extra=None, extra_bytes=0,
                           rope: Optional[ColdRope] = None, num_pages=None, hot_dtype=None,
                           status=None, stream=None):
    """Dequantize cold blocks of `cold` into hot pages (BF16 / FP16) in one pass."""
    lib = load()
    bl = nvfp4_kv_cold_block_layout(layout, extra_bytes, rope)
    kp, ks = _paged_ptr(hot_k)
    vp, vs = _paged_ptr(hot_v)
    if ks != vs:
        raise ValueError("hot_k and hot_v must have the same page stride")
    if num_pages is None:
        num_pages = cold_slot_ids.numel() if cold_slot_ids is not None else cold.numel() // bl.bytes
    ep, es, eb = _extra_args(extra, extra_bytes)
    with _on_device((cold, hot_k, hot_v, k_global_scale, v_global_scale, cold_slot_ids,
                     hot_page_ids, extra, status), stream) as s:
        code = lib.nvfp4_kv_onboard_pages(
            ctypes.byref(layout), _cold_ptr(cold), cold.numel() // bl.bytes, _ids(cold_slot_ids),
            _ptr(k_global_scale), _ptr(v_global_scale), _rope_ref(rope),
            _dtype_code(hot_k, hot_dtype), kp, vp, ks,
            hot_k.shape[0], _ids(hot_page_ids), ep, es, eb, int(num_pages), _ptr(status),
            s)
    _check("nvfp4_kv_onboard_pages", code)

