"""CPU oracle for NVFP4 paged KV -- test infrastructure only.

Thin ctypes wrapper over ``nvfp4_oracle.c`` (plain C99, fp64). Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the GPU library never
does, and the two share no code. See ``nvfp4_oracle.c`` for the arithmetic convention and
the readings taken where the source pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_SAN_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_asan_ubsan.so")

BF16, FP16, FP8_E4M3 = 0, 1, 2
DIM_PAIRS, TOKEN_PAIRS = 0, 1   # byte packing of an NVFP4 pool (see nvfp4_oracle.c, R2)

_lock = threading.Lock()
_lib = None


def build(force: bool = False, sanitize: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add, OpenMP over pages / heads).

    sanitize=True builds a second copy instrumented with AddressSanitizer and
    UndefinedBehaviorSanitizer (any finding aborts the process); a process loads it instead of
    the plain build when NVFP4_ORACLE_LIB names it, and must then preload gcc's libasan."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    path = _SAN_LIB_PATH if sanitize else _LIB_PATH
    if (not force and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    compile_to(_SRC, tmp, sanitize=sanitize)
    os.replace(tmp, path)
    return path


def compile_to(src: str, out: str, sanitize: bool = False) -> str:
    """Compile an oracle C source (this one, or a copy with a deliberate mistake planted by the
    tests that check the pins catch it) to the shared library `out`, with the oracle's flags."""
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-Wall", "-shared", "-fPIC", src, "-o", out, "-lm"]
    if sanitize:
        cmd[1:1] = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                    "-fno-omit-frame-pointer", "-g"]
    subprocess.run(cmd, check=True)
    return out


def bind(path: str):
    """The oracle library at `path` with the argument types of every exported function."""
    lib = ctypes.CDLL(path)
    d, i, p, sz = ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "orc_max_threads": (i, []),
        "orc_set_threads": (None, [i]),
        "orc_round_to_format": (d, [d, i, i]),
        "orc_fp32": (d, [d]),
        "orc_bf16_round": (d, [d]),
        "orc_fp16_round": (d, [d]),
        "orc_e2m1_value": (d, [i]),
        "orc_e2m1_encode": (i, [d]),
        "orc_e4m3_value": (d, [i]),
        "orc_e4m3_encode": (i, [d]),
        "orc_bf16_value": (d, [i]),
        "orc_bf16_bits": (i, [d]),
        "orc_fp16_value": (d, [i]),
        "orc_fp16_bits": (i, [d]),
        "orc_e2m1_encode_f32": (None, [p, sz, p]),
        "orc_e4m3_encode_f32": (None, [p, sz, p]),
        "orc_tensor_amax": (d, [i, i, i, i, p, p, i, d]),
        "orc_global_scale_from_amax": (d, [d]),
        "orc_quantize_pages": (None, [i, i, i, i, i, p, p, d, d, p, p, p, i]),
        "orc_cast_fp8_pages": (None, [i, i, i, i, p, p, d, d, p, p, i]),
        "orc_encode_2fp4_blocks": (None, [i, i, p, d, p, p, p, p]),
        "orc_decode_2fp4_blocks": (None, [i, p, p, p, p, d, i, p]),
        "orc_dequantize_pages": (None, [i, i, i, i, p, p, p, d, i, p, p, d, i]),
        "orc_paged_decode_attention": (None, [i, i, i, i, i, i, i, p, p, p, d, p, p, d,
                                              p, i, p, d, p, p, p]),
        "orc_paged_decode_attention_bf16": (None, [i, i, i, i, i, p, p, p, p, i, p,
                                                   d, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = bind(os.environ.get("NVFP4_ORACLE_LIB") or build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _ids(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


# ---------------------------------------------------------------- scalar conversions

def max_threads() -> int:
    return _load().orc_max_threads()


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def round_to_format(y: float, p: int, emin: int) -> float:
    return _load().orc_round_to_format(float(y), int(p), int(emin))


def fp32(y: float) -> float:
    return _load().orc_fp32(float(y))


def bf16_round(y: float) -> float:
    return _load().orc_bf16_round(float(y))


def fp16_round(y: float) -> float:
    return _load().orc_fp16_round(float(y))


def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e2m1_encode(y: float) -> int:
    return _load().orc_e2m1_encode(float(y))


def e4m3_value(b: int) -> float:
    return _load().orc_e4m3_value(int(b))


def e4m3_encode(y: float) -> int:
    return _load().orc_e4m3_encode(float(y))


def bf16_value(h: int) -> float:
    return _load().orc_bf16_value(int(h))


def bf16_bits(v: float) -> int:
    return _load().orc_bf16_bits(float(v))


def fp16_value(h: int) -> float:
    return _load().orc_fp16_value(int(h))


def fp16_bits(v: float) -> int:
    return _load().orc_fp16_bits(float(v))


def e2m1_encode_f32(x: np.ndarray) -> np.ndarray:
    """E2M1 codes (RNE, satfinite, sign kept) of finite fp32 values, one per byte."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_e2m1_encode_f32(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_encode_f32(x: np.ndarray) -> np.ndarray:
    """E4M3 bytes (RNE, satfinite at 448, sign kept) of finite fp32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().orc_e4m3_encode_f32(_ptr(x), x.size, _ptr(out))
    return out


# ---------------------------------------------------------------- page codec

def _src_dtype(src: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint8 if dtype == FP8_E4M3 else np.uint16
    src = np.ascontiguousarray(src)
    if src.dtype != want:
        raise TypeError(f"source bit patterns must be {want}, got {src.dtype}")
    return src


def tensor_amax(src, dtype, H, D, T, src_page_ids=None, num_pages=None, src_scale=1.0):
    src = _src_dtype(src, dtype)
    ids = _ids(src_page_ids)
    n = len(ids) if ids is not None else (num_pages if num_pages is not None
                                         else src.size // (H * T * D))
    return _load().orc_tensor_amax(H, D, T, dtype, _ptr(src), _ptr(ids), n, float(src_scale))


def global_scale(src, dtype, H, D, T, src_page_ids=None, num_pages=None, src_scale=1.0):
    """g = fp32(amax / 2688), or 1.0 when that is zero."""
    amax = tensor_amax(src, dtype, H, D, T, src_page_ids, num_pages, src_scale)
    return _load().orc_global_scale_from_amax(amax)


def pool_shapes(P, H, T, D, packing=DIM_PAIRS):
    """numpy shapes of the packed-code and scale pools of P pages."""
    if packing == TOKEN_PAIRS:
        return (P, H, T // 2, D), (P, H, T // 2, D // 16, 2)
    return (P, H, T, D // 2), (P, H, T, D // 16)


def quantize_pages(src, dtype, H, D, T, g, num_dst_pages=None, src_page_ids=None,
                   dst_page_ids=None, num_pages=None, src_scale=1.0, packing=DIM_PAIRS):
    """Encode pages to NVFP4. Returns (data, scales) shaped as pool_shapes(...) says."""
    src = _src_dtype(src, dtype)
    sids, dids = _ids(src_page_ids), _ids(dst_page_ids)
    if num_pages is None:
        num_pages = len(sids) if sids is not None else src.size // (H * T * D)
    if num_dst_pages is None:
        num_dst_pages = int(dids.max()) + 1 if dids is not None and len(dids) else num_pages
    ds, ss = pool_shapes(num_dst_pages, H, T, D, packing)
    data = np.zeros(ds, dtype=np.uint8)
    scales = np.zeros(ss, dtype=np.uint8)
    _load().orc_quantize_pages(H, D, T, int(packing), dtype, _ptr(src), _ptr(sids),
                               float(src_scale), float(g), _ptr(data), _ptr(scales), _ptr(dids),
                               int(num_pages))
    return data, scales


def cast_fp8_pages(src, dtype, H, D, T, ws_scale=1.0, num_dst_pages=None, src_page_ids=None,
                   dst_page_ids=None, num_pages=None, src_scale=1.0):
    """FP8 E4M3 copy of source pages (the extend path's workspace copy of the current chunk):
    E4M3(fp32(x * fp32(1 / ws_scale))) bytes shaped [num_dst_pages, H, T, D]; an FP8 source
    is read as x = fp32(e4m3 * src_scale)."""
    src = _src_dtype(src, dtype)
    sids, dids = _ids(src_page_ids), _ids(dst_page_ids)
    if num_pages is None:
        num_pages = len(sids) if sids is not None else src.size // (H * T * D)
    if num_dst_pages is None:
        num_dst_pages = int(dids.max()) + 1 if dids is not None and len(dids) else num_pages
    out = np.zeros((num_dst_pages, H, T, D), dtype=np.uint8)
    _load().orc_cast_fp8_pages(H, D, T, dtype, _ptr(src), _ptr(sids), float(src_scale),
                               float(ws_scale), _ptr(out), _ptr(dids), int(num_pages))
    return out


def dequantize_pages(data, scales, H, D, T, g, out_dtype=BF16, num_dst_pages=None,
                     src_page_ids=None, dst_page_ids=None, num_pages=None, out_scale=1.0,
                     packing=DIM_PAIRS):
    """Decode NVFP4 pages to BF16/FP16 bit patterns (uint16) or FP8 E4M3 bytes."""
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    sids, dids = _ids(src_page_ids), _ids(dst_page_ids)
    if num_pages is None:
        num_pages = len(sids) if sids is not None else data.size // (H * T * D // 2)
    if num_dst_pages is None:
        num_dst_pages = int(dids.max()) + 1 if dids is not None and len(dids) else num_pages
    odt = np.uint8 if out_dtype == FP8_E4M3 else np.uint16
    out = np.zeros((num_dst_pages, H, T, D), dtype=odt)
    _load().orc_dequantize_pages(H, D, T, int(packing), _ptr(data), _ptr(scales), _ptr(sids),
                                 float(g), int(out_dtype), _ptr(out), _ptr(dids),
                                 float(out_scale), int(num_pages))
    return out


# ---------------------------------------------------------------- attention

def paged_decode_attention(q_bf16, k_data, k_scales, g_k, v_data, v_scales, g_v, page_table,
                           seq_lens, sm_scale, H, T, want_lse=True, want=None,
                           k_packing=DIM_PAIRS, v_packing=DIM_PAIRS):
    """Exact (fp64) GQA decode attention over NVFP4 pages.

    q_bf16: uint16 [B, Hq, D]; page_table: int32 [B, max_pages]; seq_lens: int32 [B].
    want: optional bool [B, Hq] selecting the (sequence, head) pairs to compute (others stay 0).
    Returns (out fp64 [B, Hq, D], lse fp64 [B, Hq]).
    """
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    B, Hq, D = q.shape
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    kd, ks = np.ascontiguousarray(k_data, np.uint8), np.ascontiguousarray(k_scales, np.uint8)
    vd, vs = np.ascontiguousarray(v_data, np.uint8), np.ascontiguousarray(v_scales, np.uint8)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64) if want_lse else None
    wm = None if want is None else np.ascontiguousarray(want, dtype=np.uint8).reshape(B, Hq)
    _load().orc_paged_decode_attention(B, Hq, H, D, T, int(k_packing), int(v_packing), _ptr(q),
                                       _ptr(kd), _ptr(ks), float(g_k), _ptr(vd), _ptr(vs),
                                       float(g_v), _ptr(pt), pt.shape[1], _ptr(sl),
                                       float(sm_scale), _ptr(wm), _ptr(out), _ptr(lse))
    return out, lse


def paged_decode_attention_bf16(q_bf16, k_bf16, v_bf16, page_table, seq_lens, sm_scale, H, T):
    """The same attention over unquantized BF16 pages (uint16 [P][H][T][D]); fp64 output."""
    q = np.ascontiguousarray(q_bf16, dtype=np.uint16)
    B, Hq, D = q.shape
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    k = np.ascontiguousarray(k_bf16, dtype=np.uint16)
    v = np.ascontiguousarray(v_bf16, dtype=np.uint16)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    _load().orc_paged_decode_attention_bf16(B, Hq, H, D, T, _ptr(q), _ptr(k), _ptr(v), _ptr(pt),
                                            pt.shape[1], _ptr(sl), float(sm_scale), _ptr(out))
    return out


# ------------------------------------------------------------------------------ cold pages
# "KV Cache Compression in TensorRT LLM" (NVIDIA), "NVFP4 Cold-Page Compression": a cold page
# is one fixed-size block per page holding the NVFP4 data, the block scales and the lossless
# bytes (Figure 6); encode happens on the way out, decode on the way back (Figure 7); the
# position-encoded (RoPE) part of K may be quantized like the rest, kept at its original
# precision, or stored as two FP4 components ("The RoPE part of K"). The block order taken
# here: K codes of the other head dims (dim pairs), their scales, the RoPE part (SKIP: the
# 16-bit values; 2FP4: codes and scales of the first, then of the second component), V codes,
# V scales, extra bytes, each part starting at the previous part's end rounded up to 16 bytes.

ROPE_QUANTIZE, ROPE_SKIP, ROPE_2FP4 = 0, 1, 2


def encode_2fp4_blocks(x_bits, dtype, g):
    """Two-component encoding (R10 of nvfp4_oracle.c) of blocks of 16 consecutive 16-bit
    values: (codes1 [n, 8], scales1 [n], codes2 [n, 8], scales2 [n])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    n = x.size // 16
    c1 = np.zeros((n, 8), np.uint8)
    c2 = np.zeros((n, 8), np.uint8)
    s1 = np.zeros(n, np.uint8)
    s2 = np.zeros(n, np.uint8)
    _load().orc_encode_2fp4_blocks(n, int(dtype), _ptr(x), float(g), _ptr(c1), _ptr(s1),
                                   _ptr(c2), _ptr(s2))
    return c1, s1, c2, s2


def decode_2fp4_blocks(c1, s1, c2, s2, g, out_dtype=BF16):
    """16-bit patterns [n, 16] of two-component blocks (R10)."""
    c1, c2 = (np.ascontiguousarray(a, dtype=np.uint8) for a in (c1, c2))
    s1, s2 = (np.ascontiguousarray(a, dtype=np.uint8) for a in (s1, s2))
    n = s1.size
    out = np.zeros((n, 16), np.uint16)
    _load().orc_decode_2fp4_blocks(n, _ptr(c1), _ptr(s1), _ptr(c2), _ptr(s2), float(g),
                                   int(out_dtype), _ptr(out))
    return out


def cold_block_layout(H, D, T, extra_bytes=0, rope=None):
    """Byte offsets of the parts of one cold block and its size; rope = (mode, first_dim,
    dims) or None (quantized like the rest). Parts a mode does not use are -1."""
    def up16(x):
        return (x + 15) // 16 * 16
    mode = ROPE_QUANTIZE if rope is None else rope[0]
    R = 0 if mode == ROPE_QUANTIZE else rope[2]
    rows = H * T
    off = {}
    at = 0

    def part(name, nbytes):
        nonlocal at
        off[name] = at
        at = up16(at + nbytes)
    part("k_data", rows * (D - R) // 2)
    part("k_scales", rows * (D - R) // 16)
    for name in ("k_rope", "k_rope_scales", "k_rope2", "k_rope2_scales"):
        off[name] = -1
    if mode == ROPE_SKIP:
        part("k_rope", rows * R * 2)
    elif mode == ROPE_2FP4:
        part("k_rope", rows * R // 2)
        part("k_rope_scales", rows * R // 16)
        part("k_rope2", rows * R // 2)
        part("k_rope2_scales", rows * R // 16)
    part("v_data", rows * D // 2)
    part("v_scales", rows * D // 16)
    off["extra"] = at
    off["bytes"] = at + int(extra_bytes)
    return off


def _rope_cols(D, rope):
    """(other head dims, RoPE head dims) of a K vector."""
    mode = ROPE_QUANTIZE if rope is None else rope[0]
    if mode == ROPE_QUANTIZE:
        return np.arange(D), np.arange(0)
    rc = np.arange(rope[1], rope[1] + rope[2])
    return np.setdiff1d(np.arange(D), rc), rc


def cold_offload(k, v, dtype, H, D, T, g_k, g_v, num_slots, hot_page_ids=None,
                 cold_slot_ids=None, extra=None, extra_bytes=0, num_pages=None, rope=None):
    """Cold blocks [num_slots, bytes] (uint8, zero where nothing is written) of hot pages
    hot_page_ids[i] -> slots cold_slot_ids[i]: K's other dims and V encoded exactly as
    quantize_pages (dim pairs) with g_k / g_v, the RoPE part of K as `rope` says, placed by
    cold_block_layout, and extra[hot page, :extra_bytes] copied unchanged."""
    lay = cold_block_layout(H, D, T, extra_bytes, rope)
    hids = _ids(hot_page_ids)
    sids = _ids(cold_slot_ids)
    if num_pages is None:
        num_pages = len(hids) if hids is not None else k.size // (H * T * D)
    k = np.ascontiguousarray(k, dtype=np.uint16).reshape(-1, H, T, D)
    hot = hids if hids is not None else np.arange(num_pages, dtype=np.int32)
    kp = k[hot[:num_pages]]                               # [n, H, T, D] in batch order
    oc, rc = _rope_cols(D, rope)
    mode = ROPE_QUANTIZE if rope is None else rope[0]
    N, R = oc.size, rc.size
    if N:
        kd, ks = quantize_pages(np.ascontiguousarray(kp[..., oc]), dtype, H, N, T, g_k)
    vd, vs = quantize_pages(v, dtype, H, D, T, g_v, src_page_ids=hids, num_pages=num_pages)
    if mode == ROPE_2FP4:
        r1, rs1, r2, rs2 = encode_2fp4_blocks(np.ascontiguousarray(kp[..., rc]), dtype, g_k)
        per = H * T * R // 16
    rows = H * T
    blocks = np.zeros((num_slots, lay["bytes"]), dtype=np.uint8)

    def put(b, name, arr):
        a = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        b[lay[name]:lay[name] + a.size] = a
    for i in range(num_pages):
        s = int(sids[i]) if sids is not None else i
        hp = int(hot[i])
        b = blocks[s]
        if N:
            put(b, "k_data", kd[i])
            put(b, "k_scales", ks[i])
        if mode == ROPE_SKIP:
            put(b, "k_rope", kp[i][..., rc].reshape(rows, R))
        elif mode == ROPE_2FP4:
            put(b, "k_rope", r1[i * per:(i + 1) * per])
            put(b, "k_rope_scales", rs1[i * per:(i + 1) * per])
            put(b, "k_rope2", r2[i * per:(i + 1) * per])
            put(b, "k_rope2_scales", rs2[i * per:(i + 1) * per])
        put(b, "v_data", vd[i])
        put(b, "v_scales", vs[i])
        if extra_bytes:
            b[lay["extra"]:lay["extra"] + extra_bytes] = extra[hp, :extra_bytes]
    return blocks


def cold_onboard(blocks, H, D, T, g_k, g_v, out_dtype, num_hot_pages, cold_slot_ids=None,
                 hot_page_ids=None, extra_bytes=0, num_pages=None, rope=None):
    """(k, v, extra) hot pools [num_hot_pages, H, T, D] (16-bit patterns) and
    [num_hot_pages, extra_bytes] written from cold slots cold_slot_ids[i] into hot pages
    hot_page_ids[i]: the block's NVFP4 parts decoded exactly as dequantize_pages, the RoPE part
    of K copied back (SKIP) or decoded as two components (2FP4)."""
    lay = cold_block_layout(H, D, T, extra_bytes, rope)
    sids = _ids(cold_slot_ids)
    hids = _ids(hot_page_ids)
    if num_pages is None:
        num_pages = len(sids) if sids is not None else blocks.shape[0]
    oc, rc = _rope_cols(D, rope)
    mode = ROPE_QUANTIZE if rope is None else rope[0]
    N, R = oc.size, rc.size
    rows = H * T
    slot = [int(sids[i]) if sids is not None else i for i in range(num_pages)]
    hot = [int(hids[i]) if hids is not None else i for i in range(num_pages)]

    def part(name, size, shape, dt=np.uint8):
        if not slot:
            return np.zeros((0,) + shape, dt)
        return np.stack([blocks[s, lay[name]:lay[name] + size].view(dt).reshape(shape)
                         for s in slot])
    k = np.zeros((num_hot_pages, H, T, D), np.uint16)
    if N:
        kd = part("k_data", rows * N // 2, (H, T, N // 2))
        ks = part("k_scales", rows * N // 16, (H, T, N // 16))
        kn = dequantize_pages(kd, ks, H, N, T, g_k, out_dtype, num_pages=num_pages)
        for i in range(num_pages):
            k[hot[i]][..., oc] = kn[i]
    if mode == ROPE_SKIP:
        kr = part("k_rope", rows * R * 2, (H, T, R), np.uint16)
        for i in range(num_pages):
            k[hot[i]][..., rc] = kr[i]
    elif mode == ROPE_2FP4:
        nb = rows * R // 16
        for i, s in enumerate(slot):
            g = lambda name, sz: blocks[s, lay[name]:lay[name] + sz]  # noqa: E731
            y = decode_2fp4_blocks(g("k_rope", nb * 8).reshape(nb, 8), g("k_rope_scales", nb),
                                   g("k_rope2", nb * 8).reshape(nb, 8), g("k_rope2_scales", nb),
                                   g_k, out_dtype)
            k[hot[i]][..., rc] = y.reshape(H, T, R)
    vd = part("v_data", rows * D // 2, (H, T, D // 2))
    vs = part("v_scales", rows * D // 16, (H, T, D // 16))
    v = dequantize_pages(vd, vs, H, D, T, g_v, out_dtype, num_dst_pages=num_hot_pages,
                         dst_page_ids=hids, num_pages=num_pages)
    ex = np.zeros((num_hot_pages, extra_bytes), dtype=np.uint8)
    for i, s in enumerate(slot):
        ex[hot[i]] = blocks[s, lay["extra"]:lay["extra"] + extra_bytes]
    return k, v, ex
