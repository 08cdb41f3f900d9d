"""Pins of the CPU oracle's paged GQA decode attention over NVFP4 K/V.

Source: "Accelerating Long-Context and Agentic Inference with NVFP4 KV Cache" (LMSYS blog),
"Path 3: Decode" (decode reads NVFP4 K/V straight from the paged cache) and "NVFP4 KV Decode
Attention Kernel Implementation" with Figure 3 (BF16 queries; K/V dequantized from packed tiles
and E4M3 block scales; the global K/V scales enter through the attention scaling). Attention
itself is its textbook definition. The checks below use closed forms, invariances and an
independent brute force in 40-digit decimal arithmetic over densely gathered K/V."""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def bf16_bits_of(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def bf16_val(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def rand_nvfp4(rng, P, H, T, D, scale_lo=0x20, scale_hi=0x48):
    data = rng.integers(0, 256, (P, H, T, D // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi, (P, H, T, D // 16), dtype=np.uint8)
    return data, scales


def dense_values(data, scales, g):
    """[P,H,T,D] float64 values e(c) * s * g, decoded with an element-by-element loop that is
    independent of the oracle's helpers."""
    P, H, T, half = data.shape
    D = half * 2
    out = np.zeros((P, H, T, D))
    e4 = [oracle.e4m3_value(b) for b in range(256)]
    for p in range(P):
        for h in range(H):
            for t in range(T):
                for d in range(D):
                    byte = int(data[p, h, t, d // 2])
                    c = (byte >> 4) if d % 2 else (byte & 15)
                    mag = E2M1[c & 7]
                    out[p, h, t, d] = (-mag if c & 8 else mag) * e4[scales[p, h, t, d // 16]] * g
    return out


def brute_attention(q, kd, vd, page_table, seq_lens, sm_scale, H, T):
    """40-digit decimal attention without the max shift: out = sum e^z v / sum e^z."""
    getcontext().prec = 40
    B, Hq, D = q.shape
    G = Hq // H
    out = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), -math.inf)
    for b in range(B):
        L = int(seq_lens[b])
        # gather the sequence's tokens densely, token index -> (page, slot)
        toks = [(int(page_table[b, t // T]), t % T) for t in range(L)]
        for qh in range(Hq):
            if L == 0:
                continue
            h = qh // G
            qs = [Decimal(float(x)) for x in q[b, qh]]
            ws, num = [], [Decimal(0)] * D
            for (p, s) in toks:
                z = Decimal(sm_scale) * sum(qs[d] * Decimal(float(kd[p, h, s, d]))
                                            for d in range(D))
                w = z.exp()
                ws.append(w)
                for d in range(D):
                    num[d] += w * Decimal(float(vd[p, h, s, d]))
            den = sum(ws)
            out[b, qh] = [float(n / den) for n in num]
            lse[b, qh] = float(den.ln())
    return out, lse


@pytest.mark.parametrize("shape", [
    dict(B=2, Hq=4, H=2, D=16, T=1, lens=[3, 1]),
    dict(B=2, Hq=2, H=2, D=16, T=2, lens=[5, 4]),
    dict(B=1, Hq=4, H=1, D=32, T=3, lens=[7]),
])
def test_brute_force_tiny(shape):
    rng = np.random.default_rng(11)
    B, Hq, H, D, T, lens = (shape[k] for k in ("B", "Hq", "H", "D", "T", "lens"))
    maxp = max(-(-L // T) for L in lens)
    P = B * maxp + 2
    kd, ks = rand_nvfp4(rng, P, H, T, D)
    vd, vs = rand_nvfp4(rng, P, H, T, D)
    g_k, g_v = 0.75, 1.25
    pt = rng.permutation(P)[:B * maxp].reshape(B, maxp).astype(np.int32)
    sl = np.array(lens, np.int32)
    q = bf16_bits_of(rng.normal(0, 1, (B, Hq, D)).tolist()).reshape(B, Hq, D)
    sm = float(np.float32(1.0 / math.sqrt(D)))   # the call takes an FP32 softmax scale
    out, lse = oracle.paged_decode_attention(q, kd, ks, g_k, vd, vs, g_v, pt, sl, sm, H, T)
    kv, vv = dense_values(kd, ks, g_k), dense_values(vd, vs, g_v)
    ref, ref_lse = brute_attention(bf16_val(q), kv, vv, pt, sl, sm, H, T)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def _setup(B=1, Hq=4, H=2, D=32, T=4, L=10, seed=12):
    rng = np.random.default_rng(seed)
    maxp = -(-L // T)
    P = B * maxp
    kd, ks = rand_nvfp4(rng, P, H, T, D)
    vd, vs = rand_nvfp4(rng, P, H, T, D)
    pt = np.arange(P, dtype=np.int32).reshape(B, maxp)
    sl = np.full(B, L, np.int32)
    q = bf16_bits_of(rng.normal(0, 1, (B, Hq, D)).tolist()).reshape(B, Hq, D)
    return rng, kd, ks, vd, vs, pt, sl, q


def test_single_token_returns_its_value():
    _, kd, ks, vd, vs, pt, sl, q = _setup(L=1, T=4)
    sm = float(np.float32(0.3))
    out, lse = oracle.paged_decode_attention(q, kd, ks, 1.5, vd, vs, 0.5, pt, sl, sm, 2, 4)
    vv = dense_values(vd, vs, 0.5)
    kv = dense_values(kd, ks, 1.5)
    qv = bf16_val(q)
    for qh in range(4):
        assert np.array_equal(out[0, qh], vv[pt[0, 0], qh // 2, 0])
        assert lse[0, qh] == pytest.approx(sm * float(qv[0, qh] @ kv[pt[0, 0], qh // 2, 0]),
                                           rel=1e-14, abs=1e-14)


def test_zero_query_gives_mean_of_values_and_log_length():
    """q = 0: every score is 0, the weights are uniform, out = mean of the L values and
    lse = ln L. Values are constant per page, so the mean checks the page-table lookup and the
    partial last page (L = 10 tokens over 4-token pages)."""
    rng, kd, ks, vd, vs, pt, sl, q = _setup(L=10, T=4)
    q[:] = 0
    P = vd.shape[0]
    consts = [1, 2, 3]
    for p in range(P):                         # page p holds one value everywhere
        vd[p] = consts[p] * 0x11               # code consts[p] in both nibbles
    vs[:] = 0x38                               # scale 1.0
    perm = np.array([[2, 0, 1]], np.int32)     # physical placement
    out, lse = oracle.paged_decode_attention(q, kd, ks, 1.0, vd, vs, 2.0, perm, sl, 1.0, 2, 4)
    vv = dense_values(vd, vs, 2.0)
    page_val = [vv[p, 0, 0, 0] for p in range(P)]
    want = (4 * page_val[2] + 4 * page_val[0] + 2 * page_val[1]) / 10
    np.testing.assert_allclose(out, want, rtol=1e-15)
    np.testing.assert_allclose(lse, math.log(10), rtol=1e-15)


def test_gqa_head_mapping():
    """Constant V per KV head: query head qh must return the constant of KV head qh // (Hq/H)."""
    rng, kd, ks, vd, vs, pt, sl, q = _setup(Hq=8, H=4, L=6, T=4)
    for h in range(4):
        vd[:, h] = (h + 1) * 0x11              # code h+1 in both nibbles
    vs[:] = 0x38
    out, _ = oracle.paged_decode_attention(q, kd, ks, 1.0, vd, vs, 1.0, pt, sl, 0.2, 4, 4)
    for qh in range(8):
        np.testing.assert_allclose(out[0, qh], E2M1[qh // 2 + 1], rtol=1e-15)


def test_two_tokens_closed_form():
    """Two tokens with known scores z0, z1: out = sigmoid(z0 - z1) v0 + sigmoid(z1 - z0) v1."""
    rng, kd, ks, vd, vs, pt, sl, q = _setup(Hq=1, H=1, D=16, T=2, L=2)
    q[:] = bf16_bits_of([[[1.0] * 16]])
    kd[0, 0, 0] = 0x22                          # token 0: all codes 2 (1.0)
    kd[0, 0, 1] = 0x44                          # token 1: all codes 4 (2.0)
    ks[:] = 0x38
    g_k, sm = 0.125, 0.5
    z0, z1 = sm * 16 * 1.0 * g_k, sm * 16 * 2.0 * g_k
    out, lse = oracle.paged_decode_attention(q, kd, ks, g_k, vd, vs, 1.0, pt, sl, sm, 1, 2)
    vv = dense_values(vd, vs, 1.0)
    w0 = 1 / (1 + math.exp(z1 - z0))
    np.testing.assert_allclose(out[0, 0], w0 * vv[0, 0, 0] + (1 - w0) * vv[0, 0, 1], rtol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(z0) + math.exp(z1)), rel=1e-15)


def test_dominant_score_selects_its_value():
    rng, kd, ks, vd, vs, pt, sl, q = _setup(Hq=1, H=1, D=16, T=4, L=8)
    q[:] = bf16_bits_of([[[1.0] * 16]])
    kd[:] = 0x00
    kd[1, 0, 2] = 0x77                          # token 6: codes 6 everywhere
    ks[:] = 0x38
    out, _ = oracle.paged_decode_attention(q, kd, ks, 1.0, vd, vs, 1.0, pt, sl, 1.0, 1, 4)
    vv = dense_values(vd, vs, 1.0)
    np.testing.assert_allclose(out[0, 0], vv[1, 0, 2], rtol=1e-12, atol=1e-30)


def test_page_permutation_invariance_and_mha():
    rng, kd, ks, vd, vs, pt, sl, q = _setup(B=2, Hq=3, H=3, D=32, T=4, L=11)
    out, lse = oracle.paged_decode_attention(q, kd, ks, 0.9, vd, vs, 1.1, pt, sl, 0.25, 3, 4)
    perm = rng.permutation(kd.shape[0])          # move page p to slot perm[p]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    kd2, ks2, vd2, vs2 = (np.empty_like(a) for a in (kd, ks, vd, vs))
    for a, b in ((kd, kd2), (ks, ks2), (vd, vd2), (vs, vs2)):
        b[perm] = a
    pt2 = perm[pt].astype(np.int32)
    out2, lse2 = oracle.paged_decode_attention(q, kd2, ks2, 0.9, vd2, vs2, 1.1, pt2, sl, 0.25,
                                               3, 4)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_empty_sequence_and_selection_mask():
    rng, kd, ks, vd, vs, pt, sl, q = _setup(B=2, L=5)
    sl[1] = 0
    out, lse = oracle.paged_decode_attention(q, kd, ks, 1.0, vd, vs, 1.0, pt, sl, 0.2, 2, 4)
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    want = np.zeros((2, 4), bool)
    want[0, 2] = True
    out_s, lse_s = oracle.paged_decode_attention(q, kd, ks, 1.0, vd, vs, 1.0, pt, sl, 0.2, 2, 4,
                                                 want=want)
    assert np.array_equal(out_s[0, 2], out[0, 2]) and lse_s[0, 2] == lse[0, 2]
    assert not out_s[0, :2].any() and not out_s[0, 3].any()


def test_bf16_attention_equals_nvfp4_attention_on_representable_kv():
    """K/V pages whose values are exactly NVFP4 values give the same attention through the
    NVFP4 path (with g) and the unquantized BF16 path."""
    rng, kd, ks, vd, vs, pt, sl, q = _setup(B=2, Hq=4, H=2, D=32, T=4, L=9)
    g = 0.5
    kb = bf16_bits_of(dense_values(kd, ks, g).tolist())
    vb = bf16_bits_of(dense_values(vd, vs, g).tolist())
    out, _ = oracle.paged_decode_attention(q, kd, ks, g, vd, vs, g, pt, sl, 0.2, 2, 4)
    out_b = oracle.paged_decode_attention_bf16(q, kb, vb, pt, sl, 0.2, 2, 4)
    np.testing.assert_allclose(out, out_b, rtol=1e-13, atol=1e-15)


def test_value_packing_does_not_change_attention():
    """The same V codes and scales stored token-pair packed give the same attention as stored
    dim-pair packed (and likewise for K)."""
    rng, kd, ks, vd, vs, pt, sl, q = _setup(B=2, Hq=4, H=2, D=32, T=4, L=7)
    P, H, T, half = vd.shape
    D = 2 * half

    def to_token_pairs(data, scales):
        codes = np.stack([data & 15, data >> 4], axis=-1).reshape(P, H, T, D)
        tp = (codes[:, :, 0::2, :] | (codes[:, :, 1::2, :] << 4)).astype(np.uint8)
        sc = np.stack([scales[:, :, 0::2, :], scales[:, :, 1::2, :]], axis=-1)
        return np.ascontiguousarray(tp), np.ascontiguousarray(sc)

    vtd, vts = to_token_pairs(vd, vs)
    ktd, kts = to_token_pairs(kd, ks)
    want, want_lse = oracle.paged_decode_attention(q, kd, ks, 0.7, vd, vs, 1.3, pt, sl, 0.25, H,
                                                   T)
    got, got_lse = oracle.paged_decode_attention(q, kd, ks, 0.7, vtd, vts, 1.3, pt, sl, 0.25, H,
                                                 T, v_packing=oracle.TOKEN_PAIRS)
    assert np.array_equal(got, want) and np.array_equal(got_lse, want_lse)
    got2, _ = oracle.paged_decode_attention(q, ktd, kts, 0.7, vtd, vts, 1.3, pt, sl, 0.25, H, T,
                                            k_packing=oracle.TOKEN_PAIRS,
                                            v_packing=oracle.TOKEN_PAIRS)
    assert np.array_equal(got2, want)
