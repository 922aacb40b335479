"""Pins for the oracle's E5M2 KV format (the second FP8 cache format the
pages keep available beside E4M3) and for the E5M2 input quantiser.

* Decode: every byte against torch's float8_e5m2 cast (a library routine)
  and against the format identity that an E5M2 byte is the high byte of the
  FP16 with the same value.
* Quantiser: round trip on every finite code, ties to even, saturation,
  underflow, agreement with torch's cast.
* Attention: a tiny E5M2 workload against torch's scaled_dot_product_attention
  in float64 on the torch-decoded cache.
"""
import math

import numpy as np
import torch

import oracle
import workloads as W


def test_decode_every_byte_matches_torch_cast():
    t = oracle.fp8_table("e5m2")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(t), np.isnan(ref))
    assert np.array_equal(np.isinf(t), np.isinf(ref))
    fin = np.isfinite(ref)
    assert np.array_equal(t[fin], ref[fin])
    assert np.flatnonzero(np.isinf(t)).tolist() == [0x7C, 0xFC]
    assert np.flatnonzero(np.isnan(t)).tolist() == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]


def test_decode_is_the_fp16_high_byte():
    t = oracle.fp8_table("e5m2")
    h = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    fin = np.isfinite(t)
    assert np.array_equal(t[fin], h[fin])


def test_decode_format_landmarks():
    v = oracle.e5m2_value
    assert v(0x7B) == 57344.0 and v(0xFB) == -57344.0
    assert v(0x04) == 2.0 ** -14                 # smallest normal
    assert v(0x03) == 3 * 2.0 ** -16 and v(0x01) == 2.0 ** -16
    assert v(0x3C) == 1.0 and v(0xBC) == -1.0
    assert v(0x00) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    assert oracle.fp8_table("e4m3")[0x38] == 1.0  # the E4M3 table is unchanged


def test_quantizer_round_trip_every_finite_code():
    t = oracle.fp8_table("e5m2")
    codes = np.array([b for b in range(256) if np.isfinite(t[b])], np.uint8)
    assert np.array_equal(W.quantize_e5m2(t[codes].astype(np.float32)), codes)


def test_quantizer_midpoints_go_to_even_and_saturate():
    t = oracle.fp8_table("e5m2")
    pos = list(range(0x7C))  # 0 .. 57344
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = np.float32((t[lo] + t[hi]) / 2)
        assert float(mid) == (t[lo] + t[hi]) / 2  # exact in fp32
        got = int(W.quantize_e5m2(np.array([mid]))[0])
        assert got == (lo if lo % 2 == 0 else hi), (lo, hi, mid, got)
    big = np.array([57344.0, 57345.0, 60000.0, 61439.0, 1e9, 3.4e38], np.float32)
    assert (W.quantize_e5m2(big) == 0x7B).all()
    assert (W.quantize_e5m2(-big) == 0xFB).all()
    tiny = np.array([2.0 ** -18, 2.0 ** -17, 1e-30], np.float32)  # <= half min subnormal
    assert (W.quantize_e5m2(tiny) == 0x00).all()
    assert (W.quantize_e5m2(-tiny) == 0x80).all()


def test_quantizer_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * s
                        for s in (1e-5, 1.0, 300.0, 30000.0)])
    ref = torch.from_numpy(np.clip(x, -57344, 57344)).to(torch.float8_e5m2) \
        .view(torch.uint8).numpy()
    assert np.array_equal(W.quantize_e5m2(x), ref)


def test_attention_on_e5m2_cache_matches_torch_sdpa():
    w = W.custom("e5m2", B=2, Qmax=4, Hq=4, Hkv=2, D=16, seq_lens=[37, 5], q_lens=[4, 3],
                 seed=31, kv_format="e5m2")
    assert w.kv_scales.max() < 1e-3  # scale = amax / 57344
    got = oracle.verify_attn(w.q, w.kv_pages, w.block_table, w.seq_len, w.q_len, w.kv_scales,
                             sm_scale=w.sm_scale, kv_format="e5m2")
    kv = torch.from_numpy(w.kv_pages).view(torch.float8_e5m2).to(torch.float64)
    G = w.spec.Hq // w.spec.Hkv
    ref = np.zeros_like(got)
    sc = torch.from_numpy(w.kv_scales.astype(np.float64))
    for b in range(w.spec.B):
        L, ql = int(w.seq_len[b]), int(w.q_len[b])
        pages = w.block_table[b, : -(-L // w.spec.page)]
        k = kv[pages, 0].permute(1, 0, 2, 3).reshape(w.spec.Hkv, -1, w.spec.D)[:, :L]
        v = kv[pages, 1].permute(1, 0, 2, 3).reshape(w.spec.Hkv, -1, w.spec.D)[:, :L]
        k = (k * sc[:, 0, None, None]).repeat_interleave(G, dim=0)
        v = (v * sc[:, 1, None, None]).repeat_interleave(G, dim=0)
        q = torch.from_numpy(w.q[b, :ql].astype(np.float64)).permute(1, 0, 2)
        mask = torch.arange(L)[None, :] <= (torch.arange(ql)[:, None] + (L - ql))
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=w.sm_scale)
        ref[b, :ql] = o.permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-12
    # reading the same bytes as E4M3 gives a different result (the format
    # parameter reaches the decode)
    other = oracle.verify_attn(w.q, w.kv_pages, w.block_table, w.seq_len, w.q_len,
                               w.kv_scales, sm_scale=w.sm_scale)
    assert np.abs(other - got).max() > 1e-3
