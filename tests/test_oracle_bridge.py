"""Pins for the oracle of the paged FP8 -> FP16 bridge.

* The gather: raw values equal torch's FP8 cast of the bytes, gathered here
  with NumPy indexing through the block table (an implementation
  independent of the oracle's loops).
* The scaling: every scaled value divided by its scale gives the raw value
  back exactly (the FP64 product is exact).
* The one rounding step (NumPy's float64 -> float16 cast): ties between
  adjacent FP16 values go to the even one, values a hair off a tie go to the
  nearer one, across normal and subnormal binades.
"""
import numpy as np
import torch

import oracle
import workloads as W


def _gather(w, kv_format):
    dt = torch.float8_e5m2 if kv_format == "e5m2" else torch.float8_e4m3fn
    dec = torch.from_numpy(w.kv_pages).view(dt).to(torch.float64).numpy()
    s = w.spec
    B, Hkv, D, page, cap = s.B, s.Hkv, s.D, s.page, w.capacity
    k = np.full((B, Hkv, cap, D), np.nan)
    v = np.full((B, Hkv, cap, D), np.nan)
    for b in range(B):
        L = int(w.seq_len[b])
        t = np.arange(L)
        phys = w.block_table[b, t // page]
        k[b, :, :L] = dec[phys, 0, :, t % page].transpose(1, 0, 2)
        v[b, :, :L] = dec[phys, 1, :, t % page].transpose(1, 0, 2)
    return k, v


def test_raw_values_are_the_gathered_decode():
    for fmt, seed in (("e4m3", 71), ("e5m2", 72)):
        w = W.custom("br", B=3, Qmax=8, Hq=4, Hkv=2, D=64, seq_lens=[100, 33, 0],
                     q_lens=[8, 8, 0], seed=seed, page=32, kv_format=fmt)
        k, v = oracle.bridge_fp16(w.kv_pages, w.block_table, w.seq_len, w.kv_scales,
                                  w.capacity, kv_format=fmt, raw=True)
        gk, gv = _gather(w, fmt)
        assert np.array_equal(np.isnan(k), np.isnan(gk))
        assert np.array_equal(k[~np.isnan(k)], gk[~np.isnan(gk)])
        assert np.array_equal(v[~np.isnan(v)], gv[~np.isnan(gv)])


def test_scaled_values_are_exact_products():
    w = W.custom("br", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[300, 47], q_lens=[8, 8],
                 seed=73, outliers=True)
    k, v = oracle.bridge_fp16(w.kv_pages, w.block_table, w.seq_len, w.kv_scales, w.capacity)
    kr, vr = oracle.bridge_fp16(w.kv_pages, w.block_table, w.seq_len, w.kv_scales,
                                w.capacity, raw=True)
    live = ~np.isnan(k)
    sk, sv = np.float64(w.kv_scales[0, 0]), np.float64(w.kv_scales[0, 1])
    assert np.array_equal(k[live] / sk, kr[live])
    assert np.array_equal(v[live] / sv, vr[live])


def test_fp16_rounding_step_is_correct():
    # every adjacent pair of positive finite FP16 values (subnormals included)
    a = np.arange(0, 0x7BFF, dtype=np.uint16).view(np.float16).astype(np.float64)
    b = np.arange(1, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = (a + b) / 2  # exact in float64
    even_lo = (np.arange(0, 0x7BFF) % 2) == 0
    got = oracle.round_to_fp16(mid).astype(np.float64)
    assert np.array_equal(got, np.where(even_lo, a, b))
    eps = (b - a) * 2.0 ** -20
    assert np.array_equal(oracle.round_to_fp16(mid - eps).astype(np.float64), a)
    assert np.array_equal(oracle.round_to_fp16(mid + eps).astype(np.float64), b)
    assert np.array_equal(oracle.round_to_fp16(-(mid + eps)).astype(np.float64), -b)
