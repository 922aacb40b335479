"""Pins for the FP64 oracle: each ties it to something other than itself.

* E4M3 decode: every byte against torch's float8_e4m3fn cast (a library
  routine) and against values fixed by the format definition.
* Attention: tiny cases against torch's scaled_dot_product_attention in
  float64 (a library routine evaluating the textbook definition), plus closed
  forms (a single visible key, a dominant score, constant scores giving causal
  prefix means, exact FP16 midpoints), invariances (page relocation, partition
  length) and the q1 / q8 tail identity.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _decoded_pool(w):
    """Logical K/V per sequence, decoded with torch's e4m3 cast and scaled."""
    kv = torch.from_numpy(w.kv_pages).view(torch.float8_e4m3fn).to(torch.float64)
    out = []
    for b in range(w.spec.B):
        L = int(w.seq_len[b])
        pages = w.block_table[b, : -(-L // w.spec.page)]
        k = kv[pages, 0].permute(1, 0, 2, 3).reshape(w.spec.Hkv, -1, w.spec.D)[:, :L]
        v = kv[pages, 1].permute(1, 0, 2, 3).reshape(w.spec.Hkv, -1, w.spec.D)[:, :L]
        sc = torch.from_numpy(w.kv_scales.astype(np.float64))
        out.append((k * sc[:, 0, None, None], v * sc[:, 1, None, None]))
    return out


def _sdpa_reference(w):
    """torch SDPA (float64, CPU, explicit boolean mask) per sequence."""
    B, Qmax, Hq, D = w.q.shape
    G = Hq // w.spec.Hkv
    ref = np.zeros((B, Qmax, Hq, D))
    pool = _decoded_pool(w)
    for b in range(B):
        L, ql = int(w.seq_len[b]), int(w.q_len[b])
        if L == 0 or ql == 0 or ql > L:
            continue
        k, v = pool[b]
        k = k.repeat_interleave(G, dim=0)  # [Hq][L][D]
        v = v.repeat_interleave(G, dim=0)
        q = torch.from_numpy(w.q[b, :ql].astype(np.float64)).permute(1, 0, 2)
        pos = torch.arange(ql)[:, None] + (L - ql)
        mask = torch.arange(L)[None, :] <= pos  # [ql][L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, attn_mask=mask, scale=w.sm_scale)
        ref[b, :ql] = o.permute(1, 0, 2).numpy()
    return ref


def _run(w, **kw):
    return oracle.verify_attn(w.q, w.kv_pages, w.block_table, w.seq_len,
                              w.q_len, w.kv_scales, sm_scale=w.sm_scale, **kw)


# ---------------------------------------------------------------- decode
def test_decode_every_byte_matches_torch_cast():
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.flatnonzero(nan).tolist() == [0x7F, 0xFF]
    assert np.array_equal(t[~nan], ref[~nan])


def test_decode_format_landmarks():
    # largest finite (S.1111.110), smallest normal, largest and smallest
    # subnormal, one, and the sign bit
    v = oracle.e4m3_value
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert v(0x08) == 2.0 ** -6
    assert v(0x07) == 7 * 2.0 ** -9 and v(0x01) == 2.0 ** -9
    assert v(0x38) == 1.0 and v(0xB8) == -1.0
    assert v(0x00) == 0.0 and math.copysign(1.0, v(0x80)) == -1.0
    # every finite magnitude is an integer multiple of 2^-9 below 2^-6 and
    # has a 4-bit significand above it
    t = oracle.e4m3_table()[:0x7F]
    for b, x in enumerate(t):
        if b < 8:
            assert x == b * 2.0 ** -9
        else:
            m, e = math.frexp(x)
            assert (m * 16) == int(m * 16)


# ------------------------------------------------------------- quantiser
def test_quantizer_round_trip_every_finite_code():
    t = oracle.e4m3_table()
    codes = np.array([b for b in range(256) if b not in (0x7F, 0xFF)], np.uint8)
    vals = t[codes].astype(np.float32)
    back = W.quantize_e4m3(vals)
    # +0 / -0 keep their sign bit; every other code maps to itself
    assert np.array_equal(back, codes)


def test_quantizer_midpoints_go_to_even_and_saturate():
    t = oracle.e4m3_table()
    pos = [b for b in range(0x7F)]  # 0 .. 448
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = np.float32((t[lo] + t[hi]) / 2)
        assert float(mid) == (t[lo] + t[hi]) / 2  # exact in fp32
        got = int(W.quantize_e4m3(np.array([mid]))[0])
        want = lo if lo % 2 == 0 else hi  # even mantissa bit
        assert got == want, (lo, hi, mid, got)
    big = np.array([448.0, 449.0, 464.0, 479.0, 1e4, 3.4e38], np.float32)
    assert (W.quantize_e4m3(big) == 0x7E).all()
    assert (W.quantize_e4m3(-big) == 0xFE).all()
    tiny = np.array([2.0 ** -11, 2.0 ** -10, 1e-30], np.float32)  # <= half min subnormal
    assert (W.quantize_e4m3(tiny) == 0x00).all()
    assert (W.quantize_e4m3(-tiny) == 0x80).all()


def test_quantizer_matches_torch_cast_on_random_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * s
                        for s in (1e-3, 1.0, 30.0, 300.0)])
    ours = W.quantize_e4m3(x)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# -------------------------------------------------------------- attention
def _small(name="small", **kw):
    base = dict(B=2, Qmax=4, Hq=4, Hkv=2, D=16, seq_lens=[37, 5],
                q_lens=[4, 3], seed=21)
    base.update(kw)
    return W.custom(name, **base)


@pytest.mark.parametrize("kw", [
    dict(),
    dict(seq_lens=[1, 16], q_lens=[1, 4]),
    dict(B=3, Qmax=2, Hq=6, Hkv=1, D=8, seq_lens=[17, 2, 40], q_lens=[2, 2, 1]),
    dict(D=64, seq_lens=[100, 33], q_lens=[4, 4], outliers=True),
])
def test_attention_matches_torch_sdpa_fp64(kw):
    w = _small(**kw)
    ours = _run(w)
    ref = _sdpa_reference(w)
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-14)


def test_padded_slots_and_degenerate_lengths_are_zero():
    w = _small(seq_lens=[0, 3], q_lens=[2, 4])  # q_len > L on sequence 1
    out = _run(w)
    assert not out.any()
    w = _small(seq_lens=[20, 9], q_lens=[1, 2])
    out = _run(w)
    assert not out[0, 1:].any() and not out[1, 2:].any()
    assert np.abs(out[0, 0]).sum() > 0 and np.abs(out[1, :2]).sum() > 0


def test_single_visible_key_returns_its_value():
    w = _small(seq_lens=[1, 1], q_lens=[1, 1])
    out = _run(w)
    pool = _decoded_pool(w)
    G = w.spec.Hq // w.spec.Hkv
    for b in range(2):
        for hq in range(w.spec.Hq):
            np.testing.assert_array_equal(out[b, 0, hq], pool[b][1][hq // G, 0].numpy())


def test_dominant_score_selects_its_value():
    w = _small(B=1, Qmax=1, Hq=1, Hkv=1, D=16, seq_lens=[50], q_lens=[1])
    # queries all ones; every key zero except key 17, whose elements are 256
    w.q[:] = np.float16(1.0)
    w.kv_scales[0, 0] = np.float32(1.0)
    bt = w.block_table[0]
    w.kv_pages[bt, 0] = 0x00
    w.kv_pages[bt[17 // 16], 0, 0, 17 % 16] = 0x78
    out = _run(w)
    pool = _decoded_pool(w)
    z = w.sm_scale * 16 * 256.0  # 1024: every other weight is e^-1024 = 0
    assert z > 60
    np.testing.assert_array_equal(out[0, 0, 0], pool[0][1][0, 17].numpy())


@pytest.mark.parametrize("L,q", [(40, 4), (8, 8), (33, 1), (1000, 16)])
def test_equal_scores_give_causal_prefix_means(L, q):
    """Constant keys make every score equal, so query i's output is the mean
    of x_V over keys 0 .. L-q+i; successive queries differ by one key."""
    w = _small(B=1, Qmax=q, Hq=2, Hkv=1, D=8, seq_lens=[L], q_lens=[q], seed=5)
    w.kv_pages[:, 0] = 0x38  # every key element = 1.0 (times s_K)
    out = _run(w)
    v = _decoded_pool(w)[0][1][0].numpy()  # [L][D]
    csum = np.cumsum(v, axis=0)
    for i in range(q):
        pos = L - q + i
        mean = csum[pos] / (pos + 1)
        for hq in range(2):
            np.testing.assert_allclose(out[0, i, hq], mean, rtol=1e-13, atol=1e-15)


def test_exact_fp16_midpoints():
    """Equal scores and V bytes chosen so every output is exactly the midpoint
    between two fp16 neighbours: the ties-to-even cases that normalised
    FP16 partials round the wrong way (PR #524, final status)."""
    w = W.midpoint_case()
    out = _run(w)[0, 0, 0]
    lo, hi = W.MIDPOINT_VALUES
    h = out.shape[0] // 2
    assert (out[:h] == lo).all() and (out[h:] == hi).all()
    for x, up in ((lo, False), (hi, True)):
        a = np.float16(x)
        nb = np.nextafter(a, np.float16(-np.inf) if up else np.float16(np.inf))
        assert abs(float(a) - x) == abs(float(nb) - x)  # a true tie
        assert (a.view(np.uint16) & 1) == 0              # RNE: even neighbour
        assert (float(a) > x) == up


def test_page_relocation_is_bitwise_invariant():
    w = _small(B=2, seq_lens=[150, 77], q_lens=[4, 2], seed=13)
    a = _run(w)
    rng = np.random.default_rng(3)
    perm = rng.permutation(w.kv_pages.shape[0])
    kv2 = np.empty_like(w.kv_pages)
    kv2[perm] = w.kv_pages             # page p moves to perm[p]
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1)
    b = oracle.verify_attn(w.q, kv2, bt2.astype(np.int32), w.seq_len, w.q_len,
                           w.kv_scales, sm_scale=w.sm_scale)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("T", [16, 48, 256, 1648, 4096])
def test_partition_length_invariance(T):
    w = _small(B=2, Qmax=8, Hq=6, Hkv=1, D=32, seq_lens=[3297, 1025],
               q_lens=[8, 5], seed=17, outliers=True)
    d = _run(w)
    s = _run(w, split_tokens=T)
    rel = np.linalg.norm(s - d) / np.linalg.norm(d)
    assert rel <= 1e-12


def test_q1_equals_last_row_of_q8():
    w8 = _small(B=1, Qmax=8, Hq=6, Hkv=1, D=32, seq_lens=[500], q_lens=[8], seed=23)
    o8 = _run(w8)
    o1 = oracle.verify_attn(w8.q[:, 7:8], w8.kv_pages, w8.block_table,
                            w8.seq_len, np.array([1], np.int32), w8.kv_scales,
                            sm_scale=w8.sm_scale)
    assert np.array_equal(o1[0, 0], o8[0, 7])


def test_row_mode_matches_full_mode():
    w = _small(B=2, Qmax=4, seq_lens=[60, 31], q_lens=[4, 3], seed=29)
    full = _run(w)
    rows = W.sample_rows(w, 10, seed=1)
    part = _run(w, rows=rows)
    for r, (b, i, hq) in enumerate(rows):
        assert np.array_equal(part[r], full[b, i, hq])


def test_bad_block_id_is_reported():
    w = _small(seq_lens=[40, 5], q_lens=[1, 1])
    w.block_table[0, 1] = w.kv_pages.shape[0]
    with pytest.raises(oracle.OracleError):
        _run(w)


def test_length_beyond_the_block_table_is_reported():
    """L past the last token the block table can address (max_pages * page)
    is an input error, reported rather than read out of bounds; L exactly at
    that limit is valid and gives the same rows as a wider table."""
    w = _small(B=2, seq_lens=[40, 5], q_lens=[1, 1])
    cap = w.block_table.shape[1] * w.spec.page
    sl = w.seq_len.copy()
    sl[0] = cap + 1
    with pytest.raises(oracle.OracleError, match="beyond the block table"):
        oracle.verify_attn(w.q, w.kv_pages, w.block_table, sl, w.q_len, w.kv_scales)
    sl[0] = cap
    wide = np.concatenate([w.block_table, np.full_like(w.block_table, -1)], axis=1)
    a = oracle.verify_attn(w.q, w.kv_pages, w.block_table, sl, w.q_len, w.kv_scales)
    b = oracle.verify_attn(w.q, w.kv_pages, wide, sl, w.q_len, w.kv_scales)
    assert np.array_equal(a, b) and np.isfinite(a).all()


# ------------------------------------------------ token-major, strided cache
@pytest.mark.parametrize("kw,pad", [
    (dict(B=2, Qmax=4, Hq=4, Hkv=2, D=16, seq_lens=[37, 5], q_lens=[4, 3]), 8),
    (dict(B=1, Qmax=8, Hq=6, Hkv=1, D=32, seq_lens=[300], q_lens=[8], page=48), 8),
    (dict(B=2, Qmax=2, Hq=2, Hkv=1, D=64, seq_lens=[70, 33], q_lens=[2, 1]), 0),
])
def test_token_major_strided_cache_gives_identical_bits(kw, pad):
    """The same logical K/V in the library's pool and in the pages'
    token-major layout with a padded token stride (PR #524, AI integration
    review): the oracle reads the same bytes, so the outputs are identical
    bit for bit, in direct and in split mode.  Padding holds NaN codes, so a
    read of it would show."""
    w = _small(**kw)
    c = W.token_major(w, token_pad=pad, page_pad=16)
    k, v = c.views()
    assert k.strides[1] == w.spec.Hkv * w.spec.D + pad
    for T in (0, 16):
        a = _run(w, split_tokens=T)
        b = oracle.verify_attn_strided(w.q, k, v, w.block_table, w.seq_len, w.q_len,
                                       w.kv_scales, sm_scale=w.sm_scale, split_tokens=T)
        assert np.array_equal(a, b) and np.isfinite(b).all()


def test_token_major_counterexample_layout():
    """The pages' counterexample view: block size 848, one KV head, D = 256,
    strides [223872, 264, 256, 1].  The oracle over that layout matches torch
    SDPA (float64) on the K/V gathered from it with NumPy indexing."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_sizes.json")))
    ce = g["stride_counterexample"]
    w = _small(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[1000], q_lens=[8], page=848, seed=31)
    c = W.token_major(w, token_pad=ce["strides"][1] - 256)
    k, v = c.views()
    assert list(k.strides) == ce["strides"] and list(k.shape[1:]) == ce["shape"][1:]
    got = oracle.verify_attn_strided(w.q, k, v, w.block_table, w.seq_len, w.q_len,
                                     w.kv_scales, sm_scale=w.sm_scale)
    # independent reference: gather the logical K/V rows with NumPy, decode
    # with torch's FP8 cast, attend with torch SDPA in float64
    L, ql = int(w.seq_len[0]), int(w.q_len[0])
    pages = w.block_table[0, np.arange(L) // 848]
    slots = np.arange(L) % 848
    kk = torch.from_numpy(np.ascontiguousarray(k[pages, slots, 0])).view(
        torch.float8_e4m3fn).to(torch.float64) * float(w.kv_scales[0, 0])
    vv = torch.from_numpy(np.ascontiguousarray(v[pages, slots, 0])).view(
        torch.float8_e4m3fn).to(torch.float64) * float(w.kv_scales[0, 1])
    qq = torch.from_numpy(w.q[0, :ql].astype(np.float64)).permute(1, 0, 2)  # [Hq][ql][D]
    mask = torch.arange(L)[None, :] <= (torch.arange(ql)[:, None] + L - ql)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qq, kk[None].expand(6, -1, -1), vv[None].expand(6, -1, -1), attn_mask=mask,
        scale=w.sm_scale).permute(1, 0, 2).numpy()
    assert np.allclose(got[0, :ql], ref, rtol=1e-12, atol=1e-14)
