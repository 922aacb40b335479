"""GPU parity of the paged FP8 -> FP16 bridge against the oracle: bit-exact
FP16 for every written element (one correct rounding of the exact product),
tokens past L untouched, status bits for bad pages and lengths."""
import numpy as np
import pytest
import torch

import fp8_paged_attention_e4m3_gb300 as vae4
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

SENT = 0x7E01  # a NaN bit pattern no conversion produces


def run_bridge(w, kv_scales=None, flags=0, seq=None):
    vae4.load()
    q, kv, bt, seq_d, sc = W.to_device(w)
    if kv_scales is not None:
        sc = torch.from_numpy(np.asarray(kv_scales, np.float32)).cuda()
    if seq is not None:
        seq_d = torch.from_numpy(np.asarray(seq, np.int32)).cuda()
    s = w.spec
    shape = (s.B, s.Hkv, w.capacity, s.D)
    ko = torch.full(shape, 0, dtype=torch.int16, device="cuda").fill_(SENT).view(torch.float16)
    vo = torch.full(shape, 0, dtype=torch.int16, device="cuda").fill_(SENT).view(torch.float16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    vae4.verify_attn_e4m3_bridge_fp16(kv, bt, seq_d, sc, ko, vo, status=status, flags=flags)
    torch.cuda.synchronize()
    return (ko.cpu().numpy().view(np.uint16), vo.cpu().numpy().view(np.uint16),
            int(status.item()))


def expect_bits(w, kv_scales, fmt, raw):
    k, v = oracle.bridge_fp16(w.kv_pages, w.block_table, w.seq_len, kv_scales, w.capacity,
                              kv_format=fmt, raw=raw)
    out = []
    for x in (k, v):
        bits = np.full(x.shape, SENT, np.uint16)
        live = ~np.isnan(x)
        bits[live] = oracle.round_to_fp16(x[live]).view(np.uint16)
        out.append(bits)
    return out


CFGS = [
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3000, 47], q_lens=[8, 8], seed=81,
         outliers=True),
    dict(B=3, Qmax=8, Hq=4, Hkv=2, D=128, seq_lens=[999, 0, 1728], q_lens=[8, 0, 8], seed=82,
         page=48),
    dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[5000], q_lens=[8], seed=83, page=1728),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[700, 300], q_lens=[8, 8], seed=84,
         kv_format="e5m2"),
]


@pytest.mark.parametrize("raw", [False, True], ids=["scaled", "raw"])
@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: str(c["seed"]))
def test_bridge_bit_exact(cfg, raw):
    w = W.custom("bridge", **cfg)
    fmt = w.spec.kv_format
    flags = (vae4.FLAG_KV_E5M2 if fmt == "e5m2" else 0) | (vae4.FLAG_BRIDGE_RAW if raw else 0)
    gk, gv, st = run_bridge(w, flags=flags)
    ek, ev = expect_bits(w, w.kv_scales, fmt, raw)
    assert st == 0
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_bridge_ties_follow_the_exact_product():
    """Scales chosen so that many FP32 products land exactly on an FP16 tie
    while the exact product lies beyond it: s = fp32((3 + 2^-10) / 3) puts
    every 1.5 * 2^k byte's product within an FP32 rounding of the midpoint
    above 1.5 * 2^k."""
    w = W.custom("ties", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[4000], q_lens=[8], seed=85)
    s1 = np.float32((3 + 2.0 ** -10) / 3)
    s2 = np.float32((3 - 2.0 ** -10) / 3)
    sc = np.array([[s1, s2]], np.float32)
    p = np.float32(1.5) * s1  # the FP32 product for the byte 1.5
    assert float(p) == 1.5 + 2.0 ** -11 and float(np.float64(1.5) * np.float64(s1)) != float(p)
    gk, gv, st = run_bridge(w, kv_scales=sc)
    ek, ev = expect_bits(w, sc, "e4m3", False)
    assert st == 0
    assert np.array_equal(gk, ek) and np.array_equal(gv, ev)


def test_bridge_status_bits():
    w = W.custom("bad", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[600, 200], q_lens=[8, 8],
                 seed=86)
    w.block_table[0, 3] = 10 ** 6  # invalid page id
    _, _, st = run_bridge(w)
    assert st & vae4.STATUS_BAD_BLOCK
    w2 = W.custom("bad", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[600, 200], q_lens=[8, 8],
                  seed=86)
    gk, _, st = run_bridge(w2, seq=[[600, 8], [w2.capacity + 1, 8]])
    assert st & vae4.STATUS_BAD_LENGTH
    assert (gk[1] == SENT).all()  # the sequence was skipped
