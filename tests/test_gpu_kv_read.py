"""The streaming-read reference kernel (the gather floor bench.py compares
the step with) reads exactly the KV bytes of the step: the XOR of every
32-bit word it loads equals the XOR over K and V of tokens 0 .. L-1 of every
(sequence, KV head), computed here from the host arrays."""
import numpy as np
import pytest
import torch

import fp8_paged_attention_e4m3_gb300 as vae4
import workloads as W

pytestmark = pytest.mark.gpu


def host_xor(w):
    s = w.spec
    acc = np.uint32(0)
    pages = w.kv_pages  # [n_pages][2][Hkv][page][D] u8
    for b in range(s.B):
        L = int(w.seq_len[b])
        for lp in range((L + s.page - 1) // s.page):
            toks = min(s.page, L - lp * s.page)
            phys = int(w.block_table[b, lp])
            blk = np.ascontiguousarray(pages[phys, :, :, :toks, :])
            acc ^= np.bitwise_xor.reduce(blk.reshape(-1).view(np.uint32))
    return int(acc)


@pytest.mark.parametrize("cfg", [
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20000], q_lens=[8], seed=21),
    dict(B=3, Qmax=8, Hq=4, Hkv=2, D=128, seq_lens=[3001, 17, 640], q_lens=[8, 1, 5], seed=22),
    dict(B=2, Qmax=4, Hq=2, Hkv=1, D=64, seq_lens=[999, 0], q_lens=[4, 0], seed=23),
])
def test_kv_read_reads_the_step_bytes(cfg):
    vae4.load()
    w = W.custom("kvread", **cfg)
    q, kv, bt, seq, sc = W.to_device(w)
    s = w.spec
    out = torch.zeros_like(q)
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, 0)
    ws[:256].zero_()
    vae4.verify_attn_e4m3_kv_read(q, kv, bt, seq, sc, out, ws, max_seq_len=w.capacity)
    torch.cuda.synchronize()
    got = int(ws[128:132].cpu().numpy().view(np.uint32)[0])
    assert got == host_xor(w)
    assert vae4.read_status(ws) == 0
    assert int(out.abs().sum().item()) == 0  # out is not written
