"""verify_attn_e4m3_kv: separate K and V caches in the pages' token-major
layout [blocks][block_size][kv_heads][D] (PR #524 "[Kernel][SM70] Add opt-in
E4M3 grouped attention with FP32 partials", AI integration review and
revision-2 update), contiguous (tensor copies) and with padded token strides
that are multiples of 8 but not 16 bytes (8-byte copies), e.g. the pages'
[1,848,1,256] view with strides [223872,264,256,1].

Both copy paths fill shared memory with the same bytes as the pool form, so
the output must equal the pool form's bit for bit; it is also checked
against the FP64 oracle's strided reader.  Padding bytes hold NaN codes: a
read of them would poison the output."""
import numpy as np
import pytest
import torch

import fp8_paged_attention_e4m3_gb300 as vae4
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

REL_L2 = 5e-4
MAX_ABS = 2e-3


def abs_bound(ref):
    """2e-3, or one fp16 ulp of the exact value where that is larger."""
    a = np.abs(ref)
    ulp = np.where(a > 0, np.ldexp(1.0, np.frexp(a)[1] - 11), 0.0)
    return np.maximum(MAX_ABS, ulp)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    vae4.load()


def run_pool(w, T, **kw):
    q, kv, bt, seq, sc = W.to_device(w)
    s = w.spec
    out = torch.full_like(q, float("nan"))
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, T)
    vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=T, max_seq_len=w.capacity, **kw)
    torch.cuda.synchronize()
    assert vae4.read_status(ws) == 0
    return out.cpu().numpy()


def run_kv(w, cache, T, **kw):
    q, _, bt, seq, sc = W.to_device(w)
    k, v = cache.to_device()
    s = w.spec
    out = torch.full_like(q, float("nan"))
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, T)
    vae4.verify_attn_e4m3_kv(q, k, v, bt, seq, sc, out, ws, partition_tokens=T,
                             max_seq_len=w.capacity, **kw)
    torch.cuda.synchronize()
    assert vae4.read_status(ws) == 0
    return out.cpu().numpy()


def check_oracle(w, cache, got):
    k, v = cache.views()
    q = np.where(np.isnan(w.q), 0, w.q)
    ref = oracle.verify_attn_strided(q, k, v, w.block_table, w.seq_len, w.q_len, w.kv_scales,
                                     sm_scale=w.sm_scale, kv_format=w.spec.kv_format)
    live = np.zeros(ref.shape, bool)
    for b in range(w.spec.B):
        if w.seq_len[b] > 0 and w.q_len[b] <= w.seq_len[b]:
            live[b, :int(w.q_len[b])] = True
    g = got.astype(np.float64)
    assert not g[~live].any()
    g, r = g[live], ref[live]
    assert np.isfinite(g).all()
    rel = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert rel <= REL_L2, rel
    assert (np.abs(g - r) <= abs_bound(r)).all()


CASES = [
    # (workload, token_pad, partition_tokens): pad 0 -> tensor copies,
    # pad 8 -> 8-byte copies
    (dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3297, 1025], q_lens=[8, 5], seed=81), 0, 512),
    (dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3297, 1025], q_lens=[8, 5], seed=81), 8, 512),
    (dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20000], q_lens=[8], seed=82,
          outliers=True), 8, 0),
    (dict(B=3, Qmax=16, Hq=6, Hkv=1, D=256, seq_lens=[7000, 999, 70], q_lens=[16, 8, 1],
          seed=83), 0, 0),
    (dict(B=3, Qmax=16, Hq=6, Hkv=1, D=256, seq_lens=[7000, 999, 70], q_lens=[16, 8, 1],
          seed=83), 24, 0),
    (dict(B=2, Qmax=8, Hq=8, Hkv=2, D=128, seq_lens=[1500, 999], q_lens=[8, 3], seed=84), 0, 256),
    (dict(B=2, Qmax=8, Hq=8, Hkv=2, D=128, seq_lens=[1500, 999], q_lens=[8, 3], seed=84), 8, 256),
    (dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1025], q_lens=[8], seed=85), 8, 0),
    (dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1025], q_lens=[8], seed=85, page=48), 0, 0),
    # the pages' block: 848 tokens, one KV head, D = 256, 264-byte token stride
    (dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[5000, 848], q_lens=[8, 8], seed=86,
          page=848), 8, 0),
    (dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3000], q_lens=[8], seed=87, page=848,
          kv_format="e5m2"), 8, 1024),
]


@pytest.mark.parametrize("cfg,pad,T", CASES,
                         ids=[f"{c[0]['D']}-pad{c[1]}-T{c[2]}-{c[0].get('page', 16)}"
                              f"-{c[0].get('kv_format', 'e4m3')}" for c in CASES])
def test_token_major_matches_pool_bit_for_bit(cfg, pad, T):
    w = W.custom("layout", **cfg)
    flags = vae4.FLAG_KV_E5M2 if w.spec.kv_format == "e5m2" else 0
    cache = W.token_major(w, token_pad=pad, page_pad=32)
    a = run_pool(w, T, flags=flags)
    b = run_kv(w, cache, T, flags=flags)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    check_oracle(w, cache, b)


def test_counterexample_strides_with_hilo_and_relocation():
    """The [n,848,1,256] cache with strides [223872,264,256,1] exactly, the
    high/residual P split on, and every page moved elsewhere: same bits as
    the pool form with hilo_pv, and the relocated cache gives them too."""
    w = W.custom("ce", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[9000, 2500], q_lens=[8, 4],
                 seed=88, page=848)
    cache = W.token_major(w, token_pad=8)
    k, _ = cache.views()
    assert list(k.strides) == [223872, 264, 256, 1]
    a = run_pool(w, 0, hilo_pv=True)
    b = run_kv(w, cache, 0, hilo_pv=True)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    check_oracle(w, cache, b)
    wr = W.relocate(w, seed=9)
    c = run_kv(wr, W.token_major(wr, token_pad=8), 0, hilo_pv=True)
    assert np.array_equal(b.view(np.uint16), c.view(np.uint16))


def test_kv_caches_sharing_one_buffer():
    """K and V as two views of one [2][blocks][page][Hkv][D] buffer (vLLM's
    per-layer cache tensor), tensor copies."""
    w = W.custom("shared", B=2, Qmax=8, Hq=12, Hkv=2, D=256, seq_lens=[4000, 1234],
                 q_lens=[8, 8], seed=89)
    q, kvp, bt, seq, sc = W.to_device(w)
    both = kvp.permute(1, 0, 3, 2, 4).contiguous()  # [2][n][page][Hkv][D]
    k, v = both[0], both[1]
    s = w.spec
    out = torch.full_like(q, float("nan"))
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, 0)
    vae4.verify_attn_e4m3_kv(q, k, v, bt, seq, sc, out, ws, max_seq_len=w.capacity)
    torch.cuda.synchronize()
    a = run_pool(w, 0)
    assert np.array_equal(a.view(np.uint16), out.cpu().numpy().view(np.uint16))
