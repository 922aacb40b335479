"""verify_attn_e4m3_noalloc: the entry point for callers that cannot
allocate device memory (graph-capture regions, plugin callbacks whose host
framework owns all device memory, fixed-budget serving loops).  It must give
the same outputs as the regular entry point with a caller workspace, call
after call, while its library-owned scratch is reused.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test; it also passes alone in a fresh
process."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_paged_attention_e4m3_gb300 as vae4
import oracle
import workloads as W

pytestmark = pytest.mark.gpu

REL_L2 = 5e-4
MAX_ABS = 2e-3


def _noalloc_c_call(tensors, out, flags=0, **opt):
    """Through the C ABI: descriptors by pointer, the current stream, options."""
    lib = vae4.load()
    q, kv, bt, seq, sc = tensors
    descs = [vae4.describe(t) for t in (q, kv, bt, seq, sc, out)]
    o = vae4.Options(0.0, int(opt.get("partition_tokens", 0)), int(opt.get("max_seq_len", 0)),
                     0, int(flags))
    return lib.verify_attn_e4m3_noalloc(*[ctypes.byref(d) for d in descs],
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                        ctypes.byref(o))


def _within_tolerance(got, ref):
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    assert np.isfinite(g).all()
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    assert rel <= REL_L2, rel
    assert np.abs(g - r).max() <= MAX_ABS


def _dirty_the_scratch():
    """Leave other contents in the shared scratch: a call with another batch
    (another device-plan slot layout) and a call that aborts on purpose
    (short pipeline waits), which leaves partitions marked invalid."""
    w = W.custom("noalloc_other", B=5, Qmax=8, Hq=6, Hkv=1, D=256,
                 seq_lens=[3000, 9000, 17, 4444, 1025], q_lens=[8, 1, 8, 8, 3], seed=63)
    t = W.to_device(w)
    out = torch.zeros_like(t[0])
    assert _noalloc_c_call(t, out, max_seq_len=w.capacity) == 0
    assert _noalloc_c_call(t, out, flags=vae4.FLAG_TEST_SHORT_WAITS,
                           max_seq_len=w.capacity) == 0
    torch.cuda.synchronize()
    assert not out.any()  # the aborted call wrote zero rows


@pytest.mark.parametrize("cfg", [
    dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1024], q_lens=[8], seed=60,
         partition_tokens=256),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20000, 7777], q_lens=[8, 5], seed=61,
         partition_tokens=0),
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[30001], q_lens=[8], seed=64,
         partition_tokens=0),
])
def test_noalloc_matches_workspace_entry_point_twice(cfg):
    """Same kernels and plan as the workspace entry point, so the same bits:
    on two calls in a row, after other calls have left their contents in the
    scratch."""
    assert torch.cuda.is_available()
    w = W.custom("noalloc", **cfg)
    s = w.spec
    tensors = W.to_device(w)
    kw = dict(partition_tokens=s.partition_tokens, max_seq_len=w.capacity)
    need = vae4.workspace_bytes(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, s.partition_tokens)
    assert need <= vae4.NOALLOC_SCRATCH_BYTES
    ref_out = torch.full_like(tensors[0], float("nan"))
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, s.partition_tokens)
    vae4.verify(*tensors, ref_out, ws, **kw)
    torch.cuda.synchronize()
    ref_bits = ref_out.cpu().numpy().view(np.uint16)
    _dirty_the_scratch()
    for _ in range(2):  # the second call reuses the scratch the first left behind
        out = torch.full_like(tensors[0], float("nan"))
        assert _noalloc_c_call(tensors, out, **kw) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint16), ref_bits)
        _within_tolerance(got, ref_out.cpu().numpy())
    # and both agree with the FP64 oracle
    ref = oracle.verify_attn(w.q, w.kv_pages, w.block_table, w.seq_len, w.q_len, w.kv_scales,
                             sm_scale=w.sm_scale)
    _within_tolerance(out.cpu().numpy(), ref)
    assert vae4.read_status(ws) == 0


def test_noalloc_rejects_plans_beyond_its_scratch():
    w = W.custom("noalloc_big", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[4096], q_lens=[8],
                 seed=62)
    tensors = W.to_device(w)
    out = torch.zeros_like(tensors[0])
    # 16-token partitions of 4096 tokens: 256 partitions x 48 rows x 1 KiB of
    # FP32 partials = 12 MiB, more than the 8 MiB scratch
    need = vae4.workspace_bytes(1, 6, 1, 8, 256, 4096, 16)
    assert need > vae4.NOALLOC_SCRATCH_BYTES
    assert _noalloc_c_call(tensors, out, partition_tokens=16, max_seq_len=4096) == -8
