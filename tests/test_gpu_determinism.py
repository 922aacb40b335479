"""Bitwise determinism of the verify step on the automatic partition plans.

The contract (PR #560 "[Bugfix] Use FP32 state and E4M3 defaults for
DFlash2", Test Plan and Results: relocated pages, repeated graph replays,
changed and zero live lengths) is that the output bits do not depend on where
the pages live, on how often the step runs, or on what an earlier replay of
the same graph computed.  These tests hold it on the plans calls get by
default (partition_tokens = 0):

* one sequence: the static grid whose partition length follows the
  sequence's length on the device (the benchmarked configuration);
* a batch: the device-side balanced plan.

Each case is also checked against the FP64 oracle within the tolerance of
the other parity tests."""
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
    """Elementwise max-abs bound: 2e-3, or one fp16 ulp of the exact value
    where that is larger (|ref| >= 4, where FP16 cannot hold 2e-3)."""
    a = np.abs(ref)
    ulp = np.where(a > 0, np.ldexp(1.0, np.frexp(a)[1] - 11), 0.0)
    return np.maximum(MAX_ABS, ulp)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    vae4.load()


def bits(t):
    return t.cpu().numpy().view(np.uint16).copy()


def check_oracle(w, got, seq_len, q_len):
    q = np.where(np.isnan(w.q), 0, w.q)
    ref = oracle.verify_attn(q, w.kv_pages, w.block_table, seq_len, q_len, w.kv_scales,
                             sm_scale=w.sm_scale)
    g = got.view(np.float16).astype(np.float64)
    live = np.zeros(ref.shape, bool)
    for b in range(w.spec.B):
        live[b, :int(q_len[b]) if seq_len[b] > 0 and q_len[b] <= seq_len[b] else 0] = True
    assert not g[~live].any()
    g, r = g[live], ref[live]
    assert np.isfinite(g).all()
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    assert rel <= REL_L2, rel
    assert (np.abs(g - r) <= abs_bound(r)).all(), np.abs(g - r).max()


def run_once(w, tensors, ws, T=0):
    q, kv, bt, seq, sc = tensors
    out = torch.full_like(q, float("nan"))
    vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=T, max_seq_len=w.capacity)
    torch.cuda.synchronize()
    return bits(out)


def determinism(w, cases, T=0):
    """Direct calls, a relocated pool, repeated calls, and one captured graph
    replayed over `cases` (lists of (seq_len, q_len)) and back: every replay
    gives the bits of the direct call with the same lengths."""
    s = w.spec
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, T)
    ws2 = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, T)
    wr = W.relocate(w, seed=77)
    direct = []
    for sl, ql in cases:
        t = W.to_device(w, seq_len=sl, q_len=ql)
        a = run_once(w, t, ws, T)
        assert np.array_equal(a, run_once(w, t, ws, T)), "repeated launch"
        a_r = run_once(wr, W.to_device(wr, seq_len=sl, q_len=ql), ws2, T)
        assert np.array_equal(a, a_r), "page relocation"
        check_oracle(w, a, sl, ql)
        direct.append(a)
    # one graph, captured at the first lengths, replayed over all of them
    q, kv, bt, seq, sc = W.to_device(w, seq_len=cases[0][0], q_len=cases[0][1])
    out = torch.zeros_like(q)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=T, max_seq_len=w.capacity)
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=T, max_seq_len=w.capacity)
    order = list(range(len(cases))) + [0, len(cases) - 1, 0]
    for k in order:
        sl, ql = cases[k]
        seq.copy_(torch.from_numpy(np.stack([sl, ql], 1).astype(np.int32)))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), direct[k]), f"graph replay of case {k}"
    assert vae4.read_status(ws) == 0 and vae4.read_status(ws2) == 0


def test_single_sequence_plan_from_length_is_bitwise_stable():
    """B = 1: T follows L on the device (the benchmarked plan)."""
    cases = [(np.array([20000], np.int32), np.array([8], np.int32)),
             (np.array([12345], np.int32), np.array([8], np.int32)),
             (np.array([1000], np.int32), np.array([1], np.int32)),
             (np.array([0], np.int32), np.array([8], np.int32))]
    w = W.custom("det1", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20000], q_lens=[8],
                 capacity=20000, seed=120, outliers=True, replays=cases)
    determinism(w, cases)


def test_device_plan_is_bitwise_stable():
    """1 < B: the device-side balanced plan, whose partition length and CTA
    placement change with the lengths of each replay."""
    base = [9000, 17, 3000, 0, 40000, 1025, 3297]
    cases = [(np.array(base, np.int32), np.array([8, 8, 1, 0, 16, 8, 1], np.int32)),
             (np.array([40000, 40000, 5, 77, 0, 1025, 3297], np.int32),
              np.array([16, 1, 1, 8, 8, 8, 16], np.int32)),
             (np.array([100, 200, 300, 400, 500, 600, 700], np.int32),
              np.array([1, 8, 16, 1, 8, 16, 1], np.int32))]
    w = W.custom("detB", B=7, Qmax=16, Hq=6, Hkv=1, D=256, seq_lens=base,
                 q_lens=[8, 8, 1, 0, 16, 8, 1], capacity=40000, seed=121, replays=cases)
    determinism(w, cases)


def test_device_plan_two_kv_heads_is_bitwise_stable():
    cases = [(np.array([5000, 777, 2500], np.int32), np.array([8, 3, 8], np.int32)),
             (np.array([6000, 16, 0], np.int32), np.array([8, 8, 8], np.int32))]
    w = W.custom("detH", B=3, Qmax=8, Hq=12, Hkv=2, D=128, seq_lens=[5000, 777, 2500],
                 q_lens=[8, 3, 8], capacity=6000, seed=122, replays=cases)
    determinism(w, cases)
