"""GPU parity: the CUDA path through the C ABI against the FP64 oracle on the
same seeded inputs.  Tolerance on FP16 outputs: relative L2 <= 5e-4 and
max-abs <= 2e-3 over all live outputs (bitwise identity where the contract
asks for it: relocation, repeated launches, graph replay, exact decode)."""
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


def run_gpu(w, seq_len=None, q_len=None, partition_tokens=None, tensors=None, ws=None,
            flags=0, hilo_pv=False):
    q, kv, bt, seq, sc = tensors or W.to_device(w, seq_len=seq_len, q_len=q_len)
    s = w.spec
    T = s.partition_tokens if partition_tokens is None else partition_tokens
    out = torch.full_like(q, float("nan"))  # every element must be written
    if ws is None:
        ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, w.capacity, T)
    vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=T, max_seq_len=w.capacity,
                flags=flags, hilo_pv=hilo_pv)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ws


def compare(gpu, ref, live_mask=None):
    g = gpu.astype(np.float64)
    if live_mask is not None:
        g, ref = g[live_mask], ref[live_mask]
    assert np.isfinite(g).all()
    err = g - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(err).max() if err.size else 0.0
    assert rel <= REL_L2, rel
    assert (np.abs(err) <= abs_bound(ref)).all(), mx
    return rel, mx


def oracle_full(w, seq_len=None, q_len=None):
    sl = w.seq_len if seq_len is None else seq_len
    ql = w.q_len if q_len is None else q_len
    q = np.where(np.isnan(w.q), 0, w.q)  # padded slots are never read
    return oracle.verify_attn(q, w.kv_pages, w.block_table, sl, ql, w.kv_scales,
                              sm_scale=w.sm_scale, kv_format=w.spec.kv_format)


def check_full(w, **kw):
    if w.spec.kv_format == "e5m2":
        kw["flags"] = kw.get("flags", 0) | vae4.FLAG_KV_E5M2
    gpu, ws = run_gpu(w, **kw)
    ref = oracle_full(w)
    rel, mx = compare(gpu, ref)
    # padded slots / dead rows are exact zeros
    for b in range(w.spec.B):
        L, ql = int(w.seq_len[b]), int(w.q_len[b])
        dead = L == 0 or ql > L
        assert not gpu[b, 0 if dead else ql:].any()
    assert vae4.read_status(ws) == 0
    return rel, mx


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("flags", [0, 1], ids=["tcgen05-path", "mma-sync-path"])
def test_decode_table_is_exact(flags):
    bits, e = vae4.decode_table(flags)
    torch.cuda.synchronize()
    h = bits.cpu().numpy().view(np.float16).astype(np.float64) * 2.0 ** (-e)
    t = oracle.e4m3_table()
    finite = [b for b in range(256) if b not in (0x7F, 0xFF)]
    assert np.array_equal(h[finite], t[finite])
    assert e == (0 if flags == 0 else -8)


# ----------------------------------------------------------- small, full
SMALL = [
    dict(name="tiny", spec="tiny"),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3297, 1025], q_lens=[8, 5], seed=41,
         partition_tokens=512),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3297, 1025], q_lens=[8, 8], seed=42,
         outliers=True),
    dict(B=3, Qmax=1, Hq=6, Hkv=1, D=256, seq_lens=[700, 64, 1], q_lens=[1, 1, 1], seed=43,
         partition_tokens=128),
    dict(B=2, Qmax=16, Hq=6, Hkv=1, D=256, seq_lens=[2000, 16], q_lens=[16, 16], seed=44,
         partition_tokens=320),
    dict(B=2, Qmax=8, Hq=8, Hkv=2, D=128, seq_lens=[1500, 999], q_lens=[8, 3], seed=45,
         partition_tokens=256),
    dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1025], q_lens=[8], seed=46, page=32),
    dict(B=1, Qmax=4, Hq=12, Hkv=2, D=256, seq_lens=[3000], q_lens=[4], seed=47, page=64,
         partition_tokens=1024),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[1000, 8], q_lens=[8, 8], seed=48, page=128),
    # partition boundary +-1 (T = 512): tails of 1 and T-1 tokens
    dict(B=3, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[1025, 1023, 1024], q_lens=[8, 8, 8],
         seed=49, partition_tokens=512),
    # a query whose last partition is empty for the first rows (L = k*T + 3, q = 8)
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[515], q_lens=[8], seed=50,
         partition_tokens=512),
    # padded q slots hold NaN; a dead sequence (L = 0); q_len 0
    dict(B=3, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[900, 0, 33], q_lens=[5, 8, 0], seed=51,
         pad_q_nan=True, partition_tokens=256),
]

# Large and odd page sizes (multiples of 16 tokens): the pages run 1728-,
# 3296- and 3456-token blocks and an 848-token block (PR #560, Purpose and
# Test Plan and Results; PR #524, AI review).  Partitions cut pages in the
# middle.
LARGE_PAGES = [
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[5000, 1729], q_lens=[8, 8], seed=52,
         page=1728, partition_tokens=1024),
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[7000], q_lens=[8], seed=53, page=3296),
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[2000], q_lens=[8], seed=54, page=848,
         partition_tokens=400),
    dict(B=2, Qmax=4, Hq=4, Hkv=2, D=128, seq_lens=[1000, 333], q_lens=[4, 2], seed=55,
         page=48, partition_tokens=176),
    dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[3500], q_lens=[8], seed=56, page=3456),
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.get("name", str(c.get("seed"))))
def test_parity_small(cfg):
    cfg = dict(cfg)
    if "spec" in cfg:
        w = W.generate(cfg["spec"])
    else:
        cfg.pop("name", None)
        w = W.custom("small", **cfg)
    check_full(w)


@pytest.mark.parametrize("cfg", LARGE_PAGES, ids=lambda c: f"page{c['page']}")
@pytest.mark.parametrize("flags", [0, 1], ids=["tcgen05-path", "mma-sync-path"])
def test_parity_large_pages(cfg, flags):
    w = W.custom("pages", **cfg)
    check_full(w, flags=flags)


@pytest.mark.parametrize("cfg", [SMALL[0], SMALL[1], SMALL[4], SMALL[11]],
                         ids=["tiny", "41", "44", "51"])
def test_parity_warp_mma_path(cfg):
    """The legacy mma.sync split kernel (VAE4_FLAG_WARP_MMA) meets the same bar."""
    cfg = dict(cfg)
    w = W.generate(cfg["spec"]) if "spec" in cfg else W.custom(
        "small", **{k: v for k, v in cfg.items() if k != "name"})
    check_full(w, flags=vae4.FLAG_WARP_MMA)


def test_paths_agree():
    """Both split kernels on the same inputs: each within tolerance of the
    oracle, and close to each other (different FP32 summation orders)."""
    w = W.custom("both", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[4000, 2222], q_lens=[8, 6],
                 seed=56, partition_tokens=768)
    a, _ = run_gpu(w)
    b, _ = run_gpu(w, flags=vae4.FLAG_WARP_MMA)
    d = np.abs(a.astype(np.float64) - b.astype(np.float64))
    assert d.max() <= 2e-3


def test_parity_auto_plan():
    w = W.custom("auto", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20000], q_lens=[8],
                 seed=52)
    check_full(w, partition_tokens=0)


# ------------------------------------------------- determinism contracts
def test_relocation_and_repeat_are_bitwise():
    w = W.custom("reloc", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[2600, 1300],
                 q_lens=[8, 8], seed=53, partition_tokens=512)
    a, _ = run_gpu(w)
    a2, _ = run_gpu(w)
    assert np.array_equal(a.view(np.uint16), a2.view(np.uint16))
    perm = np.random.default_rng(5).permutation(w.kv_pages.shape[0])
    kv2 = np.empty_like(w.kv_pages)
    kv2[perm] = w.kv_pages
    w2 = W.Workload(**{**w.__dict__})
    w2.kv_pages = kv2
    w2.block_table = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)],
                              -1).astype(np.int32)
    b, _ = run_gpu(w2)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_exact_fp16_midpoints_round_to_even():
    w = W.midpoint_case()
    gpu, _ = run_gpu(w, partition_tokens=256)
    lo, hi = W.MIDPOINT_VALUES
    h = gpu.shape[-1] // 2
    assert (gpu[0, 0, 0, :h] == np.float16(lo)).all()
    assert (gpu[0, 0, 0, h:] == np.float16(hi)).all()


def test_graph_replay_with_changing_lengths():
    """One captured graph; lengths change between replays (including a zero
    live length and a shortened row)."""
    w = W.custom("graph", B=3, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3000, 1800, 900],
                 q_lens=[8, 4, 1], seed=54, partition_tokens=512)
    q, kv, bt, seq, sc = W.to_device(w)
    out = torch.zeros_like(q)
    ws = vae4.alloc_workspace(3, 6, 1, 8, 256, w.capacity, 512)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=512, max_seq_len=w.capacity)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=512, max_seq_len=w.capacity)
    cases = [([3000, 1800, 900], [8, 4, 1]), ([2999, 0, 900], [8, 4, 1]),
             ([17, 1800, 513], [8, 2, 8]), ([3000, 1800, 900], [8, 4, 1])]
    first = None
    for sl, ql in cases:
        seq.copy_(torch.tensor(np.stack([sl, ql], 1), dtype=torch.int32))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        ref = oracle_full(w, np.array(sl, np.int32), np.array(ql, np.int32))
        compare(got, ref)
        for b in range(3):
            assert not got[b, 0 if sl[b] == 0 else ql[b]:].any()
        if first is None:
            first = got
    assert np.array_equal(first.view(np.uint16), got.view(np.uint16))
    assert vae4.read_status(ws) == 0


# ------------------------------------------------------ status / faults
def test_device_status_bits_and_zeroed_rows():
    w = W.custom("status", B=3, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[600, 500, 400],
                 q_lens=[8, 8, 8], seed=55, partition_tokens=256)
    # sequence 0: a block id past the pool; sequence 2: q_len > L
    w.block_table[0, 3] = w.kv_pages.shape[0] + 7
    gpu, ws = run_gpu(w, q_len=np.array([8, 8, 8], np.int32))
    assert vae4.read_status(ws) & vae4.STATUS_BAD_BLOCK
    assert not gpu[0].any()
    ref = oracle.verify_attn(w.q[1:2], w.kv_pages, w.block_table[1:2], w.seq_len[1:2],
                             w.q_len[1:2], w.kv_scales)
    compare(gpu[1:2], ref)
    vae4.clear_status(ws)
    assert vae4.read_status(ws) == 0
    gpu, ws = run_gpu(w, seq_len=np.array([600, 5, 400], np.int32), ws=ws)
    assert vae4.read_status(ws) & vae4.STATUS_BAD_QLEN
    assert not gpu[1].any()
    vae4.clear_status(ws)
    # a length beyond the launch capacity
    q, kv, bt, seq, sc = W.to_device(w)
    seq[2, 0] = w.capacity + 16
    out = torch.zeros_like(q)
    vae4.verify(q, kv, bt, seq, sc, out, ws, partition_tokens=256, max_seq_len=w.capacity)
    torch.cuda.synchronize()
    assert vae4.read_status(ws) & vae4.STATUS_BAD_LENGTH
    assert not out[2].any()


def test_argument_errors_launch_nothing():
    w = W.generate("tiny")
    q, kv, bt, seq, sc = W.to_device(w)
    ws = vae4.alloc_workspace(1, 2, 1, 8, 64, 1024, 256)
    out = torch.zeros_like(q)
    with pytest.raises(vae4.Vae4Error) as e:
        vae4.verify(q, kv, bt, seq, sc, out, ws[:100], partition_tokens=256)
    assert e.value.code == -8
    qv = torch.zeros(q.numel() + 1, dtype=torch.float16, device="cuda")[1:].view(q.shape)
    with pytest.raises(vae4.Vae4Error) as e:   # a half-offset Q view
        vae4.verify(qv, kv, bt, seq, sc, out, ws, partition_tokens=256)
    assert e.value.code == -5


# E5M2 KV cache (the second FP8 format), default tcgen05 path only
E5M2 = [
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3297, 1025], q_lens=[8, 5], seed=61,
         partition_tokens=512, kv_format="e5m2"),
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[5000, 900], q_lens=[8, 8], seed=62,
         outliers=True, kv_format="e5m2"),
    dict(B=2, Qmax=8, Hq=8, Hkv=2, D=128, seq_lens=[1500, 999], q_lens=[8, 3], seed=63,
         partition_tokens=256, kv_format="e5m2"),
    dict(B=1, Qmax=16, Hq=4, Hkv=1, D=64, seq_lens=[2000], q_lens=[16], seed=64, page=1728,
         kv_format="e5m2"),
]


@pytest.mark.parametrize("cfg", E5M2, ids=lambda c: str(c["seed"]))
def test_parity_e5m2(cfg):
    check_full(W.custom("e5m2", **cfg))


def test_e5m2_decode_table_is_exact():
    bits, e = vae4.decode_table(vae4.FLAG_KV_E5M2)
    torch.cuda.synchronize()
    assert e == 0
    with np.errstate(invalid="ignore"):
        h = bits.cpu().numpy().view(np.float16).astype(np.float64)
    t = oracle.fp8_table("e5m2")
    fin = np.isfinite(t)
    assert np.array_equal(h[fin], t[fin])
    assert np.array_equal(np.isinf(h), np.isinf(t)) and np.array_equal(np.isnan(h), np.isnan(t))
    assert np.array_equal(np.signbit(h[np.isinf(t)]), np.signbit(t[np.isinf(t)]))


def test_e5m2_with_warp_mma_path_is_unsupported():
    w = W.custom("e5m2", **E5M2[0])
    with pytest.raises(vae4.Vae4Error):
        run_gpu(w, flags=vae4.FLAG_KV_E5M2 | vae4.FLAG_WARP_MMA)


def test_short_waits_report_timeout_and_the_context_recovers():
    """Failure path without a GPU fault: with every pipeline wait cut to ~256
    cycles the split kernel aborts (as a stalled pipeline would), drains its
    copies and MMAs, reports VAE4_STATUS_TIMEOUT and the combine writes zero
    rows.  The same workspace then serves a normal call that meets the bar."""
    w = W.custom("abort", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[3000, 1000], q_lens=[8, 8],
                 seed=91)
    tensors = W.to_device(w)
    gpu, ws = run_gpu(w, tensors=tensors, flags=vae4.FLAG_TEST_SHORT_WAITS)
    assert vae4.read_status(ws) & vae4.STATUS_TIMEOUT
    assert np.isfinite(gpu).all() and not gpu.any()
    vae4.clear_status(ws)
    assert vae4.read_status(ws) == 0
    gpu2, _ = run_gpu(w, tensors=tensors, ws=ws)
    compare(gpu2, oracle_full(w))
    assert vae4.read_status(ws) == 0


def test_device_plan_matches_static_plans_on_ragged_batches():
    """The automatic (device-side balanced) plan and two static partition
    lengths on the same ragged inputs: each meets the bar against the oracle."""
    w = W.custom("ragged", B=5, Qmax=8, Hq=6, Hkv=1, D=256,
                 seq_lens=[9000, 17, 3000, 0, 40000], q_lens=[8, 8, 1, 0, 8], seed=92)
    ref = oracle_full(w)
    live = np.zeros(ref.shape, bool)
    for b in range(w.spec.B):
        live[b, :int(w.q_len[b]) if w.seq_len[b] else 0] = True
    for T in (0, 512, 4096):
        gpu, ws = run_gpu(w, partition_tokens=T)
        compare(gpu, ref, live)
        assert not gpu[~live].any()
        assert vae4.read_status(ws) == 0


@pytest.mark.parametrize("B,Hkv,Hq,D,Qmax", [(5, 1, 6, 256, 8), (40, 2, 8, 128, 8),
                                              (100, 1, 6, 64, 8), (12, 1, 6, 128, 16),
                                              (7, 2, 12, 256, 16), (9, 1, 5, 128, 16)])
def test_device_plan_large_batches(B, Hkv, Hq, D, Qmax):
    """Up to 100 sequences, several KV heads, empty sequences and q_len = 0
    among them, up to 16 queries (two row groups, the second busy only for
    some sequences and, at 5 query heads per KV head, never full; lengths far below the launch capacity, so no CTA's
    block-table guess holds): the automatic plan meets the bar against the
    oracle and leaves the status clear."""
    rng = np.random.default_rng(B * 7 + Hkv)
    seq = rng.integers(1, 1500, size=B)
    ql = rng.integers(1, Qmax + 1, size=B)
    seq[::9] = 0
    ql[::9] = 0
    ql[min(5, B - 1)] = 0
    ql = np.minimum(ql, seq)
    w = W.custom("many", B=B, Qmax=Qmax, Hq=Hq, Hkv=Hkv, D=D, seq_lens=seq.tolist(),
                 q_lens=ql.tolist(), seed=93 + B)
    ref = oracle_full(w)
    live = np.zeros(ref.shape, bool)
    for b in range(B):
        live[b, :int(w.q_len[b]) if w.seq_len[b] else 0] = True
    gpu, ws = run_gpu(w, partition_tokens=0)
    compare(gpu, ref, live)
    assert not gpu[~live].any()
    assert vae4.read_status(ws) == 0


@pytest.mark.parametrize("B,Hkv,Hq,Lmax", [(1500, 1, 2, 80), (2100, 1, 2, 80), (1024, 4, 8, 200)])
def test_batches_past_the_combine_caches(B, Hkv, Hq, Lmax):
    """Batches past the combine's shared-memory caches: 1500 and 2100
    sequences run the static plan (more than the device plan takes), the
    latter past the cached lengths, so the combine walks the launch's whole
    capacity and skips dead rows; 1024 sequences x 4 KV heads run the device
    plan with its stream table read from global memory.  Empty sequences
    and q_len = 0 among them; every live row meets the bar, every other row
    is zero."""
    rng = np.random.default_rng(B + Hkv)
    seq = rng.integers(1, Lmax, size=B)
    ql = rng.integers(0, 3, size=B)
    seq[::7] = 0
    ql = np.minimum(ql, seq)
    w = W.custom("huge", B=B, Qmax=2, Hq=Hq, Hkv=Hkv, D=64, seq_lens=seq.tolist(),
                 q_lens=ql.tolist(), seed=97 + B)
    ref = oracle_full(w)
    live = np.zeros(ref.shape, bool)
    for b in range(B):
        live[b, :int(w.q_len[b]) if w.seq_len[b] else 0] = True
    gpu, ws = run_gpu(w, partition_tokens=0)
    compare(gpu, ref, live)
    assert not gpu[~live].any()
    assert vae4.read_status(ws) == 0


@pytest.mark.parametrize("L", [1, 700, 5000, 12345, 20000])
def test_single_sequence_auto_plan_below_capacity(L):
    """One sequence in a launch sized for 20000 tokens: the automatic plan
    spreads its L tokens over all of the launch's partitions; the result
    meets the bar against the oracle at every length."""
    w = W.custom("one", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[L], q_lens=[min(8, L)],
                 capacity=20000, seed=94)
    ref = oracle_full(w)
    gpu, ws = run_gpu(w, partition_tokens=0)
    live = np.zeros(ref.shape, bool)
    live[0, :min(8, L)] = True
    compare(gpu, ref, live)
    assert not gpu[~live].any()
    assert vae4.read_status(ws) == 0


# ------------------------------------------- unwritten pool slots past L
def _poison_past_l(w, codes):
    """Fill every pool byte of the slots past L in each sequence's last page
    (K and V, all heads) with the given codes in turn: slots a real cache
    may never have written.  The oracle reads keys < L only."""
    page = w.spec.page
    k = 0
    for b in range(w.spec.B):
        L = int(w.seq_len[b])
        if L == 0 or L % page == 0:
            continue
        phys = int(w.block_table[b, (L - 1) // page])
        for slot in range(L % page, page):
            w.kv_pages[phys, :, :, slot, :] = codes[k % len(codes)]
            k += 1
    assert k > 0
    return w


@pytest.mark.parametrize("cfg", [
    dict(B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[1000, 37], q_lens=[8, 8], seed=70,
         partition_tokens=256),
    dict(B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[20001], q_lens=[8], seed=71),
    dict(B=3, Qmax=16, Hq=6, Hkv=1, D=256, seq_lens=[5003, 999, 70], q_lens=[16, 8, 1],
         seed=72),
    dict(B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1000], q_lens=[8], seed=73, page=48,
         partition_tokens=512),
], ids=["T256", "auto-one", "auto-batch", "page48"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_nan_and_inf_codes_past_the_length_do_not_leak(cfg, fmt):
    """A masked key has P = 0, but 0 * NaN is NaN: the split kernel must not
    feed the bytes of unwritten slots past L into the value product."""
    w = W.custom("poison", kv_format=fmt, **cfg)
    codes = [0x7F, 0xFF] if fmt == "e4m3" else [0x7C, 0xFC, 0x7F, 0xFF]
    check_full(_poison_past_l(w, codes))


# --------------------------------------------- the plain 8-argument call
def test_plain_entry_point_matches_ex_with_defaults():
    """verify_attn_e4m3 (the eight-argument form) is verify_attn_e4m3_ex with
    default options: automatic plan, capacity = block-table columns x page,
    1/sqrt(D).  Same bits, and within the bar against the oracle."""
    import ctypes
    lib = vae4.load()
    w = W.custom("plain", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[7000, 3297],
                 q_lens=[8, 5], seed=74)
    q, kv, bt, seq, sc = W.to_device(w)
    s = w.spec
    cap = w.block_table.shape[1] * s.page
    ws = vae4.alloc_workspace(s.B, s.Hq, s.Hkv, s.Qmax, s.D, cap, 0)
    outs = []
    for plain in (True, False):
        out = torch.full_like(q, float("nan"))
        d = [vae4.describe(t) for t in (q, kv, bt, seq, sc, out, ws)]
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        if plain:
            rc = lib.verify_attn_e4m3(*[ctypes.byref(x) for x in d], st)
        else:
            rc = lib.verify_attn_e4m3_ex(*[ctypes.byref(x) for x in d], st, None)
        assert rc == 0
        torch.cuda.synchronize()
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint16), outs[1].view(np.uint16))
    compare(outs[0], oracle_full(w))
    assert vae4.read_status(ws) == 0


# ---------------------------------------- high/residual P (hilo_pv option)
def _cfg_workload(cfg):
    cfg = dict(cfg)
    if "spec" in cfg:
        return W.generate(cfg["spec"])
    cfg.pop("name", None)
    return W.custom("hilo", **cfg)


@pytest.mark.parametrize("cfg", SMALL + LARGE_PAGES + E5M2,
                         ids=lambda c: c.get("name", str(c.get("seed"))))
def test_parity_hilo(cfg):
    """The high/residual split of P (PR #524, Historical R6 purpose and
    evidence) meets the same bar on every small, large-page and E5M2 case."""
    check_full(_cfg_workload(cfg), hilo_pv=True)


@pytest.mark.parametrize("T", [0, 512])
def test_hilo_lowers_the_error(T):
    """P with ~22 significant bits instead of 11: the relative L2 error
    against the FP64 oracle drops, and the step stays bitwise repeatable."""
    w = W.custom("hilo_err", B=2, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[30000, 9000],
                 q_lens=[8, 8], seed=75, outliers=True)
    ref = oracle_full(w)
    plain, _ = run_gpu(w, partition_tokens=T)
    hilo, _ = run_gpu(w, partition_tokens=T, hilo_pv=True)
    hilo2, _ = run_gpu(w, partition_tokens=T, hilo_pv=True)
    assert np.array_equal(hilo.view(np.uint16), hilo2.view(np.uint16))
    r_plain, _ = compare(plain, ref)
    r_hilo, _ = compare(hilo, ref)
    # the FP16 output rounding alone leaves about 1.5e-4 (a uniform
    # half-ulp error); the P rounding adds on top of it without the split
    r_round = np.linalg.norm(ref.astype(np.float16).astype(np.float64) - ref) / \
        np.linalg.norm(ref)
    print(f"rel-L2 plain {r_plain:.3e} hilo {r_hilo:.3e} fp16 rounding floor {r_round:.3e}")
    assert r_hilo < r_plain
    assert r_hilo < 1.15 * r_round


def test_hilo_with_warp_mma_is_unsupported():
    w = _cfg_workload(SMALL[1])
    with pytest.raises(vae4.Vae4Error) as e:
        run_gpu(w, flags=vae4.FLAG_WARP_MMA, hilo_pv=True)
    assert e.value.code == -6
