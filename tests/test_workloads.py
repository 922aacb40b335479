"""The seeded input generator: reproducible, chunk-invariant, well formed."""
import numpy as np

import workloads as W


def test_reproducible_and_chunk_invariant(monkeypatch):
    s = W.Spec("t", B=2, Qmax=8, Hq=6, Hkv=1, D=32, seq_lens=[30000, 7700],
               q_lens=[8, 3], seed=5, outliers=True)
    a = W.generate(s)
    monkeypatch.setattr(W, "_CHUNK_BLOCKS", 1)  # more chunks, no caching
    b = W.generate(s)
    for f in ("q", "kv_pages", "block_table", "seq_len", "q_len", "kv_scales"):
        assert np.array_equal(getattr(a, f), getattr(b, f), equal_nan=True), f


def test_block_table_and_scales_well_formed():
    w = W.custom(B=3, Qmax=4, Hq=4, Hkv=2, D=16, seq_lens=[100, 17, 1],
                 q_lens=[4, 2, 1], seed=3)
    n = w.kv_pages.shape[0]
    live = []
    for b in range(3):
        need = -(-int(w.seq_len[b]) // 16)
        assert (w.block_table[b, :need] >= 0).all() and (w.block_table[b, :need] < n).all()
        assert (w.block_table[b, need:] == -1).all()
        live += list(w.block_table[b, :need])
    assert len(set(live)) == len(live)            # no page shared
    assert n >= 1.25 * len(live)                  # 25 % spare pages
    assert w.kv_scales.dtype == np.float32 and (w.kv_scales > 0).all()
    # saturating quantiser: every byte is a finite E4M3 code
    assert not np.isin(w.kv_pages, [0x7F, 0xFF]).any()


def test_named_workloads_shapes():
    t = W.generate("tiny")
    assert t.q.shape == (1, 8, 2, 64) and t.capacity == 1024
    assert t.spec.partition_tokens == 256 and t.kv_bytes == 2 * 64 * 1024
    r = W.spec("rag")
    assert r.B == 16 and r.Qmax == 16 and len(r.replays) == 4
    L0 = r.replays[0][0]
    assert L0[0] == 1025 and L0[1] == 3297
    assert (r.replays[3][0] == 0).sum() >= 1
    assert set(int(x) for x in r.replays[0][1]) == {1, 8, 16}
    assert all((1024 <= v[0][2:]).all() and (v[0] <= 262144).all() for v in r.replays[:3])
