"""Seeded synthetic inputs for paged GQA verify attention over E4M3 pages.

This module holds no part of the method's arithmetic: it draws random numbers,
quantises them into the stored E4M3 cache format and lays out the paged pool,
block table and length arrays.  Both the oracle and the CUDA path consume
what it produces; neither is imported here.

Recipe (the workloads of the 1Cat-vLLM pages, made synthetic):
  * queries  Q ~ N(0, 1) rounded to fp16, layout [B][Qmax][Hq][D];
  * keys/values X ~ N(0, 1) in fp32; the long-context workload adds rare
    outliers (0.1 % of values set to +-30, i.e. 30 sigma, random sign);
  * per KV head and separately for K and V, s = fp32(amax / 448) with amax
    over every token of that head in the pool, then y = fp32(x / s) clamped
    to +-448 and rounded to nearest-even onto the E4M3 grid (saturating
    quantisation; an amax that lands just above 448 after the fp32 division
    saturates);
  * 16-token pages in a pool with 25 % spare pages; each sequence's logical
    pages map to physical pages drawn from a seeded permutation, so pages
    are relocated and interleaved between sequences;
  * the q_len queries of a sequence are its last q_len positions (the causal
    verify tail); query slots beyond q_len are padding.

Generators are NumPy PCG64 streams keyed by (seed, tensor, head, chunk), so a
workload is reproducible bit for bit on any machine, whatever the chunking.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

E4M3_MAX = np.float32(448.0)
E5M2_MAX = np.float32(57344.0)
PAGE = 16
GEN_PAGES = 256      # 16-token pages per random-stream block (part of the recipe)


def gen_pages(page: int) -> int:
    """Pages per random-stream block: 4096 tokens' worth (256 pages of 16
    tokens; fewer, larger pages for larger page sizes, at least one)."""
    return max(1, GEN_PAGES * 16 // page)
_CHUNK_BLOCKS = 8    # blocks per processing chunk (memory only)


# ----------------------------------------------------------------------------
# E4M3 quantiser (input generation: produces the bytes the cache stores)
# ----------------------------------------------------------------------------
def quantize_e4m3(y: np.ndarray) -> np.ndarray:
    """fp32 -> E4M3FN bytes, round-to-nearest-even, saturating at +-448.

    Normal range (|y| >= 2^-6): round the fp32 significand to 3 bits with the
    usual add-half-minus-one-plus-lsb trick, then re-bias the exponent
    (fp32 bias 127 -> E4M3 bias 7).  Subnormal range: round |y| * 2^9 to an
    integer with numpy's half-to-even rint; 8 lands on the smallest normal.
    """
    y = np.asarray(y, dtype=np.float32)
    y = np.clip(y, -E4M3_MAX, E4M3_MAX)
    sign = (y.view(np.uint32) >> 31).astype(np.uint8)
    a = np.abs(y)
    normal = a >= np.float32(2.0 ** -6)
    u = a.view(np.uint32)
    lsb = (u >> 20) & 1
    ur = (u + np.uint32(0x7FFFF) + lsb) & np.uint32(0xFFF00000)
    e4 = ((ur >> 23).astype(np.int32) - 127 + 7)
    mant = ((ur >> 20) & 7).astype(np.int32)
    code_n = (e4 << 3) | mant
    code_s = np.rint(a * np.float32(512.0)).astype(np.int32)
    code = np.where(normal, code_n, code_s).astype(np.uint8)
    return code | (sign << 7)


def quantize_e5m2(y: np.ndarray) -> np.ndarray:
    """fp32 -> E5M2 bytes, round-to-nearest-even, saturating at +-57344.

    Normal range (|y| >= 2^-14): round the fp32 significand to 2 bits the
    same way as for E4M3 and re-bias the exponent (127 -> 15).  Subnormal
    range: round |y| * 2^16 to an integer (half to even); 4 lands on the
    smallest normal.
    """
    y = np.asarray(y, dtype=np.float32)
    y = np.clip(y, -E5M2_MAX, E5M2_MAX)
    sign = (y.view(np.uint32) >> 31).astype(np.uint8)
    a = np.abs(y)
    normal = a >= np.float32(2.0 ** -14)
    u = a.view(np.uint32)
    lsb = (u >> 21) & 1
    ur = (u + np.uint32(0xFFFFF) + lsb) & np.uint32(0xFFE00000)
    e5 = ((ur >> 23).astype(np.int32) - 127 + 15)
    mant = ((ur >> 21) & 3).astype(np.int32)
    code_n = (e5 << 2) | mant
    code_s = np.rint(np.minimum(a, np.float32(2.0 ** -14)) * np.float32(65536.0)).astype(np.int32)
    code = np.where(normal, code_n, code_s).astype(np.uint8)
    return code | (sign << 7)


def quantize(y: np.ndarray, kv_format: str = "e4m3") -> np.ndarray:
    return quantize_e5m2(y) if kv_format == "e5m2" else quantize_e4m3(y)


def fp8_scale(amax: np.float32, kv_format: str = "e4m3") -> np.float32:
    """Per-head scale s = fp32(amax / largest finite value); zero amax -> 1."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / (E5M2_MAX if kv_format == "e5m2" else E4M3_MAX))


def e4m3_scale(amax: np.float32) -> np.float32:
    """Per-head scale s = fp32(amax / 448); a zero amax gives s = 1."""
    amax = np.float32(amax)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / E4M3_MAX)


# ----------------------------------------------------------------------------
# Workload specification
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class Spec:
    name: str
    B: int
    Qmax: int
    Hq: int
    Hkv: int
    D: int
    seq_lens: list            # replay 0 lengths (L, including the q tail)
    q_lens: list
    seed: int
    page: int = PAGE
    outliers: bool = False
    partition_tokens: int = 0  # 0 = the library's automatic plan
    capacity: int = 0          # max_seq_len the launch is sized for (0 = max L)
    replays: list = dataclasses.field(default_factory=list)  # [(seq_lens, q_lens)]
    pad_q_nan: bool = False    # fill padded query slots with NaN
    q_from: tuple | None = None  # (spec name, row slice) to reuse queries
    kv_format: str = "e4m3"    # stored FP8 format: "e4m3" or "e5m2"


@dataclasses.dataclass
class Workload:
    spec: Spec
    q: np.ndarray            # float16 [B][Qmax][Hq][D]
    kv_pages: np.ndarray     # uint8 [n_pages][2][Hkv][page][D]
    block_table: np.ndarray  # int32 [B][max_pages]
    seq_len: np.ndarray      # int32 [B]
    q_len: np.ndarray        # int32 [B]
    kv_scales: np.ndarray    # float32 [Hkv][2]
    sm_scale: float
    capacity: int
    replays: list            # [(seq_len int32[B], q_len int32[B])], replay 0 first

    @property
    def kv_bytes(self) -> int:
        """Algorithmic KV bytes of replay 0: K and V, 1 byte per element."""
        return int(2 * self.spec.Hkv * self.spec.D * int(self.seq_len.sum()))


def _rag_lengths(rng: np.random.Generator, B: int) -> np.ndarray:
    lo, hi = math.log(1024), math.log(262144)
    L = np.rint(np.exp(rng.uniform(lo, hi, size=B))).astype(np.int64)
    L[0], L[1] = 1025, 3297
    return L.astype(np.int32)


def spec(name: str) -> Spec:
    """Named workloads.  Seeds 0..4 = tiny, tp4, long, rag, tp2."""
    if name == "tiny":
        return Spec("tiny", B=1, Qmax=8, Hq=2, Hkv=1, D=64, seq_lens=[1024],
                    q_lens=[8], seed=0, partition_tokens=256)
    if name == "tp4":
        return Spec("tp4", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[131072],
                    q_lens=[8], seed=1)
    if name == "long":
        return Spec("long", B=1, Qmax=8, Hq=6, Hkv=1, D=256, seq_lens=[262144],
                    q_lens=[8], seed=2, outliers=True)
    if name == "long_q1":
        return Spec("long_q1", B=1, Qmax=1, Hq=6, Hkv=1, D=256,
                    seq_lens=[262144], q_lens=[1], seed=2, outliers=True,
                    q_from=("long", 7))
    if name == "rag":
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([3, 99])))
        B = 16
        vecs = [_rag_lengths(rng, B) for _ in range(3)]
        ql = np.array([(1, 8, 16)[b % 3] for b in range(B)], dtype=np.int32)
        zero = vecs[0].copy()
        zero[5] = 0
        replays = [(v, ql) for v in vecs] + [(zero, ql)]
        return Spec("rag", B=B, Qmax=16, Hq=6, Hkv=1, D=256,
                    seq_lens=list(vecs[0]), q_lens=list(ql), seed=3,
                    capacity=262144, replays=replays, pad_q_nan=True)
    if name == "tp2":
        return Spec("tp2", B=4, Qmax=8, Hq=12, Hkv=2, D=256,
                    seq_lens=[262144] * 4, q_lens=[8] * 4, seed=4)
    raise KeyError(name)


NAMES = ("tiny", "tp4", "long", "long_q1", "rag", "tp2")


def _rng(*key) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _kv_block(seed: int, kv_sel: int, h: int, block: int, page: int, D: int,
              outliers: bool) -> np.ndarray:
    """fp32 K or V values of pages [block*gp, (block+1)*gp), gp = gen_pages(page)."""
    rng = _rng(seed, 1000 + kv_sel, h, block)
    shape = (gen_pages(page), page, D)
    x = rng.standard_normal(shape, dtype=np.float32)
    if outliers:
        # one uniform draw: u < 1e-3 marks an outlier, u < 5e-4 makes it negative
        u = rng.random(shape, dtype=np.float32)
        x = np.where(u < np.float32(1e-3),
                     np.where(u < np.float32(5e-4), np.float32(-30.0), np.float32(30.0)),
                     x)
    return x


def _kv_chunk(seed, kv_sel, h, chunk, n_pages, page, D, outliers):
    """Pages [chunk*_CHUNK_BLOCKS*gp, ...) of the pool, n_pages of them."""
    b0 = chunk * _CHUNK_BLOCKS
    nb = -(-n_pages // gen_pages(page))
    x = np.concatenate([_kv_block(seed, kv_sel, h, b0 + k, page, D, outliers)
                        for k in range(nb)])
    return x[:n_pages]


def generate(s: Spec | str) -> Workload:
    if isinstance(s, str):
        s = spec(s)
    B, Qmax, Hq, Hkv, D, page = s.B, s.Qmax, s.Hq, s.Hkv, s.D, s.page
    assert Hq % Hkv == 0
    replays = s.replays or [(np.asarray(s.seq_lens, np.int32),
                             np.asarray(s.q_lens, np.int32))]
    replays = [(np.asarray(a, np.int32), np.asarray(b, np.int32)) for a, b in replays]
    cap_rows = np.max(np.stack([r[0] for r in replays]), axis=0)  # per sequence
    capacity = s.capacity or int(cap_rows.max())
    max_pages = max(1, -(-capacity // page))
    need = [-(-int(c) // page) for c in cap_rows]
    total_need = int(sum(need))
    n_pages = max(total_need + 1, -(-total_need * 5 // 4))

    # physical placement: a seeded permutation of the pool
    prng = _rng(s.seed, 7)
    perm = prng.permutation(n_pages).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        bt[b, :need[b]] = perm[k:k + need[b]]
        k += need[b]

    # K/V: per (K|V, head) two passes over chunks: amax, then quantise
    kv = np.empty((n_pages, 2, Hkv, page, D), dtype=np.uint8)
    scales = np.empty((Hkv, 2), dtype=np.float32)
    chunk_pages = _CHUNK_BLOCKS * gen_pages(page)
    n_chunks = -(-n_pages // chunk_pages)
    for sel in range(2):
        for h in range(Hkv):
            amax = np.float32(0.0)
            cache = []
            for c in range(n_chunks):
                n = min(chunk_pages, n_pages - c * chunk_pages)
                x = _kv_chunk(s.seed, sel, h, c, n, page, D, s.outliers)
                amax = max(amax, np.float32(np.abs(x).max()))
                if n_chunks <= 4:
                    cache.append(x)
            sc = fp8_scale(amax, s.kv_format)
            scales[h, sel] = sc
            for c in range(n_chunks):
                n = min(chunk_pages, n_pages - c * chunk_pages)
                x = cache[c] if cache else _kv_chunk(s.seed, sel, h, c, n, page, D,
                                                     s.outliers)
                kv[c * chunk_pages:c * chunk_pages + n, sel, h] = \
                    quantize(x / sc, s.kv_format)

    # queries
    if s.q_from is not None:
        src_name, row = s.q_from
        src = spec(src_name)
        qsrc = _rng(src.seed, 5).standard_normal(
            (src.B, src.Qmax, src.Hq, src.D), dtype=np.float32).astype(np.float16)
        q = np.ascontiguousarray(qsrc[:, row:row + 1])
    else:
        q = _rng(s.seed, 5).standard_normal((B, Qmax, Hq, D),
                                            dtype=np.float32).astype(np.float16)
    seq_len, q_len = replays[0]
    if s.pad_q_nan:
        for b in range(B):
            q[b, q_len[b]:] = np.float16(np.nan)
    return Workload(spec=s, q=q, kv_pages=kv, block_table=bt,
                    seq_len=seq_len.copy(), q_len=q_len.copy(), kv_scales=scales,
                    sm_scale=1.0 / math.sqrt(D), capacity=capacity,
                    replays=replays)


def custom(name: str = "custom", **kw) -> Workload:
    """A workload from explicit parameters (same recipe), for tests."""
    kw.setdefault("seed", 11)
    return generate(Spec(name=name, **kw))


def sample_rows(w: Workload, n: int, seed: int = 0, seq_len=None, q_len=None):
    """n distinct live (b, i, hq) triples, always including each sequence's
    first and last live query of its first and last q head."""
    sl = w.seq_len if seq_len is None else seq_len
    ql = w.q_len if q_len is None else q_len
    live = [(b, i, hq) for b in range(w.spec.B) if sl[b] > 0 and ql[b] <= sl[b]
            for i in range(int(ql[b])) for hq in range(w.spec.Hq)]
    must = set()
    for b in range(w.spec.B):
        if sl[b] > 0 and 0 < ql[b] <= sl[b]:
            for i in (0, int(ql[b]) - 1):
                for hq in (0, w.spec.Hq - 1):
                    must.add((b, i, hq))
    rest = [r for r in live if r not in must]
    rng = _rng(seed, 31337)
    k = max(0, min(len(rest), n - len(must)))
    pick = [rest[j] for j in rng.choice(len(rest), size=k, replace=False)] if k else []
    rows = sorted(must) + pick
    return np.asarray(rows, dtype=np.int32)


# Exact outputs of midpoint_case(): 0.25 + 2^-13 (d < D/2) and 0.25 + 3*2^-13
# (d >= D/2), each the midpoint of two adjacent fp16 values.
MIDPOINT_VALUES = (0.25 + 2.0 ** -13, 0.25 + 3 * 2.0 ** -13)


def midpoint_case(n: int = 1024, D: int = 64) -> Workload:
    """One query, zero Q (every score equal), n keys.  Even keys hold V bytes
    0x78 (256), odd keys 0x20 (0.125) in columns 0..D/2-1 and 0x2C (0.375) in
    columns D/2..D-1; s_V = 2^-9.  The mean over all n keys is then
    (256 + 0.125) / 2 * 2^-9 and (256 + 0.375) / 2 * 2^-9: exact fp16
    midpoints (the first rounds down to even, the second up)."""
    w = custom("midpoint", B=1, Qmax=1, Hq=1, Hkv=1, D=D, seq_lens=[n],
               q_lens=[1], seed=9)
    w.q[:] = 0
    w.kv_scales[:, 1] = np.float32(2.0 ** -9)
    bt = w.block_table[0]
    for j in range(n):
        p, s = bt[j // w.spec.page], j % w.spec.page
        if j % 2 == 0:
            w.kv_pages[p, 1, 0, s, :] = 0x78
        else:
            w.kv_pages[p, 1, 0, s, :D // 2] = 0x20
            w.kv_pages[p, 1, 0, s, D // 2:] = 0x2C
    return w


def relocate(w: Workload, seed: int) -> Workload:
    """The same logical cache with every physical page moved to a seeded
    random place in the pool: the pages and the block table are permuted
    together, so every sequence reads the same bytes from other addresses."""
    perm = _rng(seed, 4242).permutation(w.kv_pages.shape[0]).astype(np.int32)
    kv = np.empty_like(w.kv_pages)
    kv[perm] = w.kv_pages  # page p moves to perm[p]
    bt = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1)
    return dataclasses.replace(w, kv_pages=kv, block_table=bt.astype(np.int32))


PAD_BYTE = 0x7F  # an E4M3 NaN code: padding that is read would show up as NaN


@dataclasses.dataclass
class TokenMajorCache:
    """The workload's cache in the token-major layout of the pages:
    separate K and V caches [n_pages][page][Hkv][D] (page = the block size),
    token stride Hkv * D + token_pad bytes, head stride D, page stride
    page * token stride + page_pad; d contiguous.  Padding bytes hold
    PAD_BYTE.  K and V live in buffers of their own."""
    k_buf: np.ndarray
    v_buf: np.ndarray
    shape: tuple    # (n_pages, page, Hkv, D)
    strides: tuple  # bytes (page, token, head, 1)

    def views(self):
        """(K, V) as numpy strided views into the buffers."""
        st = np.lib.stride_tricks.as_strided
        return (st(self.k_buf, self.shape, self.strides, writeable=False),
                st(self.v_buf, self.shape, self.strides, writeable=False))

    def to_device(self, device="cuda"):
        """(K, V) as torch strided views into device copies of the buffers."""
        import torch
        out = []
        for buf in (self.k_buf, self.v_buf):
            d = torch.from_numpy(buf).to(device)
            out.append(torch.as_strided(d, self.shape, self.strides, 0))
        return tuple(out)


def token_major(w: Workload, token_pad: int = 0, page_pad: int = 0) -> TokenMajorCache:
    """The same logical K/V bytes as w.kv_pages, laid out token-major with a
    padded token stride (e.g. the pages' [1,848,1,256] block with a 264-byte
    token stride: token_pad = 8)."""
    n_pages, _, Hkv, page, D = w.kv_pages.shape
    tok = Hkv * D + token_pad
    pst = page * tok + page_pad
    shape, strides = (n_pages, page, Hkv, D), (pst, tok, D, 1)
    bufs = []
    for sel in range(2):
        buf = np.full(n_pages * pst, PAD_BYTE, dtype=np.uint8)
        view = np.lib.stride_tricks.as_strided(buf, shape, strides)
        view[...] = w.kv_pages[:, sel].transpose(0, 2, 1, 3)  # [n][Hkv][page][D] -> [n][page][Hkv][D]
        bufs.append(buf)
    return TokenMajorCache(bufs[0], bufs[1], shape, strides)


def to_device(w: Workload, device="cuda", seq_len=None, q_len=None):
    """The workload's inputs as device tensors for the library:
    (q, kv_pages, block_table, seq_lens [B][2] = (L, q_len), kv_scales)."""
    import torch
    sl = w.seq_len if seq_len is None else seq_len
    ql = w.q_len if q_len is None else q_len
    seq = np.stack([np.asarray(sl, np.int32), np.asarray(ql, np.int32)], axis=1)
    return (torch.from_numpy(w.q).to(device),
            torch.from_numpy(w.kv_pages).to(device),
            torch.from_numpy(w.block_table).to(device),
            torch.from_numpy(np.ascontiguousarray(seq)).to(device),
            torch.from_numpy(w.kv_scales).to(device))
