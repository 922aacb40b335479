"""The C-ABI library on the host: it loads, exports every declared symbol,
reports its ABI revision, plans partitions, sizes workspaces and rejects bad
arguments before touching CUDA.  No compute call is made here."""
import ctypes
import json
import os
import re

import pytest

import fp8_paged_attention_e4m3_gb300 as vae4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "verify_attn_e4m3.h")
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "page_sizes.json")))


@pytest.fixture(scope="module")
def lib():
    return vae4.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(verify_attn_e4m3\w*)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert declared and set(declared) == set(vae4.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version_and_strerror(lib):
    assert lib.verify_attn_e4m3_abi_version() == vae4.ABI_VERSION
    for code, name in vae4.ERRORS.items():
        assert vae4.strerror(code) and vae4.strerror(code) != "unknown error", name
    assert vae4.strerror(-999) == "unknown error"


@pytest.mark.parametrize("B,Hkv,cap,sms,T,P", [
    (1, 1, 262144, 152, 1728, 152),   # long context: one partition per SM
    (1, 1, 131072, 152, 864, 152),    # TP4 shard
    (4, 2, 262144, 152, 13808, 19),   # TP2 shard: 8 units x 19 partitions
    (1, 1, 1024, 152, 64, 16),        # never below 64 tokens
    (200, 1, 5000, 152, 5008, 1),     # more units than SMs: one partition each
])
def test_auto_plan(B, Hkv, cap, sms, T, P):
    assert vae4.plan(B, Hkv, cap, 0, sms) == (T, P)
    assert B * Hkv * P <= max(sms, B * Hkv)


def test_explicit_plan_and_errors():
    assert vae4.plan(1, 1, 1024, 256, 152) == (256, 4)   # tiny: 4 partitions
    assert vae4.plan(1, 1, 1025, 256, 152) == (256, 5)
    for bad in (-16, 8, 100):
        with pytest.raises(vae4.Vae4Error):
            vae4.plan(1, 1, 1024, bad, 152)
    assert vae4.plan(1, 1, 131072, 16, 152) == (16, 8192)
    with pytest.raises(vae4.Vae4Error):             # more than 8192 partitions
        vae4.plan(1, 1, 262144, 16, 152)


def test_workspace_matches_the_pages_max_sum_layout():
    g = GOLD["max_sum_workspace"]
    P, q, G, D = g["partitions"], g["queries"], g["group_heads"], g["head_dim"]
    T = 3296  # 80 partitions of 3296 tokens cover 262144 (the pages' page3296)
    assert vae4.plan(1, 1, 262144, T, 80) == (T, P)
    n = vae4.workspace_bytes(1, G, 1, q, D, 262144, T, 80)
    ml = 1
    for s in g["new_shape"]:
        ml *= s
    ml *= g["element_bytes"]
    assert ml - g["delta_bytes"] == 80 * 8 * 6 * 4            # the old [80,8,6]
    o = P * q * G * D * 4                                     # FP32 unnormalised PV
    # status + (max,sum) + PV + (first slot, partitions) of the one stream
    assert n == 256 + ml + o + 8
    qc = GOLD["q_copy"]
    assert qc["shape"][0] * qc["shape"][1] * qc["shape"][2] * qc["element_bytes"] == qc["max_bytes"]


def test_workspace_of_the_device_plan():
    """Automatic plans of a batch (1 < B <= 1024) size the partials for the
    device-side plan's grid, max(B*Hkv*P, SMs, B*Hkv*row groups) slots, plus
    8 bytes per (sequence, KV head) stream for the stream table; one
    sequence and explicit partition lengths keep the static B*Hkv*P."""
    def layout(slots, rows_pad, D, streams):
        al = lambda x: (x + 255) // 256 * 256
        o_off = al(256 + slots * rows_pad * 2 * 4)
        return al(o_off + slots * rows_pad * D * 4) + streams * 8

    # ragged shape: 16 sequences, q16 x GQA6 = 96 rows in two row groups of 48
    B, Hq, Hkv, Qmax, D, cap = 16, 6, 1, 16, 256, 262144
    T, P = vae4.plan(B, Hkv, cap, 0, 152)
    slots = max(B * Hkv * P, 152, B * Hkv * 2)
    assert vae4.workspace_bytes(B, Hq, Hkv, Qmax, D, cap, 0, 152) == layout(slots, 96, D, B * Hkv)
    # more streams than SMs: the grid covers one CTA per (stream, row group)
    B, Hkv, Hq = 100, 2, 12
    T, P = vae4.plan(B, Hkv, cap, 0, 152)
    slots = max(B * Hkv * P, 152, B * Hkv * 2)
    assert vae4.workspace_bytes(B, Hq, Hkv, Qmax, D, cap, 0, 152) == layout(slots, 96, D, B * Hkv)
    # one sequence (length-derived T on the static grid), an explicit T, and a
    # batch above the device plan's limit: the static slot count
    for B, T_req in ((1, 0), (16, 2048), (1025, 0)):
        T, P = vae4.plan(B, 1, cap, T_req, 152)
        assert vae4.workspace_bytes(B, 6, 1, 8, D, cap, T_req, 152) == layout(B * P, 48, D, B)


def test_workspace_errors():
    with pytest.raises(vae4.Vae4Error):
        vae4.workspace_bytes(1, 6, 4, 8, 256, 1000, 0, 152)   # GQA mismatch
    with pytest.raises(vae4.Vae4Error):
        vae4.workspace_bytes(1, 6, 1, 8, 96, 1000, 0, 152)    # unsupported D
    with pytest.raises(vae4.Vae4Error):
        vae4.workspace_bytes(1, 12, 1, 16, 256, 1000, 0, 152)  # 192 rows > 96
    assert vae4.workspace_bytes(1, 6, 1, 16, 256, 1000, 0, 152) > 0  # q16 x G6 = 96


# -------------------------------------------------- argument validation
FAKE = 0x100000  # never dereferenced: every case below fails validation


def _t(dtype, shape, strides=None, data=FAKE):
    d = vae4.Tensor()
    d.data = data
    d.dtype = dtype
    d.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for k, (s, st) in enumerate(zip(shape, strides)):
        d.shape[k] = s
        d.stride[k] = st
    return d


def _args(**over):
    B, Q, Hq, Hkv, D, page, npg, mp = 1, 8, 6, 1, 256, 16, 80, 64
    a = dict(
        q=_t(vae4.VAE4_F16, [B, Q, Hq, D]),
        kv=_t(vae4.VAE4_U8, [npg, 2, Hkv, page, D]),
        bt=_t(vae4.VAE4_I32, [B, mp]),
        seq=_t(vae4.VAE4_I32, [B, 2]),
        sc=_t(vae4.VAE4_F32, [Hkv, 2]),
        out=_t(vae4.VAE4_F16, [B, Q, Hq, D], data=FAKE * 2),
        ws=_t(vae4.VAE4_U8, [1 << 24], data=FAKE * 4),
    )
    a.update(over)
    return a


def _call(lib, a, opt=None):
    o = opt or vae4.Options(0.0, 0, 0, 152, 0)
    return lib.verify_attn_e4m3_ex(*[ctypes.byref(a[k]) for k in
                                     ("q", "kv", "bt", "seq", "sc", "out", "ws")],
                                   None, ctypes.byref(o))


@pytest.mark.parametrize("over,code", [
    (dict(q=_t(vae4.VAE4_F32, [1, 8, 6, 256])), -2),
    (dict(q=_t(vae4.VAE4_F16, [1, 8, 6, 96])), -3),                 # out shape differs
    (dict(q=_t(vae4.VAE4_F16, [1, 8, 6, 256], data=FAKE + 2)), -5), # half-offset view
    (dict(q=_t(vae4.VAE4_F16, [1, 8, 6, 256], [12288, 1536, 256, 2])), -4),
    (dict(q=_t(vae4.VAE4_F16, [1, 8, 6, 256], [12290, 1536, 256, 1])), -4),
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 1, 24, 256])), -6),           # page 24
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 1, 40, 256])), -6),           # page 40
    # pages that are multiples of 16 pass the page check (and then fail on
    # the head grouping, 6 q heads over 4 KV heads)
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 4, 48, 256])), -7),           # page 48
    (dict(kv=_t(vae4.VAE4_U8, [8, 2, 4, 3296, 256])), -7),          # page 3296
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 4, 16, 256])), -7),           # 6 % 4
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 1, 16, 256], data=FAKE + 8)), -5),
    (dict(kv=_t(vae4.VAE4_U8, [80, 2, 1, 16, 256], [8448, 4224, 4224, 264, 1])), -4),
    (dict(bt=_t(vae4.VAE4_F32, [1, 64])), -2),
    (dict(bt=_t(vae4.VAE4_I32, [2, 64])), -3),
    (dict(seq=_t(vae4.VAE4_I32, [1, 3])), -3),
    (dict(sc=_t(vae4.VAE4_F32, [2, 2])), -3),
    (dict(ws=_t(vae4.VAE4_U8, [1 << 24], data=FAKE + 16)), -8),
    (dict(ws=_t(vae4.VAE4_U8, [1000], data=FAKE * 4)), -8),
])
def test_validation_rejects(lib, over, code):
    assert _call(lib, _args(**over)) == code


def test_validation_options(lib):
    assert _call(lib, _args(), vae4.Options(0.0, 24, 0, 152, 0)) == -10
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 4)) == -11
    # E5M2 exists on the tcgen05 path only
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 3)) == -6
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 9)) == -6   # short waits + mma.sync
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 16)) == -11
    assert _call(lib, _args(), vae4.Options(-1.0, 0, 0, 152, 0)) == -11
    # the high/residual P split: 0 or 1, tcgen05 path only
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 0, 2)) == -11
    assert _call(lib, _args(), vae4.Options(0.0, 0, 0, 152, 1, 1)) == -6
    # capacity beyond what the block table can address
    assert _call(lib, _args(), vae4.Options(0.0, 0, 64 * 16 + 1, 152, 0)) == -3
    a = _args()
    a["q"].data = None
    assert _call(lib, a) == -1


def test_stride_counterexample_is_rejected_by_the_pool_form(lib):
    """The pool form [n_pages][2][Hkv][page][D] must be contiguous, so the
    pages' 8-but-not-16-byte token stride (264 B) is a stride error there;
    verify_attn_e4m3_kv takes that layout (next tests)."""
    g = GOLD["stride_counterexample"]
    assert g["strides"][1] == g["second_token_byte"] and g["second_token_byte"] % 16 == 8
    kv = _t(vae4.VAE4_U8, [80, 2, 1, 16, 256], [2 * 16 * 264, 16 * 264, 16 * 264, 264, 1])
    assert _call(lib, _args(kv=kv)) == -4


# ------------------------------------- separate, strided K and V caches
def _kv_args(k=None, v=None, **over):
    """The pages' counterexample layout: [n][848][1][256], strides
    [223872, 264, 256, 1] for both caches."""
    g = GOLD["stride_counterexample"]
    n = 40
    shape, strides = [n] + g["shape"][1:], g["strides"]
    a = _args(**over)
    a["k"] = k or _t(vae4.VAE4_U8, shape, strides, data=FAKE * 8)
    a["v"] = v or _t(vae4.VAE4_U8, shape, strides, data=FAKE * 16)
    a["bt"] = _t(vae4.VAE4_I32, [1, 400])
    return a


def _call_kv(lib, a, opt=None):
    o = opt or vae4.Options(0.0, 0, 0, 152, 0)
    return lib.verify_attn_e4m3_kv(*[ctypes.byref(a[k]) for k in
                                     ("q", "k", "v", "bt", "seq", "sc", "out", "ws")],
                                   None, ctypes.byref(o))


def test_kv_entry_accepts_the_counterexample_layout(lib):
    """The [1,848,1,256] view with strides [223872,264,256,1] (PR #524, AI
    integration review) passes every layout check: the call only fails on
    the too-small workspace, which is checked after the caches."""
    a = _kv_args(ws=_t(vae4.VAE4_U8, [1000], data=FAKE * 4))
    assert _call_kv(lib, a) == -8
    # a contiguous token-major cache (vLLM's layout) likewise
    k = _t(vae4.VAE4_U8, [80, 16, 1, 256], data=FAKE * 8)
    v = _t(vae4.VAE4_U8, [80, 16, 1, 256], data=FAKE * 16)
    a = _kv_args(k=k, v=v, ws=_t(vae4.VAE4_U8, [1000], data=FAKE * 4))
    a["bt"] = _t(vae4.VAE4_I32, [1, 64])
    assert _call_kv(lib, a) == -8


@pytest.mark.parametrize("which,bad,code", [
    ("k", dict(strides=[223872, 260, 256, 1]), -4),   # not a multiple of 8
    ("v", dict(strides=[223872, 264, 256, 2]), -4),   # d not contiguous
    ("k", dict(data=FAKE * 8 + 4), -5),               # base not 8-byte aligned
    ("v", dict(shape=[40, 848, 1, 128]), -3),         # D differs from q
    ("k", dict(shape=[40, 840, 1, 256]), -3),         # K and V shapes differ
    ("k", dict(dtype=vae4.VAE4_I32), -2),
])
def test_kv_entry_rejects(lib, which, bad, code):
    g = GOLD["stride_counterexample"]
    d = dict(shape=[40] + g["shape"][1:], strides=g["strides"], data=FAKE * 8,
             dtype=vae4.VAE4_U8)
    d.update(bad)
    t = _t(d["dtype"], d["shape"], d["strides"], data=d["data"])
    a = _kv_args(**{which: t})
    assert _call_kv(lib, a) == code


def test_kv_entry_page_size_and_flags(lib):
    k = _t(vae4.VAE4_U8, [40, 40, 1, 256], [40 * 264, 264, 256, 1], data=FAKE * 8)
    v = _t(vae4.VAE4_U8, [40, 40, 1, 256], [40 * 264, 264, 256, 1], data=FAKE * 16)
    assert _call_kv(lib, _kv_args(k=k, v=v)) == -6    # page 40: not a multiple of 16
    # the legacy mma.sync kernel reads the pool form only
    assert _call_kv(lib, _kv_args(), vae4.Options(0.0, 0, 0, 152, vae4.FLAG_WARP_MMA)) == -6
