"""FP64 CPU oracle for paged GQA verify attention over an FP8 E4M3 KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library under
``fp8_paged_attention_e4m3_gb300/`` and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, FP64, OpenMP over output rows);
this module compiles it with gcc and marshals numpy arrays.  What it computes,
and the passages it follows, are stated in the header comment of ``oracle.c``.

Pins (tests that tie the oracle to something other than itself) live in
``tests/test_oracle_pins.py``; every function here is pinned there.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, FP64, no fast-math).

    ``-ffp-contract=off`` keeps gcc from fusing multiply-adds, so the x86 and
    Arm builds give the same bits.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint32]
            lib.oracle_e4m3_table.restype = None
            lib.oracle_e4m3_table.argtypes = [ctypes.c_void_p]
            lib.oracle_e5m2_value.restype = ctypes.c_double
            lib.oracle_e5m2_value.argtypes = [ctypes.c_uint32]
            lib.oracle_fp8_table.restype = None
            lib.oracle_fp8_table.argtypes = [ctypes.c_void_p, ctypes.c_int]
            args = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                    ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                    ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                    ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                    ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]
            lib.oracle_verify_attn.restype = ctypes.c_int
            lib.oracle_verify_attn.argtypes = args
            lib.oracle_verify_attn_fmt.restype = ctypes.c_int
            lib.oracle_verify_attn_fmt.argtypes = args + [ctypes.c_int]
            lib.oracle_verify_attn_strided.restype = ctypes.c_int
            lib.oracle_verify_attn_strided.argtypes = (
                [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 3 + [ctypes.c_void_p] * 4 +
                [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                      ctypes.c_int, ctypes.c_int])
            lib.oracle_bridge_fp16.restype = ctypes.c_int
            lib.oracle_bridge_fp16.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def e4m3_value(byte: int) -> float:
    """Exact value of one E4M3FN byte (NaN for 0x7F / 0xFF)."""
    return _load().oracle_e4m3_value(int(byte) & 0xFF)


def e4m3_table() -> np.ndarray:
    """All 256 E4M3FN byte values as float64 (index = byte)."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(out.ctypes.data)
    return out


KV_FORMATS = {"e4m3": 0, "e5m2": 1}


def e5m2_value(byte: int) -> float:
    """OCP FP8 E5M2 decode of one byte (inf / NaN at exponent 31)."""
    return _load().oracle_e5m2_value(int(byte) & 0xFF)


def fp8_table(kv_format: str = "e4m3") -> np.ndarray:
    """All 256 decoded values of the format, float64."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_fp8_table(out.ctypes.data, KV_FORMATS[kv_format])
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


class OracleError(RuntimeError):
    pass


_ERRORS = {-1: "bad arguments", -2: "block id out of range",
           -3: "sequence length beyond the block table"}


def verify_attn(q, kv_pages, block_table, seq_len, q_len, kv_scales,
                sm_scale: float | None = None, split_tokens: int = 0,
                rows=None, threads: int = 0, kv_format: str = "e4m3") -> np.ndarray:
    """Exact (FP64) verify attention.

    q           float16/float32/float64 [B][Qmax][Hq][D]
    kv_pages    uint8 [n_pages][2][Hkv][page][D] (FP8 bytes; K at index 0)
    block_table int32 [B][max_pages]
    seq_len     int32 [B]  (L, including the q tail)
    q_len       int32 [B]
    kv_scales   float32 [Hkv][2] = (s_K, s_V)
    sm_scale    softmax scale; default 1/sqrt(D)
    split_tokens 0 = direct mode, else split mode with partitions of T tokens
    rows        None (all rows; returns [B][Qmax][Hq][D]) or an int array of
                (b, i, hq) triples (returns [n_rows][D])
    kv_format   "e4m3" (default) or "e5m2": how the KV bytes decode
    """
    lib = _load()
    q64 = np.ascontiguousarray(np.asarray(q).astype(np.float64))
    kv = np.ascontiguousarray(kv_pages, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_len, dtype=np.int32)
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    sc = np.ascontiguousarray(np.asarray(kv_scales).astype(np.float64))
    B, Qmax, Hq, D = q64.shape
    n_pages, two, Hkv, page, D2 = kv.shape
    if two != 2 or D2 != D or bt.ndim != 2 or bt.shape[0] != B:
        raise ValueError("inconsistent shapes")
    if sc.shape != (Hkv, 2) or sl.shape != (B,) or ql.shape != (B,):
        raise ValueError("inconsistent shapes")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    if rows is None:
        out = np.zeros((B, Qmax, Hq, D), dtype=np.float64)
        rows_ptr, n_rows = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        out = np.zeros((r.shape[0], D), dtype=np.float64)
        rows_ptr, n_rows = r.ctypes.data, r.shape[0]
        rows = r  # keep alive
    rc = lib.oracle_verify_attn_fmt(
        q64.ctypes.data, kv.ctypes.data, bt.ctypes.data, sl.ctypes.data,
        ql.ctypes.data, sc.ctypes.data, B, Qmax, Hq, Hkv, D, page,
        n_pages, bt.shape[1], float(sm_scale), int(split_tokens), rows_ptr,
        n_rows, out.ctypes.data, int(threads), KV_FORMATS[kv_format])
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    return out


def verify_attn_strided(q, k_cache, v_cache, block_table, seq_len, q_len, kv_scales,
                        sm_scale: float | None = None, split_tokens: int = 0, rows=None,
                        threads: int = 0, kv_format: str = "e4m3") -> np.ndarray:
    """Exact (FP64) verify attention over a cache given as separate K and V
    arrays uint8 [n_pages][page][Hkv][D] -- any byte strides (views into a
    padded buffer included; K and V with the same strides), d contiguous.
    Other arguments and the result as verify_attn."""
    lib = _load()
    k, v = np.asarray(k_cache), np.asarray(v_cache)
    if k.dtype != np.uint8 or v.dtype != np.uint8 or k.ndim != 4 or k.shape != v.shape:
        raise ValueError("k_cache / v_cache: uint8 [n_pages][page][Hkv][D] of one shape")
    if k.strides != v.strides or k.strides[3] != 1:
        raise ValueError("k_cache / v_cache: equal strides, d contiguous")
    n_pages, page, Hkv, D = k.shape
    q64 = np.ascontiguousarray(np.asarray(q).astype(np.float64))
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_len, dtype=np.int32)
    ql = np.ascontiguousarray(q_len, dtype=np.int32)
    sc = np.ascontiguousarray(np.asarray(kv_scales).astype(np.float64))
    B, Qmax, Hq, D2 = q64.shape
    if D2 != D or bt.ndim != 2 or bt.shape[0] != B or sc.shape != (Hkv, 2):
        raise ValueError("inconsistent shapes")
    if sl.shape != (B,) or ql.shape != (B,):
        raise ValueError("inconsistent shapes")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    if rows is None:
        out = np.zeros((B, Qmax, Hq, D), dtype=np.float64)
        rows_ptr, n_rows = None, 0
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        out = np.zeros((r.shape[0], D), dtype=np.float64)
        rows_ptr, n_rows = r.ctypes.data, r.shape[0]
        rows = r  # keep alive
    rc = lib.oracle_verify_attn_strided(
        q64.ctypes.data, k.ctypes.data, v.ctypes.data, k.strides[0], k.strides[1],
        k.strides[2], bt.ctypes.data, sl.ctypes.data, ql.ctypes.data, sc.ctypes.data,
        B, Qmax, Hq, Hkv, D, page, n_pages, bt.shape[1], float(sm_scale), int(split_tokens),
        rows_ptr, n_rows, out.ctypes.data, int(threads), KV_FORMATS[kv_format])
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    return out


def bridge_fp16(kv_pages, block_table, seq_len, kv_scales, cap: int,
                kv_format: str = "e4m3", raw: bool = False):
    """Exact values of the paged FP8 -> FP16 bridge, float64 [B][Hkv][cap][D]
    for K and V: dec(byte) * scale for tokens t < L (dec(byte) when raw), NaN
    where nothing is written (t >= L).  Round with round_to_fp16 to get the
    FP16 the bridge must produce."""
    lib = _load()
    kv = np.ascontiguousarray(kv_pages, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_len, dtype=np.int32)
    sc = np.ascontiguousarray(np.asarray(kv_scales).astype(np.float64))
    n_pages, two, Hkv, page, D = kv.shape
    B = sl.shape[0]
    if two != 2 or bt.ndim != 2 or bt.shape[0] != B or sc.shape != (Hkv, 2):
        raise ValueError("inconsistent shapes")
    k = np.full((B, Hkv, cap, D), np.nan)
    v = np.full((B, Hkv, cap, D), np.nan)
    rc = lib.oracle_bridge_fp16(kv.ctypes.data, bt.ctypes.data, sl.ctypes.data, sc.ctypes.data,
                                B, Hkv, D, page, n_pages, bt.shape[1], int(cap),
                                KV_FORMATS[kv_format], int(bool(raw)), k.ctypes.data,
                                v.ctypes.data)
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"oracle error {rc}"))
    return k, v


def round_to_fp16(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even onto float16 (numpy's cast), for disagreement
    counts against FP16 outputs."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)
