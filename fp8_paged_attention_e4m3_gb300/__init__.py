"""Paged GQA verify attention over an FP8 E4M3 KV cache, for GB300 (sm_103a).

Thin Python binding of the C ABI in ``include/verify_attn_e4m3.h``: it turns
torch tensors into ``vae4_tensor`` descriptors and passes torch's current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
this module does argument marshalling only and has no fallback: if the
library cannot be built or loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

ABI_VERSION = 2

VAE4_U8, VAE4_I32, VAE4_F16, VAE4_F32 = 1, 2, 3, 4

FLAG_WARP_MMA = 0x1
FLAG_KV_E5M2 = 0x2
FLAG_BRIDGE_RAW = 0x4
FLAG_TEST_SHORT_WAITS = 0x8

STATUS_BAD_BLOCK = 0x1
STATUS_BAD_LENGTH = 0x2
STATUS_BAD_QLEN = 0x4
STATUS_TIMEOUT = 0x8
STATUS_PLAN = 0x10

ERRORS = {
    0: "VAE4_OK", -1: "VAE4_ERR_NULL", -2: "VAE4_ERR_DTYPE", -3: "VAE4_ERR_SHAPE",
    -4: "VAE4_ERR_STRIDE", -5: "VAE4_ERR_MISALIGNED", -6: "VAE4_ERR_UNSUPPORTED",
    -7: "VAE4_ERR_GQA", -8: "VAE4_ERR_WORKSPACE", -9: "VAE4_ERR_CUDA",
    -10: "VAE4_ERR_PARTITION", -11: "VAE4_ERR_OPTIONS",
}

# Every symbol include/verify_attn_e4m3.h declares.
EXPORTS = (
    "verify_attn_e4m3", "verify_attn_e4m3_ex", "verify_attn_e4m3_partials",
    "verify_attn_e4m3_combine", "verify_attn_e4m3_plan",
    "verify_attn_e4m3_workspace_bytes", "verify_attn_e4m3_abi_version",
    "verify_attn_e4m3_strerror", "verify_attn_e4m3_read_status",
    "verify_attn_e4m3_clear_status", "verify_attn_e4m3_decode_table",
    "verify_attn_e4m3_noalloc", "verify_attn_e4m3_kv_read",
    "verify_attn_e4m3_bridge_fp16", "verify_attn_e4m3_kv",
)

NOALLOC_SCRATCH_BYTES = 8 << 20


class Tensor(ctypes.Structure):
    """vae4_tensor"""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 5),
                ("stride", ctypes.c_int64 * 5)]


class Options(ctypes.Structure):
    """vae4_options"""
    _fields_ = [("softmax_scale", ctypes.c_float), ("partition_tokens", ctypes.c_int32),
                ("max_seq_len", ctypes.c_int32), ("num_sms", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("hilo_pv", ctypes.c_int32)]


class Vae4Error(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({strerror(code)})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    from . import _build
    return _build.LIB


def load(build_if_stale: bool = True):
    """Load libvae4.so (building it first if it is missing or stale) and check
    its ABI revision; raises if either step fails."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import _build
        if build_if_stale and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing; build it with "
                               "fp8_paged_attention_e4m3_gb300._build.build()")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER(Tensor)
        for name in ("verify_attn_e4m3",):
            getattr(lib, name).argtypes = [P] * 7 + [ctypes.c_void_p]
            getattr(lib, name).restype = ctypes.c_int
        for name in ("verify_attn_e4m3_ex", "verify_attn_e4m3_partials",
                     "verify_attn_e4m3_combine", "verify_attn_e4m3_kv_read"):
            getattr(lib, name).argtypes = [P] * 7 + [ctypes.c_void_p, ctypes.POINTER(Options)]
            getattr(lib, name).restype = ctypes.c_int
        lib.verify_attn_e4m3_kv.argtypes = [P] * 8 + [ctypes.c_void_p, ctypes.POINTER(Options)]
        lib.verify_attn_e4m3_kv.restype = ctypes.c_int
        lib.verify_attn_e4m3_bridge_fp16.argtypes = [P] * 6 + [ctypes.c_void_p, ctypes.c_int32,
                                                               ctypes.c_void_p]
        lib.verify_attn_e4m3_bridge_fp16.restype = ctypes.c_int
        lib.verify_attn_e4m3_plan.argtypes = [ctypes.c_int] * 5 + [
            ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
        lib.verify_attn_e4m3_plan.restype = ctypes.c_int
        lib.verify_attn_e4m3_workspace_bytes.argtypes = [ctypes.c_int] * 8
        lib.verify_attn_e4m3_workspace_bytes.restype = ctypes.c_int64
        lib.verify_attn_e4m3_abi_version.argtypes = []
        lib.verify_attn_e4m3_abi_version.restype = ctypes.c_int
        lib.verify_attn_e4m3_strerror.argtypes = [ctypes.c_int]
        lib.verify_attn_e4m3_strerror.restype = ctypes.c_char_p
        lib.verify_attn_e4m3_read_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32),
                                                     ctypes.c_void_p]
        lib.verify_attn_e4m3_read_status.restype = ctypes.c_int
        lib.verify_attn_e4m3_clear_status.argtypes = [P, ctypes.c_void_p]
        lib.verify_attn_e4m3_clear_status.restype = ctypes.c_int
        lib.verify_attn_e4m3_decode_table.argtypes = [ctypes.c_void_p,
                                                      ctypes.POINTER(ctypes.c_int32),
                                                      ctypes.c_int32, ctypes.c_void_p]
        lib.verify_attn_e4m3_decode_table.restype = ctypes.c_int
        lib.verify_attn_e4m3_noalloc.argtypes = [P] * 6 + [ctypes.c_void_p,
                                                           ctypes.POINTER(Options)]
        lib.verify_attn_e4m3_noalloc.restype = ctypes.c_int
        v = lib.verify_attn_e4m3_abi_version()
        if v != ABI_VERSION:
            raise RuntimeError(f"stale library: ABI revision {v}, binding expects "
                               f"{ABI_VERSION}; rebuild it")
        _lib = lib
        return lib


def strerror(code: int) -> str:
    try:
        return load().verify_attn_e4m3_strerror(int(code)).decode()
    except Exception:  # library unavailable
        return ERRORS.get(code, "unknown")


# ----------------------------------------------------------------------------
# torch tensor -> vae4_tensor
# ----------------------------------------------------------------------------
def _dtype_code(t) -> int:
    import torch
    m = {torch.uint8: VAE4_U8, torch.int32: VAE4_I32, torch.float16: VAE4_F16,
         torch.float32: VAE4_F32}
    if t.dtype == getattr(torch, "float8_e4m3fn", None):
        return VAE4_U8
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def describe(t) -> Tensor:
    """A vae4_tensor view of a torch tensor (no copy)."""
    if t.dim() > 5:
        raise ValueError("at most 5 dimensions")
    d = Tensor()
    d.data = t.data_ptr() if t.numel() > 0 or t.data_ptr() else None
    d.dtype = _dtype_code(t)
    d.ndim = t.dim()
    for k in range(t.dim()):
        d.shape[k] = t.shape[k]
        d.stride[k] = t.stride(k)
    return d


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(rc: int, where: str):
    if rc != 0:
        raise Vae4Error(rc, where)


# ----------------------------------------------------------------------------
# public API (same names as the C ABI)
# ----------------------------------------------------------------------------
def verify_attn_e4m3(q, kv_pages, block_table, seq_lens, kv_scales, out, workspace, *,
                     softmax_scale: float = 0.0, partition_tokens: int = 0,
                     max_seq_len: int = 0, num_sms: int = 0, flags: int = 0,
                     hilo_pv: bool = False, stream=None):
    """Run the verify step into ``out``.  All tensors on the current device;
    see include/verify_attn_e4m3.h for layouts.  Asynchronous on ``stream``
    (torch's current stream by default).  ``partition_tokens=0`` selects the
    automatic plan, made on the device from the lengths of each call (a
    captured graph stays balanced as they change); a positive multiple of 16
    fixes T.  ``hilo_pv=True`` carries P into the value product as an FP16
    high part plus a residual scaled by 2^11 (about 22 significant bits)."""
    lib = load()
    opt = Options(float(softmax_scale), int(partition_tokens), int(max_seq_len),
                  int(num_sms), int(flags), int(bool(hilo_pv)))
    descs = [describe(t) for t in (q, kv_pages, block_table, seq_lens, kv_scales, out,
                                   workspace)]
    rc = lib.verify_attn_e4m3_ex(*[ctypes.byref(x) for x in descs],
                                 ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(opt))
    _check(rc, "verify_attn_e4m3")
    return out


verify = verify_attn_e4m3


def verify_attn_e4m3_kv(q, k_cache, v_cache, block_table, seq_lens, kv_scales, out, workspace,
                        *, softmax_scale: float = 0.0, partition_tokens: int = 0,
                        max_seq_len: int = 0, num_sms: int = 0, flags: int = 0,
                        hilo_pv: bool = False, stream=None):
    """The verify step over separate K and V caches uint8 [n_pages][page]
    [Hkv][D] in any strided layout (token-major, padded token strides that
    are multiples of 8 bytes); see the header.  Other arguments as
    verify_attn_e4m3."""
    lib = load()
    opt = Options(float(softmax_scale), int(partition_tokens), int(max_seq_len),
                  int(num_sms), int(flags), int(bool(hilo_pv)))
    descs = [describe(t) for t in (q, k_cache, v_cache, block_table, seq_lens, kv_scales,
                                   out, workspace)]
    rc = lib.verify_attn_e4m3_kv(*[ctypes.byref(x) for x in descs],
                                 ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(opt))
    _check(rc, "verify_attn_e4m3_kv")
    return out


def _stage(name, q, kv_pages, block_table, seq_lens, kv_scales, out, workspace, *,
           softmax_scale=0.0, partition_tokens=0, max_seq_len=0, num_sms=0, flags=0,
           hilo_pv=False, stream=None):
    lib = load()
    opt = Options(float(softmax_scale), int(partition_tokens), int(max_seq_len),
                  int(num_sms), int(flags), int(bool(hilo_pv)))
    descs = [describe(t) for t in (q, kv_pages, block_table, seq_lens, kv_scales, out,
                                   workspace)]
    rc = getattr(lib, name)(*[ctypes.byref(x) for x in descs],
                            ctypes.c_void_p(_stream_handle(stream)), ctypes.byref(opt))
    _check(rc, name)
    return out


def verify_attn_e4m3_partials(*args, **kw):
    """Split stage only (see the header)."""
    return _stage("verify_attn_e4m3_partials", *args, **kw)


def verify_attn_e4m3_combine(*args, **kw):
    """Combine stage only (see the header)."""
    return _stage("verify_attn_e4m3_combine", *args, **kw)


def verify_attn_e4m3_bridge_fp16(kv_pages, block_table, seq_lens, kv_scales, k_out, v_out,
                                 *, status=None, flags: int = 0, stream=None):
    """Paged FP8 -> dense FP16 K and V (see the header): k_out / v_out are
    fp16 [B][Hkv][cap][D]; status is an optional int32 device tensor whose
    first element receives the status bits."""
    lib = load()
    descs = [describe(t) for t in (kv_pages, block_table, seq_lens, kv_scales, k_out, v_out)]
    st = ctypes.c_void_p(status.data_ptr()) if status is not None else ctypes.c_void_p(None)
    rc = lib.verify_attn_e4m3_bridge_fp16(*[ctypes.byref(x) for x in descs], st,
                                          ctypes.c_int32(int(flags)),
                                          ctypes.c_void_p(_stream_handle(stream)))
    _check(rc, "verify_attn_e4m3_bridge_fp16")
    return k_out, v_out


def verify_attn_e4m3_kv_read(*args, **kw):
    """Streaming read of the step's KV bytes, no compute (see the header):
    the gather floor the step is measured against."""
    return _stage("verify_attn_e4m3_kv_read", *args, **kw)


def verify_attn_e4m3_noalloc(q, kv_pages, block_table, seq_lens, kv_scales, out, *,
                             softmax_scale: float = 0.0, partition_tokens: int = 0,
                             max_seq_len: int = 0, num_sms: int = 0, hilo_pv: bool = False,
                             stream=None):
    """The verify step without a workspace, for callers that cannot allocate
    device memory: the library's own fixed 8 MiB scratch holds the partials.
    Calls on one device share that scratch, so they must not overlap on the
    GPU; the first call on a device must precede any stream capture."""
    lib = load()
    opt = Options(float(softmax_scale), int(partition_tokens), int(max_seq_len),
                  int(num_sms), 0, int(bool(hilo_pv)))
    descs = [describe(t) for t in (q, kv_pages, block_table, seq_lens, kv_scales, out)]
    rc = lib.verify_attn_e4m3_noalloc(*[ctypes.byref(x) for x in descs],
                                      ctypes.c_void_p(_stream_handle(stream)),
                                      ctypes.byref(opt))
    _check(rc, "verify_attn_e4m3_noalloc")
    return out


def verify_attn_e4m3_plan(B: int, Hkv: int, max_seq_len: int, partition_tokens: int = 0,
                          num_sms: int = 0):
    """(T, P) of the split-K plan for sequences at the capacity (with
    partition_tokens == 0 a call refines it on the device from the lengths it
    reads); num_sms == 0 uses the current device."""
    lib = load()
    if num_sms == 0:
        import torch
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()) \
            .multi_processor_count
    T, P = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.verify_attn_e4m3_plan(B, Hkv, max_seq_len, partition_tokens, num_sms,
                                     ctypes.byref(T), ctypes.byref(P)), "plan")
    return T.value, P.value


plan = verify_attn_e4m3_plan


def verify_attn_e4m3_workspace_bytes(B, Hq, Hkv, Qmax, D, max_seq_len,
                                     partition_tokens=0, num_sms=0) -> int:
    n = load().verify_attn_e4m3_workspace_bytes(B, Hq, Hkv, Qmax, D, max_seq_len,
                                                 partition_tokens, num_sms)
    if n < 0:
        raise Vae4Error(int(n), "workspace_bytes")
    return int(n)


workspace_bytes = verify_attn_e4m3_workspace_bytes


def verify_attn_e4m3_read_status(workspace, stream=None) -> int:
    """Status word of ``workspace`` (synchronises the stream)."""
    import torch
    lib = load()
    host = ctypes.c_int32(0)
    st = stream or torch.cuda.current_stream()
    _check(lib.verify_attn_e4m3_read_status(ctypes.byref(describe(workspace)),
                                            ctypes.byref(host),
                                            ctypes.c_void_p(_stream_handle(st))),
           "read_status")
    st.synchronize()
    return host.value & 0xFFFFFFFF


read_status = verify_attn_e4m3_read_status


def verify_attn_e4m3_clear_status(workspace, stream=None):
    _check(load().verify_attn_e4m3_clear_status(ctypes.byref(describe(workspace)),
                                                ctypes.c_void_p(_stream_handle(stream))),
           "clear_status")


clear_status = verify_attn_e4m3_clear_status


def verify_attn_e4m3_decode_table(flags: int = 0, stream=None):
    """(fp16 bit patterns of the 256 decoded codes as a device uint16-in-int16
    tensor, scale exponent): code b decodes to dec(b) * 2^scale_log2.  flags
    picks the kernel whose decoder runs (0 = tcgen05 path)."""
    import torch
    out = torch.empty(256, dtype=torch.int16, device="cuda")
    e = ctypes.c_int32(0)
    _check(load().verify_attn_e4m3_decode_table(ctypes.c_void_p(out.data_ptr()),
                                                ctypes.byref(e), int(flags),
                                                ctypes.c_void_p(_stream_handle(stream))),
           "decode_table")
    return out, e.value


decode_table = verify_attn_e4m3_decode_table


def alloc_workspace(B, Hq, Hkv, Qmax, D, max_seq_len, partition_tokens=0, device=None):
    """A zeroed workspace of the right size (torch allocation, 256-B aligned)."""
    import torch
    n = workspace_bytes(B, Hq, Hkv, Qmax, D, max_seq_len, partition_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
