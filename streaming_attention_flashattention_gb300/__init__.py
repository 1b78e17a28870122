"""Python binding of libgbattn.so (GB300 streaming attention), argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module checks
tensor properties, passes raw device pointers and the current CUDA stream through ctypes,
and turns status codes into exceptions.  There is no fallback: if the library is missing
or was not built for this machine, loading raises.

Entry points (same names as the C ABI in include/gbattn.h):
  attn_fwd(q, k, v, causal, scale=None, out=None, lse=None)
  attn_fwd_counted(q, k, v, causal, s_tiles, ...)   attn_fwd plus the S tile products issued
  attn_fwd_positions(q, k, v, q_pos0, k_pos0, ...)  causal attention at explicit positions
  attn_merge(o_a, lse_a, o_b, lse_b, ...)           log-sum-exp merge of two partials
  attn_decode_splitkv(q, kcache, vcache, kv_lens, num_splits=0, scale=None, ...)
  attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, num_splits)
  attn_last_device_error(stream=None)
  attn_status_string(status)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY_PATH = os.path.join(_PKG, "libgbattn.so")

GBATTN_BF16 = 0
GBATTN_FP32 = 1
GBATTN_OK = 0
GBATTN_ERR_INVALID_ARG = -1
GBATTN_ERR_UNSUPPORTED = -2
GBATTN_ERR_MISALIGNED = -3
GBATTN_ERR_CUDA = -4
GBATTN_ERR_TIMEOUT = -5
GBATTN_ERR_WORKSPACE = -6
GBATTN_ERR_TOO_LARGE = -7

_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every exported symbol
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_LL = ctypes.c_longlong
EXPORTS = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "attn_fwd_counted": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P]),
    "attn_fwd_positions": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _LL, _LL, _P]),
    "attn_merge": (_I, [_P, _P, _I, _P, _P, _I, _P, _P, _I, _LL, _I, _P]),
    "attn_fwd_host_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "attn_decode_host_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode_host": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P]),
    "attn_prefill_kvcache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "attn_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "attn_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "attn_decode_multitoken_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "attn_decode_multitoken": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]),
    "attn_decode_splitkv_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_decode_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "attn_prefill_plan": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "attn_last_device_error": (_I, [_P, ctypes.POINTER(ctypes.c_int)]),
    "attn_selftest_bounded_wait": (_I, [_P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_version": (_I, []),
}


class GbAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {attn_status_string(status)} (status {status})")
        self.status = status


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libgbattn.so (built by build.build()); raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIBRARY_PATH
        if not os.path.exists(p):
            raise ImportError(
                f"{p} is missing: build it with streaming_attention_flashattention_gb300.build.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream) -> int:
    """cudaStream_t of `stream`, or of the current stream of the current device (read
    through torch's raw accessor when it has one: a tenth of the cost of building the
    Stream object, which small calls feel)."""
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_stream is not None:
        return int(_raw_stream(torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


def _check(fn: str, status: int):
    if status != GBATTN_OK:
        raise GbAttnError(fn, status)


def _dev_tensor(name: str, t: torch.Tensor, dtypes):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_version() -> int:
    return int(load_library().attn_version())


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
             scale: float | None = None, out: torch.Tensor | None = None,
             lse: torch.Tensor | None = None, stream=None):
    """O = softmax(scale * Q K^T + mask) V for BHSD tensors; returns (out, lse).

    q [B, Hq, Sq, d], k/v [B, Hkv, Skv, d], bf16 (tensor-core path) or fp32 (exact fp32
    path), contiguous CUDA tensors.  lse is fp32 [B, Hq, Sq].
    """
    lib = load_library()
    dts = (torch.bfloat16, torch.float32)
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev_tensor(n, t, dts)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,d] and k, v [B,Hkv,Skv,d]")
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _dev_tensor("out", out, (q.dtype,))
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    else:
        _dev_tensor("lse", lse, (torch.float32,))
    dtype = GBATTN_BF16 if q.dtype == torch.bfloat16 else GBATTN_FP32
    st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, Hq, Hkv, Sq, Skv, d, float(scale), 1 if causal else 0, dtype,
                      _stream_ptr(stream))
    _check("attn_fwd", st)
    return out, lse


def attn_fwd_counted(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
                     s_tiles: torch.Tensor, scale: float | None = None,
                     out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                     stream=None):
    """attn_fwd (bf16) that also adds the S = Q K^T tile products its kernels issued to
    s_tiles (an int32 CUDA tensor of one element, zeroed by the caller).  Returns (out, lse)."""
    lib = load_library()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev_tensor(n, t, (torch.bfloat16,))
    _dev_tensor("s_tiles", s_tiles, (torch.int32,))
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,d] and k, v [B,Hkv,Skv,d]")
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    st = lib.attn_fwd_counted(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, Hq, Hkv, Sq, Skv, d, float(scale),
                              1 if causal else 0, s_tiles.data_ptr(), _stream_ptr(stream))
    _check("attn_fwd_counted", st)
    return out, lse


def attn_fwd_positions(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, q_pos0: int,
                       k_pos0: int, scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, stream=None):
    """Causal attention with query i at position q_pos0 + i and key j at k_pos0 + j (a query
    sees the keys not after it); bf16 BHSD tensors.  Rows that see no key get O = 0 and
    LSE = -inf.  Returns (out, lse)."""
    lib = load_library()
    for n, t in (("q", q), ("k", k), ("v", v)):
        _dev_tensor(n, t, (torch.bfloat16,))
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,d] and k, v [B,Hkv,Skv,d]")
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _dev_tensor("out", out, (torch.bfloat16,))
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    else:
        _dev_tensor("lse", lse, (torch.float32,))
        if tuple(lse.shape) != (B, Hq, Sq):
            raise ValueError("lse must be [B, Hq, Sq]")
    st = lib.attn_fwd_positions(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, Hq, Hkv, Sq, Skv, d, float(scale),
                                int(q_pos0), int(k_pos0), _stream_ptr(stream))
    _check("attn_fwd_positions", st)
    return out, lse


_DT = {torch.bfloat16: GBATTN_BF16, torch.float32: GBATTN_FP32}


def attn_merge(o_a: torch.Tensor, lse_a: torch.Tensor, o_b: torch.Tensor, lse_b: torch.Tensor,
               out: torch.Tensor | None = None, lse_out: torch.Tensor | None = None,
               out_dtype: torch.dtype = torch.float32, stream=None):
    """Log-sum-exp merge of two partial results over disjoint key sets, row by row.

    o_a, o_b [..., d] (bf16 or fp32), lse_a, lse_b [...] fp32.  out (dtype out_dtype, or
    out.dtype when given) and lse_out may be o_a / lse_a or o_b / lse_b for an in-place
    accumulator.  Returns (out, lse_out)."""
    lib = load_library()
    for n, t in (("o_a", o_a), ("o_b", o_b)):
        _dev_tensor(n, t, tuple(_DT))
    for n, t in (("lse_a", lse_a), ("lse_b", lse_b)):
        _dev_tensor(n, t, (torch.float32,))
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape or o_a.shape[:-1] != lse_a.shape:
        raise ValueError("o_a, o_b must be [..., d] and lse_a, lse_b [...] of the same rows")
    d = o_a.shape[-1]
    rows = lse_a.numel()
    if out is None:
        out = torch.empty(o_a.shape, dtype=out_dtype, device=o_a.device)
    else:
        _dev_tensor("out", out, tuple(_DT))
        if out.shape != o_a.shape:
            raise ValueError("out must have o_a's shape")
    if lse_out is None:
        lse_out = torch.empty(lse_a.shape, dtype=torch.float32, device=o_a.device)
    else:
        _dev_tensor("lse_out", lse_out, (torch.float32,))
        if lse_out.shape != lse_a.shape:
            raise ValueError("lse_out must have lse_a's shape")
    st = lib.attn_merge(o_a.data_ptr(), lse_a.data_ptr(), _DT[o_a.dtype], o_b.data_ptr(),
                        lse_b.data_ptr(), _DT[o_b.dtype], out.data_ptr(), lse_out.data_ptr(),
                        _DT[out.dtype], rows, d, _stream_ptr(stream))
    _check("attn_merge", st)
    return out, lse_out


def _host_tensor(name: str, t: torch.Tensor, dtypes):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_host_ws = {}


def attn_fwd_host_workspace_size(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, d: int,
                                 dtype: int = GBATTN_BF16) -> int:
    return int(load_library().attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, d, dtype))


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
                  scale: float | None = None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                  stream=None):
    """attn_fwd on host (CPU) tensors: inputs copied in and outputs copied back by the call,
    overlapped with the kernel chunk by chunk.  Pinned (page-locked) tensors make the copies
    asynchronous; out / lse are allocated pinned when not given.  Returns (out, lse) on the
    host; they are complete once `stream` (default: the current stream) has been
    synchronised.  The device workspace is allocated and cached per size when not given.
    """
    lib = load_library()
    dts = (torch.bfloat16, torch.float32)
    for n, t in (("q", q), ("k", k), ("v", v)):
        _host_tensor(n, t, dts)
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,d] and k, v [B,Hkv,Skv,d]")
    B, Hq, Sq, d = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    else:
        _host_tensor("out", out, (q.dtype,))
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32).pin_memory()
    else:
        _host_tensor("lse", lse, (torch.float32,))
    dtype = GBATTN_BF16 if q.dtype == torch.bfloat16 else GBATTN_FP32
    need = attn_fwd_host_workspace_size(B, Hq, Hkv, Sq, Skv, d, dtype)
    if need == 0:
        raise GbAttnError("attn_fwd_host", GBATTN_ERR_INVALID_ARG)
    if workspace is None:
        key = (torch.cuda.current_device(), need)
        workspace = _host_ws.get(key)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
            _host_ws[key] = workspace
    st = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           B, Hq, Hkv, Sq, Skv, d, float(scale), 1 if causal else 0, dtype,
                           workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _check("attn_fwd_host", st)
    return out, lse


def attn_decode_host_workspace_size(B: int, Hq: int, Hkv: int, Lmax: int, d: int,
                                    num_splits: int = 0) -> int:
    return int(load_library().attn_decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits))


def attn_decode_host(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                     kv_lens: torch.Tensor, num_splits: int = 0, scale: float | None = None,
                     out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """attn_decode_splitkv on host (CPU) tensors: q [B,Hq,1,d], caches [B,Hkv,Lmax,d] bf16,
    kv_lens int32 [B], all on the host; inputs copied in and outputs copied back by the
    call.  Returns (out [B,Hq,1,d], lse [B,Hq]) on the host, complete once `stream` (default:
    the current stream) has been synchronised."""
    lib = load_library()
    for n, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _host_tensor(n, t, (torch.bfloat16,))
    _host_tensor("kv_lens", kv_lens, (torch.int32,))
    B, Hq, one, d = q.shape
    _, Hkv, Lmax, _ = kcache.shape
    if one != 1 or vcache.shape != kcache.shape or tuple(kv_lens.shape) != (B,):
        raise ValueError("expected q [B,Hq,1,d], caches [B,Hkv,Lmax,d], kv_lens [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    else:
        _host_tensor("out", out, (torch.bfloat16,))
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32).pin_memory()
    else:
        _host_tensor("lse", lse, (torch.float32,))
    need = attn_decode_host_workspace_size(B, Hq, Hkv, Lmax, d, num_splits)
    if need == 0:
        raise GbAttnError("attn_decode_host", GBATTN_ERR_INVALID_ARG)
    if workspace is None:
        key = ("decode_host", torch.cuda.current_device(), need)
        workspace = _host_ws.get(key)
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
            _host_ws[key] = workspace
    st = lib.attn_decode_host(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                              kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                              Lmax, d, float(scale), int(num_splits), workspace.data_ptr(),
                              workspace.numel(), _stream_ptr(stream))
    _check("attn_decode_host", st)
    return out, lse


def attn_prefill_kvcache(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                         kv_len: int, causal: bool = True, scale: float | None = None,
                         out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                         stream=None):
    """Chunked prefill: q [B,Hq,Sq,d] against the first kv_len rows of caches [B,Hkv,Lmax,d]
    (bf16).  Returns (out [B,Hq,Sq,d] bf16, lse [B,Hq,Sq] fp32)."""
    lib = load_library()
    for n, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _dev_tensor(n, t, (torch.bfloat16,))
    B, Hq, Sq, d = q.shape
    _, Hkv, Lmax, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    st = lib.attn_prefill_kvcache(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                  out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, int(kv_len),
                                  Lmax, d, float(scale), 1 if causal else 0, _stream_ptr(stream))
    _check("attn_prefill_kvcache", st)
    return out, lse


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, Lmax: int, d: int,
                               num_splits: int = 0) -> int:
    """Workspace bytes of attn_decode_splitkv on the current device (0: invalid, or no
    device to query)."""
    return int(load_library().attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, num_splits))


def attn_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Tq: int, Lmax: int, d: int,
                                num_splits: int, num_sms: int) -> int:
    """Workspace bytes of a decode call on a GPU with num_sms SMs (host only)."""
    return int(load_library().attn_decode_workspace_bytes(B, Hq, Hkv, Tq, Lmax, d, num_splits,
                                                          num_sms))


def attn_decode_splitkv(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                        kv_lens: torch.Tensor, num_splits: int = 0, scale: float | None = None,
                        out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None):
    """Single-token decode: q [B,Hq,1,d], caches [B,Hkv,Lmax,d] bf16, kv_lens int32 [B].

    Returns (out [B,Hq,1,d] bf16, lse [B,Hq] fp32).  `workspace` (uint8, on the device) is
    allocated here when not given; pass one to keep allocations out of a hot loop.
    """
    lib = load_library()
    for n, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _dev_tensor(n, t, (torch.bfloat16,))
    _dev_tensor("kv_lens", kv_lens, (torch.int32,))
    B, Hq, one, d = q.shape
    if one != 1:
        raise ValueError("decode takes one query token per sequence")
    _, Hkv, Lmax, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_decode_workspace_size(B, Hq, Hkv, Lmax, d, num_splits)
    if need == 0:
        _check("attn_decode_workspace_size", -1)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.attn_decode_splitkv(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                 kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 B, Hq, Hkv, Lmax, d, float(scale), int(num_splits),
                                 workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                 _stream_ptr(stream))
    _check("attn_decode_splitkv", st)
    return out, lse


def attn_decode_multitoken(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                           kv_lens: torch.Tensor, num_splits: int = 0, scale: float | None = None,
                           out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, stream=None):
    """Decode of Tq new tokens per sequence: q [B,Hq,Tq,d], caches [B,Hkv,Lmax,d] bf16,
    kv_lens int32 [B] (new tokens included).  Returns (out [B,Hq,Tq,d], lse [B,Hq,Tq])."""
    lib = load_library()
    for n, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _dev_tensor(n, t, (torch.bfloat16,))
    _dev_tensor("kv_lens", kv_lens, (torch.int32,))
    B, Hq, Tq, d = q.shape
    _, Hkv, Lmax, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    need = int(lib.attn_decode_multitoken_workspace_size(B, Hq, Hkv, Tq, Lmax, d, num_splits))
    if need == 0:
        _check("attn_decode_multitoken_workspace_size", -1)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = lib.attn_decode_multitoken(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                    kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                    B, Hq, Hkv, Tq, Lmax, d, float(scale), int(num_splits),
                                    workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                    _stream_ptr(stream))
    _check("attn_decode_multitoken", st)
    return out, lse


# Scratch the no-allocation decode entry point holds (bytes), as documented in gbattn.h.
NOALLOC_SCRATCH_BYTES = 8 << 20


def attn_decode_splitkv_noalloc(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                                kv_lens: torch.Tensor, out: torch.Tensor,
                                lse: torch.Tensor, num_splits: int = 0,
                                scale: float | None = None, stream=None):
    """attn_decode_splitkv without a workspace: the library's own fixed scratch is used, so
    nothing is allocated (the caller passes preallocated `out` and `lse`).  Calls must be
    ordered on one stream; see include/gbattn.h."""
    lib = load_library()
    for n, t in (("q", q), ("kcache", kcache), ("vcache", vcache), ("out", out)):
        _dev_tensor(n, t, (torch.bfloat16,))
    _dev_tensor("kv_lens", kv_lens, (torch.int32,))
    _dev_tensor("lse", lse, (torch.float32,))
    B, Hq, _, d = q.shape
    _, Hkv, Lmax, _ = kcache.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = lib.attn_decode_splitkv_noalloc(q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(),
                                         kv_lens.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         B, Hq, Hkv, Lmax, d, float(scale), int(num_splits),
                                         _stream_ptr(stream))
    _check("attn_decode_splitkv_noalloc", st)
    return out, lse


def attn_decode_plan(B: int, Hq: int, Hkv: int, Tq: int, Lmax: int, d: int, num_splits: int,
                     num_sms: int) -> dict:
    """The decode call's choices for these sizes on a GPU with num_sms SMs (host only)."""
    plan = (ctypes.c_int * 7)()
    _check("attn_decode_plan", load_library().attn_decode_plan(
        B, Hq, Hkv, Tq, Lmax, d, num_splits, num_sms, plan))
    return {"splits": plan[0], "kernel": "tcgen05" if plan[1] else "warp",
            "merge": {0: "combine", 1: "single_launch", 2: "combine_per_group"}[plan[2]],
            "items": plan[3],
            "rows_per_kv_head": plan[4], "combine_lanes": plan[5], "pieces": plan[6]}


def attn_prefill_plan(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, causal: bool,
                      num_sms: int) -> dict:
    """The bf16 prefill's work split for these sizes on a GPU with num_sms SMs (host only)."""
    plan = (ctypes.c_int * 4)()
    _check("attn_prefill_plan", load_library().attn_prefill_plan(
        B, Hq, Hkv, Sq, Skv, 1 if causal else 0, num_sms, plan))
    return {"mode": "kv_split" if plan[0] else "pairs", "first_launch_ctas": plan[1],
            "tail_pairs": plan[2], "q_tiles": plan[3]}


def attn_selftest_bounded_wait(stream=None) -> None:
    """Launch the never-satisfied bounded wait (see include/gbattn.h); read the outcome with
    attn_last_device_error()."""
    _check("attn_selftest_bounded_wait",
           load_library().attn_selftest_bounded_wait(_stream_ptr(stream)))


def attn_last_device_error(stream=None) -> tuple[int, int]:
    """Synchronise the stream and read+clear the bounded-wait error word: (status, word)."""
    lib = load_library()
    detail = ctypes.c_int(0)
    st = lib.attn_last_device_error(_stream_ptr(stream), ctypes.byref(detail))
    return int(st), int(detail.value)
