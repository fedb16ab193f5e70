"""Python binding of libqkmla.so, the QK-Normed MLA decode library for GB300.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI declared in include/qkmla.h.  PyTorch provides device
memory and streams.  There is no fallback: if the shared library is missing
or a call fails, an exception is raised.

Calls: absorb_query, append, decode (or make_decode_args + decode_raw to keep
one argument block); prepare_absorb_query / prepare_append return a Prepared
call whose arguments are marshalled once, for loops over fixed buffers.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqkmla.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_DEVICE_BOUNDS, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
F32, BF16 = 0, 1
FLAG_PLAIN_MLA = 1
FLAG_FORCE_SIMT = 2
FLAG_TEST_STALL = 4
FLAG_ALPHA_F16 = 8

SYMBOLS = [
    "qkmla_absorb_query", "qkmla_append", "qkmla_decode_workspace_size", "qkmla_decode",
    "qkmla_get_device_status", "qkmla_status_string", "qkmla_version", "qkmla_decode_kernel_name",
    "qkmla_decode_launch_count", "qkmla_up_project", "qkmla_append_rope", "qkmla_project_query",
]


class QkmlaError(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call} failed: {code} ({status_string(code)})")


class DecodeArgs(ctypes.Structure):
    """Mirror of `qkmla_decode_args` in include/qkmla.h (same field order)."""
    _fields_ = [
        ("q_tilde", ctypes.c_void_p),
        ("alpha_q", ctypes.c_void_p),
        ("q_rope", ctypes.c_void_p),
        ("gamma_rope_q", ctypes.c_void_p),
        ("kv_cache", ctypes.c_void_p),
        ("ak_cache", ctypes.c_void_p),
        ("seq_lens", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p),
        ("num_slots", ctypes.c_int64),
        ("page_size", ctypes.c_int),
        ("max_pages", ctypes.c_int),
        ("B", ctypes.c_int),
        ("s_q", ctypes.c_int),
        ("H", ctypes.c_int),
        ("G", ctypes.c_int),
        ("d_c", ctypes.c_int),
        ("d_r", ctypes.c_int),
        ("cache_dtype", ctypes.c_int),
        ("softmax_scale", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("flags", ctypes.c_uint),
        ("num_splits", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("o", ctypes.c_void_p),
        ("o_dtype", ctypes.c_int),
        ("lse", ctypes.c_void_p),
    ]


_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libqkmla.so (built by qk_normed_latent_gb300.build.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with qk_normed_latent_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, u, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint, ctypes.c_int64, ctypes.c_size_t
        L.qkmla_absorb_query.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, u, vp, i, vp, vp]
        L.qkmla_absorb_query.restype = i
        L.qkmla_append.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, u, vp, i, vp, i64, vp]
        L.qkmla_append.restype = i
        L.qkmla_decode_workspace_size.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.qkmla_decode_workspace_size.restype = sz
        L.qkmla_decode.argtypes = [ctypes.POINTER(DecodeArgs), vp]
        L.qkmla_decode.restype = i
        L.qkmla_get_device_status.argtypes = [vp]
        L.qkmla_get_device_status.restype = i
        L.qkmla_status_string.argtypes = [i]
        L.qkmla_status_string.restype = ctypes.c_char_p
        L.qkmla_version.argtypes = []
        L.qkmla_version.restype = i
        L.qkmla_decode_kernel_name.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.qkmla_decode_kernel_name.restype = ctypes.c_char_p
        L.qkmla_decode_launch_count.argtypes = [ctypes.POINTER(DecodeArgs)]
        L.qkmla_decode_launch_count.restype = i
        L.qkmla_up_project.argtypes = [vp, i, vp, i, i, i, i, i, vp, i, vp]
        L.qkmla_up_project.restype = i
        L.qkmla_append_rope.argtypes = [vp, vp, vp, f, vp, vp, vp, i, i, i, i, i, f, u, vp, i, vp, i64, vp]
        L.qkmla_append_rope.restype = i
        L.qkmla_project_query.argtypes = [vp, vp, vp, f, i, i, i, i, i, vp, vp, vp]
        L.qkmla_project_query.restype = i
        if hasattr(L, "qkmla_decode_noalloc"):
            L.qkmla_decode_noalloc.argtypes = [ctypes.POINTER(DecodeArgs), vp]
            L.qkmla_decode_noalloc.restype = i
            L.qkmla_decode_noalloc_max_workspace.argtypes = []
            L.qkmla_decode_noalloc_max_workspace.restype = sz
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().qkmla_status_string(int(code)).decode()


def _check(call: str, code: int) -> None:
    if code != OK:
        raise QkmlaError(call, code)


# ----------------------------------------------------------------------------
# torch-tensor front end (marshalling only)
# ----------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("qkmla: tensors must be contiguous")
    if not t.is_cuda:
        raise ValueError("qkmla: tensors must live on a CUDA device")
    return t.data_ptr()


def _dtype_code(dt) -> int:
    torch = _torch()
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError(f"qkmla: unsupported dtype {dt}")


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Prepared:
    """One library call with its arguments marshalled once: the tensors must stay
    alive and in place; a call only adds the stream."""

    def __init__(self, name: str, args: tuple):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = args

    def __call__(self, stream=None) -> None:
        _check(self.name, self.fn(*self.args, _stream(stream)))


def prepare_absorb_query(q, gamma_q, gamma_k, w_k, eps: float, q_tilde, alpha_q, plain: bool = False) -> Prepared:
    """qkmla_absorb_query for fixed tensors (see absorb_query)."""
    rows, H, d_h = q.shape
    G, d_c, _ = w_k.shape
    return Prepared("qkmla_absorb_query",
                    (_ptr(q), _ptr(gamma_q), _ptr(gamma_k), _ptr(w_k), rows, H, G, d_h, d_c, float(eps),
                     FLAG_PLAIN_MLA if plain else 0, _ptr(q_tilde), _dtype_code(q_tilde.dtype), _ptr(alpha_q)))


def absorb_query(q, gamma_q, gamma_k, w_k, eps: float, q_tilde, alpha_q, plain: bool = False, stream=None):
    """q [rows, H, d_h] fp32 -> q_tilde [rows, H, d_c] (fp32/bf16), alpha_q [rows, H] fp32."""
    prepare_absorb_query(q, gamma_q, gamma_k, w_k, eps, q_tilde, alpha_q, plain)(stream)
    return q_tilde, alpha_q


def _alpha_flag(ak_cache) -> int:
    """QKMLA_FLAG_ALPHA_F16 for a float16 A^k_cache, 0 for fp32."""
    torch = _torch()
    if ak_cache is None or ak_cache.dtype == torch.float32:
        return 0
    if ak_cache.dtype == torch.float16:
        return FLAG_ALPHA_F16
    raise ValueError(f"qkmla: the A^k_cache is float32 or float16, not {ak_cache.dtype}")


def prepare_append(c_new, k_rope_new, w_k, gamma_rope_k, slot_mapping, kv_cache, ak_cache, eps: float,
                   plain: bool = False) -> Prepared:
    """qkmla_append for fixed tensors (see append)."""
    N, d_c = c_new.shape
    d_r = k_rope_new.shape[1]
    G, _, d_h = w_k.shape
    flags = (FLAG_PLAIN_MLA if plain else 0) | _alpha_flag(ak_cache)
    return Prepared("qkmla_append",
                    (_ptr(c_new), _ptr(k_rope_new), _ptr(w_k), _ptr(gamma_rope_k), _ptr(slot_mapping), N, G, d_c,
                     d_h, d_r, float(eps), flags, _ptr(kv_cache),
                     _dtype_code(kv_cache.dtype), _ptr(ak_cache), kv_cache.shape[0]))


def append(c_new, k_rope_new, w_k, gamma_rope_k, slot_mapping, kv_cache, ak_cache, eps: float,
           plain: bool = False, stream=None):
    """Write new tokens (c_new [N, d_c], k_rope_new [N, d_r], fp32) into kv_cache
    [num_slots, d_c+d_r] and ak_cache [num_slots, G] (fp32, or float16 for the
    reduced-precision scalar cache) at slot_mapping [N] (int64)."""
    prepare_append(c_new, k_rope_new, w_k, gamma_rope_k, slot_mapping, kv_cache, ak_cache, eps, plain)(stream)


def prepare_append_rope(c_new, k_rope_raw, positions, rope_theta: float, w_k, gamma_rope_k, slot_mapping, kv_cache,
                        ak_cache, eps: float, plain: bool = False) -> Prepared:
    """qkmla_append_rope for fixed tensors: like prepare_append with unrotated RoPE
    keys and their positions [N] (int32)."""
    N, d_c = c_new.shape
    d_r = k_rope_raw.shape[1]
    G, _, d_h = w_k.shape
    flags = (FLAG_PLAIN_MLA if plain else 0) | _alpha_flag(ak_cache)
    return Prepared("qkmla_append_rope",
                    (_ptr(c_new), _ptr(k_rope_raw), _ptr(positions), float(rope_theta), _ptr(w_k), _ptr(gamma_rope_k),
                     _ptr(slot_mapping), N, G, d_c, d_h, d_r, float(eps), flags, _ptr(kv_cache),
                     _dtype_code(kv_cache.dtype), _ptr(ak_cache), kv_cache.shape[0]))


def append_rope(c_new, k_rope_raw, positions, rope_theta: float, w_k, gamma_rope_k, slot_mapping, kv_cache,
                ak_cache, eps: float, plain: bool = False, stream=None):
    """append() for RoPE keys before rotation: rotated by positions [N], then normalised and stored."""
    prepare_append_rope(c_new, k_rope_raw, positions, rope_theta, w_k, gamma_rope_k, slot_mapping, kv_cache,
                        ak_cache, eps, plain)(stream)


def prepare_project_query(x, w_q, positions, rope_theta: float, q, q_rope) -> Prepared:
    """qkmla_project_query for fixed tensors: x [rows, d_x] bf16, w_q [H, d_h + d_r, d_x] bf16,
    positions [rows] int32 -> q [rows, H, d_h] fp32, q_rope [rows, H, d_r] fp32 (rotated)."""
    rows, d_x = x.shape
    H, d_h = q.shape[-2], q.shape[-1]
    d_r = q_rope.shape[-1] if q_rope is not None else 0
    return Prepared("qkmla_project_query", (_ptr(x), _ptr(w_q), _ptr(positions), float(rope_theta), rows, d_x, H,
                                            d_h, d_r, _ptr(q), _ptr(q_rope)))


def project_query(x, w_q, positions, rope_theta: float, q, q_rope, stream=None):
    prepare_project_query(x, w_q, positions, rope_theta, q, q_rope)(stream)
    return q, q_rope


def make_decode_args(q_tilde, alpha_q, q_rope, gamma_rope_q, kv_cache, ak_cache, seq_lens, page_table,
                     page_size: int, max_pages: int, G: int, softmax_scale: float, eps: float, o, lse,
                     plain: bool = False, force_simt: bool = False, num_splits: int = 0,
                     workspace=None) -> DecodeArgs:
    B, s_q, H, d_c = q_tilde.shape
    d_r = q_rope.shape[-1] if q_rope is not None else 0
    a = DecodeArgs()
    a.q_tilde, a.alpha_q, a.q_rope = _ptr(q_tilde), _ptr(alpha_q), _ptr(q_rope)
    a.gamma_rope_q = _ptr(gamma_rope_q)
    a.kv_cache, a.ak_cache = _ptr(kv_cache), _ptr(ak_cache)
    a.seq_lens, a.page_table = _ptr(seq_lens), _ptr(page_table)
    a.num_slots = kv_cache.shape[0]
    a.page_size, a.max_pages = int(page_size), int(max_pages)
    a.B, a.s_q, a.H, a.G, a.d_c, a.d_r = B, s_q, H, int(G), d_c, d_r
    a.cache_dtype = _dtype_code(kv_cache.dtype)
    a.softmax_scale, a.eps = float(softmax_scale), float(eps)
    a.flags = (FLAG_PLAIN_MLA if plain else 0) | (FLAG_FORCE_SIMT if force_simt else 0) | _alpha_flag(ak_cache)
    a.num_splits = int(num_splits)
    a.o, a.o_dtype = _ptr(o), _dtype_code(o.dtype)
    a.lse = _ptr(lse)
    if workspace is not None:
        a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    return a


def decode_workspace_size(args: DecodeArgs) -> int:
    return int(lib().qkmla_decode_workspace_size(ctypes.byref(args)))


def decode_kernel_name(args: DecodeArgs) -> str:
    return lib().qkmla_decode_kernel_name(ctypes.byref(args)).decode()


def decode_launch_count(args: DecodeArgs) -> int:
    return int(lib().qkmla_decode_launch_count(ctypes.byref(args)))


def decode_raw(args: DecodeArgs, stream=None) -> None:
    _check("qkmla_decode", lib().qkmla_decode(ctypes.byref(args), _stream(stream)))


def decode(q_tilde, alpha_q, q_rope, gamma_rope_q, kv_cache, ak_cache, seq_lens, page_table, page_size: int,
           max_pages: int, G: int, softmax_scale: float, eps: float, o, lse, plain: bool = False,
           force_simt: bool = False, num_splits: int = 0, workspace=None, stream=None):
    """QK-Normed MLA decode; allocates the workspace with torch when none is given."""
    torch = _torch()
    a = make_decode_args(q_tilde, alpha_q, q_rope, gamma_rope_q, kv_cache, ak_cache, seq_lens, page_table,
                         page_size, max_pages, G, softmax_scale, eps, o, lse, plain, force_simt, num_splits,
                         workspace)
    need = decode_workspace_size(a)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q_tilde.device)
        a.workspace, a.workspace_bytes = workspace.data_ptr(), need
    decode_raw(a, stream)
    return o, lse


def prepare_up_project(o, w_v, out) -> Prepared:
    """qkmla_up_project for fixed tensors (see up_project)."""
    H, d_c = o.shape[-2], o.shape[-1]
    rows = o.numel() // (H * d_c)
    G_v, _, d_v = w_v.shape
    return Prepared("qkmla_up_project", (_ptr(o), _dtype_code(o.dtype), _ptr(w_v), rows, H, G_v, d_c, d_v, _ptr(out),
                                         _dtype_code(out.dtype)))


def up_project(o, w_v, out, stream=None):
    """out [..., H, d_v] = o [..., H, d_c] @ W^V[g(h)] with w_v [G_v, d_c, d_v] (bf16)."""
    prepare_up_project(o, w_v, out)(stream)
    return out


def get_device_status(stream=None) -> int:
    return int(lib().qkmla_get_device_status(_stream(stream)))
