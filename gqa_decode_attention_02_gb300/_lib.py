"""Thin ctypes binding over libgqa_decode.so (include/gqa_decode.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  torch supplies device memory and the current
stream.  If the library is missing the calls raise: there is no fallback.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_decode.so")

_lock = threading.Lock()
_lib = None


class Status(enum.IntEnum):
    OK = 0
    ERR_NULL = 1
    ERR_SHAPE = 2
    ERR_DTYPE = 3
    ERR_ALIGN = 4
    ERR_WORKSPACE = 5
    ERR_CUDA = 6
    ERR_CONTEXT = 7
    ERR_BLOCK_ID = 8
    ERR_TIMEOUT = 9
    ERR_PROBS = 10
    ERR_TREE = 11


KV_DTYPES = {"same": 0, "int8": 1, "e4m3": 2}


class GqaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{fn}: {status_string(status)} (status {int(status)})")


class Shape(ctypes.Structure):
    """gqa_shape of include/gqa_decode.h."""
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("H", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int),
                ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("flags", ctypes.c_uint), ("window", ctypes.c_int),
                ("kv_dtype", ctypes.c_int)]


FLAG_PDL = 1
FLAG_EARLY_KV = 2
FLAG_WARP_MMA = 4
FLAG_TENSOR_MEMORY = 8
FLAG_DIRECT = 16
ENGINES = {"auto": 0, "warp": FLAG_WARP_MMA, "tmem": FLAG_TENSOR_MEMORY, "direct": FLAG_DIRECT}
ENGINE_NAMES = {1: "warp", 2: "tmem", 3: "direct"}


EXPORTS = ("gqa_version", "gqa_status_string", "gqa_kv_append",
           "gqa_attention_workspace_size", "gqa_workspace_clear", "gqa_decode_attention",
           "gqa_verify_attention", "gqa_append_decode_attention", "gqa_append_verify_attention",
           "gqa_accept_workspace_size", "gqa_accept_prefix", "gqa_accept_sampled", "gqa_tree_verify_attention",
           "gqa_append_tree_verify_attention", "gqa_kv_append_quant",
           "gqa_decode_attention_quant", "gqa_verify_attention_quant",
           "gqa_append_decode_attention_quant", "gqa_append_verify_attention_quant",
           "gqa_tree_verify_attention_quant", "gqa_accept_tree", "gqa_kv_compact",
           "gqa_attention_engine")


def lib() -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m gqa_decode_attention_02_gb300.build` (no CPU fallback exists)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(Shape)
        L.gqa_version.restype = I
        L.gqa_version.argtypes = []
        L.gqa_status_string.restype = ctypes.c_char_p
        L.gqa_status_string.argtypes = [I]
        L.gqa_kv_append.restype = I
        L.gqa_kv_append.argtypes = [S, P, P, P, P, P, P, P, P]
        L.gqa_attention_workspace_size.restype = ctypes.c_size_t
        L.gqa_attention_workspace_size.argtypes = [S]
        L.gqa_workspace_clear.restype = I
        L.gqa_workspace_clear.argtypes = [P, ctypes.c_size_t, P]
        for name in ("gqa_decode_attention", "gqa_verify_attention"):
            f = getattr(L, name)
            f.restype = I
            f.argtypes = [S, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
        for name in ("gqa_append_decode_attention", "gqa_append_verify_attention"):
            f = getattr(L, name)
            f.restype = I
            f.argtypes = [S, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
        L.gqa_tree_verify_attention.restype = I
        L.gqa_tree_verify_attention.argtypes = [S, P, P, P, P, P, P, P, P, ctypes.c_size_t, P, P]
        L.gqa_append_tree_verify_attention.restype = I
        L.gqa_append_tree_verify_attention.argtypes = [S] + [P] * 10 + [ctypes.c_size_t, P, P]
        L.gqa_kv_append_quant.restype = I
        L.gqa_kv_append_quant.argtypes = [S] + [P] * 10
        for name in ("gqa_decode_attention_quant", "gqa_verify_attention_quant"):
            f = getattr(L, name)
            f.restype = I
            f.argtypes = [S] + [P] * 9 + [ctypes.c_size_t, P, P]
        L.gqa_tree_verify_attention_quant.restype = I
        L.gqa_tree_verify_attention_quant.argtypes = [S] + [P] * 10 + [ctypes.c_size_t, P, P]
        for name in ("gqa_append_decode_attention_quant", "gqa_append_verify_attention_quant"):
            f = getattr(L, name)
            f.restype = I
            f.argtypes = [S] + [P] * 11 + [ctypes.c_size_t, P, P]
        L.gqa_accept_workspace_size.restype = ctypes.c_size_t
        L.gqa_accept_workspace_size.argtypes = [I, I]
        L.gqa_accept_prefix.restype = I
        L.gqa_accept_prefix.argtypes = [I, I, I, P, P, P, P, P, P, ctypes.c_size_t, P, P]
        L.gqa_accept_sampled.restype = I
        L.gqa_accept_sampled.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P]
        L.gqa_accept_tree.restype = I
        L.gqa_accept_tree.argtypes = [I, I, I] + [P] * 8 + [ctypes.c_size_t, P, P]
        L.gqa_kv_compact.restype = I
        L.gqa_kv_compact.argtypes = [S] + [P] * 10
        _lib = L
        return L


def status_string(code: int) -> str:
    return lib().gqa_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_DTYPES = {torch.float16: 0, torch.bfloat16: 1}


def _check(fn: str, rc: int):
    if rc != 0:
        raise GqaError(fn, rc)


def _need(t, name, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def make_shape(q_or_new: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
               scale: float | None, heads_dim: int = 2, flags: int = 0,
               window: int = 0, kv: str = "same") -> Shape:
    B, T, X, H = q_or_new.shape
    NB, bs, K, H2 = k_cache.shape
    if H2 != H:
        raise ValueError(f"head size mismatch: {H} vs {H2}")
    if q_or_new.dtype not in _DTYPES:
        raise ValueError(f"dtype {q_or_new.dtype} unsupported (fp16 / bf16)")
    return Shape(B=B, T=T, N=X if heads_dim == 2 else K, K=K, H=H, block_size=bs,
                 num_blocks=NB, max_blocks_per_seq=block_tables.shape[1],
                 dtype=_DTYPES[q_or_new.dtype], scale=float(scale or 0.0), flags=int(flags),
                 window=int(window), kv_dtype=KV_DTYPES[kv])


_ws_cache: dict = {}


def workspace_size(shape: Shape) -> int:
    n = lib().gqa_attention_workspace_size(ctypes.byref(shape))
    if n == 0:
        raise GqaError("gqa_attention_workspace_size", Status.ERR_SHAPE)
    return n


def get_workspace(nbytes: int, device, stream=None, kind: str = "attention") -> torch.Tensor:
    """A zero-filled workspace of at least nbytes for calls on `stream`
    (default: the current stream of `device`), cached per (device, stream,
    kind) and reused: the library returns a workspace zero-filled after every
    call, and calls on one stream never overlap, so one buffer per stream is
    race-free.  The buffer is allocated and zero-filled on that stream, so the
    caching allocator hands its memory back only in that stream's order when
    a larger one replaces it."""
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    key = (dev.index, int(stream.cuda_stream), kind)
    with _lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(stream):
                ws = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=dev)
            _ws_cache[key] = ws
    return ws


def reset_workspaces() -> None:
    """Drop every cached workspace (the next call allocates a fresh, zeroed
    one).  Needed only after a call reported GQA_ERR_TIMEOUT through its
    status word, which may leave a workspace's flags set."""
    with _lock:
        _ws_cache.clear()
