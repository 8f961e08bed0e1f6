"""ctypes binding of libgemma_attn.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

from . import _build

GEMMA_SLIDING, GEMMA_GLOBAL, GEMMA_SLIDING_RING = 0, 1, 2
GEMMA_BF16, GEMMA_FP32 = 0, 1
GEMMA_OK = 0
GEMMA_DEVERR_SEQ_LEN, GEMMA_DEVERR_WRITE_POS, GEMMA_DEVERR_TIMEOUT = 1, 2, 4
GEMMA_DEVERR_N_REAL = 8
GEMMA_DEVERR_PAGE = 16

_c_int, _c_void_p, _c_size_t, _c_float = ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
_PVOID = ctypes.POINTER(ctypes.c_void_p)
_PI32 = ctypes.POINTER(ctypes.c_int32)

_SIGNATURES = {
    "gemma_kv_append": (_c_int, [_PVOID, _PVOID, _PI32, _c_int, _c_int, _c_void_p, _c_void_p,
                                 _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _c_void_p, _c_void_p]),
    "gemma_attn_decode": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int, _c_int,
                                   _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_float, _c_int, _c_void_p, _c_size_t,
                                   _c_void_p, _c_void_p]),
    "gemma_attn_prefill": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int, _c_int,
                                    _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_int, _c_float, _c_int, _c_void_p,
                                    _c_size_t, _c_void_p, _c_void_p]),
    "gemma_attn_decode_static": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int,
                                          _c_int, _c_void_p, _c_int, _c_int, _c_int, _c_int,
                                          _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _c_int,
                                          _c_void_p, _c_void_p]),
    "gemma_attn_softcap": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int, _c_int,
                                    _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _c_int, _c_int, _c_float, _c_float, _c_int,
                                    _c_void_p, _c_size_t, _c_void_p, _c_void_p]),
    "gemma_attn_decode_append": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int,
                                          _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                          _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                          _c_int, _c_int, _c_float, _c_int, _c_void_p, _c_size_t,
                                          _c_void_p, _c_void_p]),
    "gemma_kv_append_ring": (_c_int, [_PVOID, _PVOID, _PI32, _c_int, _c_int, _c_void_p,
                                      _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_void_p, _c_void_p]),
    "gemma_kv_append_bucket": (_c_int, [_PVOID, _PVOID, _PI32, _c_int, _c_int, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                        _c_int, _c_int, _c_int, _c_int, _c_void_p, _c_void_p]),
    "gemma_attn_prefill_bucket": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int,
                                           _c_int, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                           _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                           _c_int, _c_float, _c_int, _c_void_p, _c_size_t,
                                           _c_void_p, _c_void_p]),
    "gemma_attn_workspace_size": (_c_size_t, [_c_int] * 8),
    "gemma_kv_append_paged": (_c_int, [_PVOID, _PVOID, _PI32, _c_int, _c_int, _c_void_p,
                                       _c_void_p, _c_void_p, _c_void_p, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_void_p,
                                       _c_void_p]),
    "gemma_attn_paged": (_c_int, [_c_void_p, _c_void_p, _PVOID, _PVOID, _PI32, _c_int, _c_int,
                                  _c_void_p, _c_void_p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_float, _c_int, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                  _c_size_t, _c_void_p, _c_void_p]),
    "gemma_attn_workspace_size_paged": (_c_size_t, [_c_int, _c_int, _c_int, _c_int, _c_int,
                                                    _c_int, _c_int, _c_int]),
    "gemma_logit_softcap_argmax": (_c_int, [_c_void_p, _c_int, _c_int, _c_int, _c_float,
                                            _c_void_p, _c_void_p, _c_void_p, _c_size_t,
                                            _c_void_p]),
    "gemma_logit_workspace_size": (_c_size_t, [_c_int, _c_int]),
    "gemma_status_string": (ctypes.c_char_p, [_c_int]),
    "gemma_abi_version": (_c_int, []),
}


class GemmaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({gemma_status_string(status)})")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgemma_attn.so (building it first when it is missing or stale and nvcc exists)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with mixed_sliding_global_gb300._build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def exported_symbols():
    """Function names declared in include/gemma_attn.h."""
    with open(_build.HEADER) as f:
        text = f.read()
    return re.findall(r"^\s*(?:int|size_t|const char\*)\s+(gemma_\w+)\s*\(", text, re.M)


def gemma_status_string(status: int) -> str:
    return library().gemma_status_string(int(status)).decode()


def gemma_abi_version() -> int:
    return library().gemma_abi_version()


# ---------------------------------------------------------------------------------------------
def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GEMMA_BF16
    if t.dtype == torch.float32:
        return GEMMA_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _dev_ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _ptr_array(ts: Sequence[Optional[torch.Tensor]]):
    return (ctypes.c_void_p * len(ts))(*[_dev_ptr(t) for t in ts])


def _i32_array(xs: Sequence[int]):
    return (ctypes.c_int32 * len(xs))(*[int(x) for x in xs])


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, status: int) -> None:
    if status != GEMMA_OK:
        raise GemmaError(fn, status)


def _cache_of(caches, owner_map, layer):
    return caches[int(owner_map[layer])]


def gemma_kv_append(k_cache: Sequence[Optional[torch.Tensor]],
                    v_cache: Optional[Sequence[Optional[torch.Tensor]]],
                    owner_map: Sequence[int], layer: int, k_new: torch.Tensor,
                    v_new: Optional[torch.Tensor], write_pos: torch.Tensor, *, k_eq_v: bool,
                    kv_capacity: Optional[int] = None, device_error: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    """k_cache[l]: [B][n_kv][cap][d]; k_new/v_new: [B][n_new][n_kv][d]; write_pos: int32 [B]."""
    B, n_new, n_kv, d = k_new.shape
    n_layers = len(owner_map)
    kc = k_cache[int(owner_map[layer])]
    cap = kv_capacity if kv_capacity is not None else (kc.shape[2] if kc is not None else 0)
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    st = library().gemma_kv_append(
        _ptr_array(list(k_cache)), _ptr_array(vcs), _i32_array(owner_map), n_layers, layer,
        _dev_ptr(k_new), _dev_ptr(v_new), _dev_ptr(write_pos), B, n_new, n_kv, d, cap,
        int(bool(k_eq_v)), _dtype(k_new), _dev_ptr(device_error), _stream(stream))
    _check("gemma_kv_append", st)


def gemma_attn_decode_append(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map,
                             layer: int, k_new: Optional[torch.Tensor],
                             v_new: Optional[torch.Tensor], write_pos: torch.Tensor,
                             seq_lens: torch.Tensor, max_seq_len: int, *, kind: int, window: int,
                             n_kv: int, k_eq_v: bool, scale: float,
                             kv_capacity: Optional[int] = None,
                             workspace: Optional[torch.Tensor] = None,
                             device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Append this step's K/V row ([B][1][n_kv][d]) and decode, in one launch (bf16)."""
    B = q.shape[0]
    n_q, d = q.shape[-2], q.shape[-1]
    n_layers = len(owner_map)
    kc = _cache_of(k_cache, owner_map, layer)
    cap = kv_capacity if kv_capacity is not None else kc.shape[2]
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    ws_ptr = _dev_ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = library().gemma_attn_decode_append(
        _dev_ptr(out), _dev_ptr(q), _ptr_array(list(k_cache)), _ptr_array(vcs),
        _i32_array(owner_map), n_layers, layer, _dev_ptr(k_new), _dev_ptr(v_new),
        _dev_ptr(write_pos), _dev_ptr(seq_lens), int(max_seq_len), B, int(kind), int(window), n_q,
        int(n_kv), d, int(bool(k_eq_v)), int(cap), float(scale), _dtype(q), ws_ptr, ws_bytes,
        _dev_ptr(device_error), _stream(stream))
    _check("gemma_attn_decode_append", st)


def gemma_kv_append_ring(k_cache: Sequence[Optional[torch.Tensor]],
                         v_cache: Optional[Sequence[Optional[torch.Tensor]]],
                         owner_map: Sequence[int], layer: int, k_new: torch.Tensor,
                         v_new: Optional[torch.Tensor], write_pos: torch.Tensor, *, k_eq_v: bool,
                         kv_capacity: Optional[int] = None,
                         device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """gemma_kv_append into a ring cache: row t goes to slot (write_pos[b] + t) % capacity."""
    B, n_new, n_kv, d = k_new.shape
    n_layers = len(owner_map)
    kc = k_cache[int(owner_map[layer])]
    cap = kv_capacity if kv_capacity is not None else (kc.shape[2] if kc is not None else 0)
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    st = library().gemma_kv_append_ring(
        _ptr_array(list(k_cache)), _ptr_array(vcs), _i32_array(owner_map), n_layers, layer,
        _dev_ptr(k_new), _dev_ptr(v_new), _dev_ptr(write_pos), B, n_new, n_kv, d, cap,
        int(bool(k_eq_v)), _dtype(k_new), _dev_ptr(device_error), _stream(stream))
    _check("gemma_kv_append_ring", st)


def gemma_kv_append_bucket(k_cache: Sequence[Optional[torch.Tensor]],
                           v_cache: Optional[Sequence[Optional[torch.Tensor]]],
                           owner_map: Sequence[int], layer: int, k_new: torch.Tensor,
                           v_new: Optional[torch.Tensor], write_pos: torch.Tensor,
                           n_real: torch.Tensor, *, k_eq_v: bool, kv_capacity: Optional[int] = None,
                           device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """gemma_kv_append for a padded bucket: only rows t < n_real[b] (int32 [B]) are written."""
    B, n_new, n_kv, d = k_new.shape
    n_layers = len(owner_map)
    kc = k_cache[int(owner_map[layer])]
    cap = kv_capacity if kv_capacity is not None else (kc.shape[2] if kc is not None else 0)
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    st = library().gemma_kv_append_bucket(
        _ptr_array(list(k_cache)), _ptr_array(vcs), _i32_array(owner_map), n_layers, layer,
        _dev_ptr(k_new), _dev_ptr(v_new), _dev_ptr(write_pos), _dev_ptr(n_real), B, n_new, n_kv,
        d, cap, int(bool(k_eq_v)), _dtype(k_new), _dev_ptr(device_error), _stream(stream))
    _check("gemma_kv_append_bucket", st)


def gemma_attn_prefill_bucket(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map,
                              layer: int, seq_lens: torch.Tensor, n_real: torch.Tensor,
                              max_seq_len: int, *, kind: int, window: int, n_kv: int,
                              k_eq_v: bool, scale: float, kv_capacity: Optional[int] = None,
                              workspace: Optional[torch.Tensor] = None,
                              device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Prefill of a padded bucket: q, out [B][n_new][n_q][d], the first n_real[b] rows real;
    pad rows' outputs are zero."""
    B, n_new = q.shape[0], q.shape[1]
    n_q, d = q.shape[-2], q.shape[-1]
    n_layers = len(owner_map)
    kc = _cache_of(k_cache, owner_map, layer)
    cap = kv_capacity if kv_capacity is not None else kc.shape[2]
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    ws_ptr = _dev_ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = library().gemma_attn_prefill_bucket(
        _dev_ptr(out), _dev_ptr(q), _ptr_array(list(k_cache)), _ptr_array(vcs),
        _i32_array(owner_map), n_layers, layer, _dev_ptr(seq_lens), _dev_ptr(n_real),
        int(max_seq_len), n_new, B, int(kind), int(window), n_q, int(n_kv), d,
        int(bool(k_eq_v)), int(cap), float(scale), _dtype(q), ws_ptr, ws_bytes,
        _dev_ptr(device_error), _stream(stream))
    _check("gemma_attn_prefill_bucket", st)


def gemma_attn_workspace_size(batch: int, kind: int, window: int, n_q: int, n_kv: int,
                              head_dim: int, max_seq_len: int, n_new: int = 1) -> int:
    n = library().gemma_attn_workspace_size(batch, kind, window, n_q, n_kv, head_dim, max_seq_len,
                                            n_new)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid arguments for gemma_attn_workspace_size")
    return int(n)


def gemma_kv_append_paged(k_pool: Sequence[Optional[torch.Tensor]],
                          v_pool: Optional[Sequence[Optional[torch.Tensor]]], owner_map,
                          layer: int, k_new: torch.Tensor, v_new: Optional[torch.Tensor],
                          write_pos: torch.Tensor, block_table: torch.Tensor, *, k_eq_v: bool,
                          device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_pool[l], v_pool[l]: [n_pages][n_kv][page_size][d]; k_new, v_new: [B][n_new][n_kv][d];
    block_table: int32 [B][max_pages]."""
    n_layers = len(owner_map)
    kp = _cache_of(k_pool, owner_map, layer)
    n_pages, _, page_size, d = kp.shape
    B, n_new, n_kv, _ = k_new.shape
    vps = list(v_pool) if v_pool is not None else [None] * n_layers
    st = library().gemma_kv_append_paged(
        _ptr_array(list(k_pool)), _ptr_array(vps), _i32_array(owner_map), n_layers, layer,
        _dev_ptr(k_new), _dev_ptr(v_new), _dev_ptr(write_pos), _dev_ptr(block_table),
        int(block_table.shape[1]), int(page_size), int(n_pages), B, n_new, n_kv, d,
        int(bool(k_eq_v)), _dtype(k_new), _dev_ptr(device_error), _stream(stream))
    _check("gemma_kv_append_paged", st)


def gemma_attn_paged(out: torch.Tensor, q: torch.Tensor, k_pool, v_pool, owner_map, layer: int,
                     seq_lens: torch.Tensor, block_table: torch.Tensor, max_seq_len: int, *,
                     kind: int, window: int, n_kv: int, k_eq_v: bool, scale: float,
                     k_new: Optional[torch.Tensor] = None, v_new: Optional[torch.Tensor] = None,
                     write_pos: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """q, out: [B][n_new][n_q][d]; pools per layer [n_pages][n_kv][page_size][d]; block_table
    int32 [B][max_pages]; k_new/v_new/write_pos: the fused append of a decode step."""
    n_layers = len(owner_map)
    kp = _cache_of(k_pool, owner_map, layer)
    n_pages, _, page_size, _ = kp.shape
    B, n_tok, n_q, d = q.shape
    vps = list(v_pool) if v_pool is not None else [None] * n_layers
    ws_ptr = _dev_ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = library().gemma_attn_paged(
        _dev_ptr(out), _dev_ptr(q), _ptr_array(list(k_pool)), _ptr_array(vps),
        _i32_array(owner_map), n_layers, layer, _dev_ptr(seq_lens), _dev_ptr(block_table),
        int(block_table.shape[1]), int(page_size), int(n_pages), int(max_seq_len), n_tok, B,
        int(kind), int(window), n_q, int(n_kv), d, int(bool(k_eq_v)), float(scale), _dtype(q),
        _dev_ptr(k_new), _dev_ptr(v_new), _dev_ptr(write_pos), ws_ptr, ws_bytes,
        _dev_ptr(device_error), _stream(stream))
    _check("gemma_attn_paged", st)


def gemma_attn_workspace_size_paged(batch: int, kind: int, window: int, n_q: int, n_kv: int,
                                    head_dim: int, max_seq_len: int, n_new: int = 1) -> int:
    n = library().gemma_attn_workspace_size_paged(batch, kind, window, n_q, n_kv, head_dim,
                                                  max_seq_len, n_new)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid arguments for gemma_attn_workspace_size_paged")
    return int(n)


def gemma_logit_workspace_size(batch: int, vocab: int) -> int:
    n = library().gemma_logit_workspace_size(int(batch), int(vocab))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid arguments for gemma_logit_workspace_size")
    return int(n)


def gemma_logit_softcap_argmax(logits: torch.Tensor, softcap: float, argmax_out: torch.Tensor,
                               capped_out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """logits, capped_out: [B][V] bf16 or fp32 (capped_out may be logits itself, or None);
    argmax_out: int32 [B]."""
    if logits.dim() != 2:
        raise ValueError("logits must be [B][V]")
    if argmax_out.dtype != torch.int32:
        raise TypeError("argmax_out must be int32")
    B, V = logits.shape
    ws_ptr = _dev_ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = library().gemma_logit_softcap_argmax(_dev_ptr(logits), B, V, _dtype(logits),
                                              float(softcap), _dev_ptr(capped_out),
                                              _dev_ptr(argmax_out), ws_ptr, ws_bytes,
                                              _stream(stream))
    _check("gemma_logit_softcap_argmax", st)


def _attn(fn_name, out, q, k_cache, v_cache, owner_map, layer, seq_lens, max_seq_len, n_tok, *,
          kind, window, n_kv, k_eq_v, scale, kv_capacity, workspace, device_error, stream,
          softcap=None):
    B = q.shape[0]
    n_q, d = q.shape[-2], q.shape[-1]
    n_layers = len(owner_map)
    kc = _cache_of(k_cache, owner_map, layer)
    cap = kv_capacity if kv_capacity is not None else kc.shape[2]
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    ws_ptr = _dev_ptr(workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lib = library()
    common = (_ptr_array(list(k_cache)), _ptr_array(vcs), _i32_array(owner_map), n_layers, layer,
              _dev_ptr(seq_lens), int(max_seq_len))
    tail = (B, int(kind), int(window), n_q, int(n_kv), d, int(bool(k_eq_v)), int(cap), float(scale),
            _dtype(q), ws_ptr, ws_bytes, _dev_ptr(device_error), _stream(stream))
    if fn_name == "gemma_attn_decode":
        st = lib.gemma_attn_decode(_dev_ptr(out), _dev_ptr(q), *common, *tail)
    elif fn_name == "gemma_attn_softcap":
        st = lib.gemma_attn_softcap(_dev_ptr(out), _dev_ptr(q), *common, int(n_tok), *tail[:9],
                                    float(softcap), *tail[9:])
    else:
        st = lib.gemma_attn_prefill(_dev_ptr(out), _dev_ptr(q), *common, int(n_tok), *tail)
    _check(fn_name, st)


def gemma_attn_decode(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map, layer: int,
                      seq_lens: torch.Tensor, max_seq_len: int, *, kind: int, window: int,
                      n_kv: int, k_eq_v: bool, scale: float, kv_capacity: Optional[int] = None,
                      workspace: Optional[torch.Tensor] = None,
                      device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """q, out: [B][1][n_q][d] (or [B][n_q][d]); caches per layer [B][n_kv][cap][d]."""
    _attn("gemma_attn_decode", out, q, k_cache, v_cache, owner_map, layer, seq_lens, max_seq_len,
          1, kind=kind, window=window, n_kv=n_kv, k_eq_v=k_eq_v, scale=scale,
          kv_capacity=kv_capacity, workspace=workspace, device_error=device_error, stream=stream)


def gemma_attn_prefill(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map,
                       layer: int, seq_lens: torch.Tensor, max_seq_len: int, *, kind: int,
                       window: int, n_kv: int, k_eq_v: bool, scale: float,
                       kv_capacity: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                       device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """q, out: [B][n_new][n_q][d]; caches per layer [B][n_kv][cap][d]."""
    _attn("gemma_attn_prefill", out, q, k_cache, v_cache, owner_map, layer, seq_lens, max_seq_len,
          q.shape[1], kind=kind, window=window, n_kv=n_kv, k_eq_v=k_eq_v, scale=scale,
          kv_capacity=kv_capacity, workspace=workspace, device_error=device_error, stream=stream)


def gemma_attn_softcap(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map,
                       layer: int, seq_lens: torch.Tensor, max_seq_len: int, *, kind: int,
                       window: int, n_kv: int, k_eq_v: bool, scale: float, softcap: float,
                       kv_capacity: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                       device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """Decode (q.shape[1] == 1) or prefill with each scaled score s capped to
    softcap * tanh(s / softcap) (softcap 0: no cap). q, out: [B][n_tok][n_q][d]."""
    _attn("gemma_attn_softcap", out, q, k_cache, v_cache, owner_map, layer, seq_lens, max_seq_len,
          q.shape[1], kind=kind, window=window, n_kv=n_kv, k_eq_v=k_eq_v, scale=scale,
          kv_capacity=kv_capacity, workspace=workspace, device_error=device_error, stream=stream,
          softcap=softcap)


def gemma_attn_decode_static(out: torch.Tensor, q: torch.Tensor, k_cache, v_cache, owner_map,
                             layer: int, seq_lens: torch.Tensor, max_seq_len: int, *, kind: int,
                             window: int, n_kv: int, k_eq_v: bool, scale: float,
                             kv_capacity: Optional[int] = None,
                             device_error: Optional[torch.Tensor] = None, stream=None) -> None:
    """gemma_attn_decode with the library's built-in scratch instead of a workspace tensor, for
    callers that cannot allocate device memory (see include/gemma_attn.h)."""
    B = q.shape[0]
    n_q, d = q.shape[-2], q.shape[-1]
    n_layers = len(owner_map)
    kc = _cache_of(k_cache, owner_map, layer)
    cap = kv_capacity if kv_capacity is not None else kc.shape[2]
    vcs = list(v_cache) if v_cache is not None else [None] * n_layers
    st = library().gemma_attn_decode_static(
        _dev_ptr(out), _dev_ptr(q), _ptr_array(list(k_cache)), _ptr_array(vcs),
        _i32_array(owner_map), n_layers, layer, _dev_ptr(seq_lens), int(max_seq_len), B,
        int(kind), int(window), n_q, int(n_kv), d, int(bool(k_eq_v)), int(cap), float(scale),
        _dtype(q), _dev_ptr(device_error), _stream(stream))
    _check("gemma_attn_decode_static", st)
