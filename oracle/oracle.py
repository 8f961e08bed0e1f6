"""ctypes wrapper of ``attn_oracle.c`` -- TEST INFRASTRUCTURE ONLY.

Argument marshalling only: the arithmetic is in the C file. Tensors are torch CPU tensors
(bf16 or fp32 inputs, fp64 output) passed by pointer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import List, Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "attn_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

SLIDING, GLOBAL = 0, 1
BF16, FP32 = 0, 1


class OracleError(RuntimeError):
    pass


class _Layer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("window", ctypes.c_int32), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("k_eq_v", ctypes.c_int32)]


def build_oracle(out: str = LIB, mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable C99, no target-specific flags)."""
    if not force and mutant == 0 and os.path.exists(out) and \
            os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-o", out, SRC, "-lm"]
    if mutant:
        cmd.insert(1, f"-DORACLE_MUTANT={int(mutant)}")
    tmp = out + f".tmp{os.getpid()}"
    cmd[cmd.index(out)] = tmp
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def oracle_layers(layers) -> List[_Layer]:
    """Convert objects with kind/window/n_q/n_kv/head_dim/k_eq_v attributes."""
    return [_Layer(int(l.kind), int(l.window), int(l.n_q), int(l.n_kv), int(l.head_dim),
                   int(bool(l.k_eq_v))) for l in layers]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if t.device.type != "cpu" or not t.is_contiguous():
        raise OracleError("oracle inputs must be contiguous CPU tensors")
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise OracleError(f"unsupported dtype {t.dtype}")


class Oracle:
    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [
            ctypes.POINTER(_Layer), ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int,
            ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p), ctypes.c_int,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
            ctypes.c_int, ctypes.c_double, ctypes.c_void_p]
        lib.oracle_attention_softcap.restype = ctypes.c_int
        lib.oracle_attention_softcap.argtypes = lib.oracle_attention.argtypes[:-1] + [
            ctypes.c_double, ctypes.c_void_p]
        lib.oracle_kv_append.restype = ctypes.c_int
        lib.oracle_kv_append.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_resolve_owner.restype = ctypes.c_int
        lib.oracle_resolve_owner.argtypes = [ctypes.POINTER(_Layer), ctypes.POINTER(ctypes.c_int32),
                                             ctypes.c_int, ctypes.c_int]
        lib.oracle_logit_softcap_argmax.restype = ctypes.c_int
        lib.oracle_logit_softcap_argmax.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
        lib.oracle_mutant.restype = ctypes.c_int
        self.lib = lib
        self.mutant = lib.oracle_mutant()

    # ------------------------------------------------------------------------------------------
    def resolve_owner(self, layers, owner_map: Sequence[int], layer: int) -> int:
        arr = (_Layer * len(layers))(*oracle_layers(layers))
        om = (ctypes.c_int32 * len(owner_map))(*owner_map)
        return self.lib.oracle_resolve_owner(arr, om, len(layers), layer)

    def kv_append(self, cache: torch.Tensor, rows: torch.Tensor, write_pos: Sequence[int]) -> None:
        """cache [B][n_kv][cap][d] (modified in place), rows [B][n_new][n_kv][d]."""
        B, n_kv, cap, d = cache.shape
        n_new = rows.shape[1]
        if rows.dtype != cache.dtype or tuple(rows.shape) != (B, n_new, n_kv, d):
            raise OracleError("rows must be [B][n_new][n_kv][d] of the cache dtype")
        wp = (ctypes.c_int32 * B)(*[int(x) for x in write_pos])
        st = self.lib.oracle_kv_append(_ptr(cache), _ptr(rows), wp, B, n_new, n_kv, d, cap,
                                       cache.element_size())
        if st != 0:
            raise OracleError(f"oracle_kv_append status {st}")

    def attention(self, layers, owner_map: Sequence[int], layer: int,
                  k_caches: Sequence[Optional[torch.Tensor]],
                  v_caches: Sequence[Optional[torch.Tensor]],
                  q: torch.Tensor, seq_lens: Sequence[int], scale: float,
                  softcap: float = 0.0) -> torch.Tensor:
        """q [B][n_tok][n_q][d]; k_caches[o] [B][n_kv][cap][d] for owner layers (None elsewhere).
        softcap > 0 caps each scaled score s to softcap * tanh(s / softcap); 0 applies none.
        Returns fp64 [B][n_tok][n_q][d]."""
        n_layers = len(layers)
        B, n_tok, n_q, d = q.shape
        spec = layers[layer]
        o = self.resolve_owner(layers, owner_map, layer)
        if o < 0:
            raise OracleError(f"owner resolution failed with status {o}")
        kc = k_caches[o]
        cap = kc.shape[2]
        dt = _dtype_code(q)
        if _dtype_code(kc) != dt:
            raise OracleError("q and caches must share a dtype")
        kp = (ctypes.c_void_p * n_layers)(*[_ptr(t) for t in k_caches])
        vp = (ctypes.c_void_p * n_layers)(*[_ptr(t) for t in v_caches])
        sl = (ctypes.c_int32 * B)(*[int(x) for x in seq_lens])
        om = (ctypes.c_int32 * n_layers)(*[int(x) for x in owner_map])
        arr = (_Layer * n_layers)(*oracle_layers(layers))
        out = torch.empty((B, n_tok, n_q, d), dtype=torch.float64)
        st = self.lib.oracle_attention_softcap(arr, om, n_layers, layer, kp, vp, dt, cap, _ptr(q),
                                               n_tok, sl, B, float(scale), float(softcap),
                                               _ptr(out))
        if st != 0:
            raise OracleError(f"oracle_attention status {st}")
        return out

    def logit_softcap_argmax(self, logits: torch.Tensor, softcap: float):
        """logits [B][V] (bf16 or fp32). Returns (capped fp64 [B][V], index int32 [B]): capped
        = softcap * tanh(x / softcap) (x when softcap == 0), index = the lowest argmax of the raw
        logits, NaN never selected."""
        if logits.dim() != 2:
            raise OracleError("logits must be [B][V]")
        B, V = logits.shape
        capped = torch.empty((B, V), dtype=torch.float64)
        idx = (ctypes.c_int32 * max(B, 1))()
        st = self.lib.oracle_logit_softcap_argmax(_ptr(logits), _dtype_code(logits), B, V,
                                                  float(softcap), _ptr(capped), idx)
        if st != 0:
            raise OracleError(f"oracle_logit_softcap_argmax status {st}")
        return capped, torch.tensor([idx[i] for i in range(B)], dtype=torch.int32)


_cached: dict = {}


def load_oracle(path: Optional[str] = None) -> Oracle:
    path = path or build_oracle()
    if path not in _cached:
        _cached[path] = Oracle(path)
    return _cached[path]
