"""ctypes wrapper around the C oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. It imports nothing
from the CUDA library's package and the CUDA library never imports it.

Every function takes and returns numpy arrays. bf16 tensors are passed as
``uint16`` arrays holding the raw bf16 bits.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "moe_oracle.c")
LIB = os.path.join(_HERE, "libmoe_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(src: str = SRC, out: str = LIB, extra: list[str] | None = None) -> str:
    """Compile the oracle into a shared library (plain cc, portable flags)."""
    cc = os.environ.get("CC", "cc")
    cmd = [cc, *CFLAGS, *(extra or []), src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build(src: str, out: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_logits.restype = ctypes.c_int
    lib.oracle_logits.argtypes = [i64, i32, i32, P, P, P, P]
    lib.oracle_topk.restype = ctypes.c_int
    lib.oracle_topk.argtypes = [i64, i32, i32, P, P, P]
    lib.oracle_route.restype = ctypes.c_int
    lib.oracle_route.argtypes = [i64, i32, i32, i32, P, P, P, P, P, P]
    lib.oracle_gate_weights_full.restype = ctypes.c_int
    lib.oracle_gate_weights_full.argtypes = [i64, i32, i32, P, P, P]
    lib.oracle_shared_gate.restype = ctypes.c_int
    lib.oracle_shared_gate.argtypes = [i64, i32, P, P, P]
    lib.oracle_layer_rows_gated.restype = ctypes.c_int
    lib.oracle_layer_rows_gated.argtypes = [i64, i32, i32, i32, i32, i32, P, i64, P, P,
                                            P, P, P, P, P, P, P, P, P]
    lib.oracle_permute.restype = ctypes.c_int
    lib.oracle_permute.argtypes = [i64, i32, P, P, P, P, P]
    lib.oracle_expert_row.restype = ctypes.c_int
    lib.oracle_expert_row.argtypes = [i32, i32, P, P, P, P, P]
    lib.oracle_layer_rows.restype = ctypes.c_int
    lib.oracle_layer_rows.argtypes = [i64, i32, i32, i32, i32, i32, P, i64, P, P,
                                      P, P, P, P, P, P, P, P]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if stale) the oracle library. ``path`` loads a variant."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build(SRC, LIB):
                build()
            _lib = _declare(ctypes.CDLL(LIB))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected raw bf16 bits as uint16, got {a.dtype}")
    return a


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


class Oracle:
    """Bound view of one oracle library build (the default one unless ``path``)."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def logits(self, x, Wg, bias=None) -> np.ndarray:
        x, Wg = _u16(x), _u16(Wg)
        T, H = x.shape
        E = Wg.shape[1]
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        out = np.empty((T, E), np.float32)
        _check(self.lib.oracle_logits(T, H, E, _ptr(x), _ptr(Wg), _ptr(b), _ptr(out)), "logits")
        return out

    def topk(self, logits, k: int):
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        _check(self.lib.oracle_topk(T, E, k, _ptr(logits), _ptr(idx), _ptr(w)), "topk")
        return idx, w

    def gate_weights_full(self, logits, topk_idx) -> np.ndarray:
        """Weights without renormalisation (softmax over all E at the selected ids)."""
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        T, E = logits.shape
        k = idx.shape[1]
        w = np.empty((T, k), np.float32)
        _check(self.lib.oracle_gate_weights_full(T, E, k, _ptr(logits), _ptr(idx), _ptr(w)),
               "gate_weights_full")
        return w

    def shared_gate(self, x, wsg) -> np.ndarray:
        """s[t] = sigmoid(x[t] . wsg) (fp64)."""
        x, wsg = _u16(x), _u16(wsg)
        T, H = x.shape
        out = np.empty(T, np.float64)
        _check(self.lib.oracle_shared_gate(T, H, _ptr(x), _ptr(wsg), _ptr(out)), "shared_gate")
        return out

    def route(self, x, Wg, k: int, bias=None):
        """Returns (logits[T,E] f32, topk_idx[T,k] i32, topk_w[T,k] f32)."""
        x, Wg = _u16(x), _u16(Wg)
        T, H = x.shape
        E = Wg.shape[1]
        b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
        logits = np.empty((T, E), np.float32)
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        _check(self.lib.oracle_route(T, H, E, k, _ptr(x), _ptr(Wg), _ptr(b), _ptr(logits),
                                     _ptr(idx), _ptr(w)), "route")
        return logits, idx, w

    def permute(self, topk_idx, E: int):
        """Returns (counts[E], offsets[E+1], src_row[R], inv_pos[R]), all int32."""
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32).reshape(-1)
        R = idx.size
        counts = np.empty(E, np.int32)
        offsets = np.empty(E + 1, np.int32)
        src_row = np.empty(R, np.int32)
        inv_pos = np.empty(R, np.int32)
        _check(self.lib.oracle_permute(R, E, _ptr(idx), _ptr(counts), _ptr(offsets),
                                       _ptr(src_row), _ptr(inv_pos)), "permute")
        return counts, offsets, src_row, inv_pos

    def expert_row(self, xrow, W1e, W3e, W2e) -> np.ndarray:
        xrow, W1e, W3e, W2e = _u16(xrow), _u16(W1e), _u16(W3e), _u16(W2e)
        H, F = W1e.shape
        y = np.empty(H, np.float64)
        _check(self.lib.oracle_expert_row(H, F, _ptr(xrow), _ptr(W1e), _ptr(W3e), _ptr(W2e),
                                          _ptr(y)), "expert_row")
        return y

    def layer_rows(self, tokens, topk_idx, topk_w, x, W1, W3, W2, W1s=None, W3s=None,
                   W2s=None, shared_scale=None) -> np.ndarray:
        """out[len(tokens), H] (fp64) for the listed tokens, given the routing;
        shared_scale[T] (fp64) scales the shared expert (default 1)."""
        x, W1, W3, W2 = _u16(x), _u16(W1), _u16(W3), _u16(W2)
        T, H = x.shape
        E, _, F = W1.shape
        k = topk_idx.shape[1]
        Fs = 0
        if W1s is not None:
            W1s, W3s, W2s = _u16(W1s), _u16(W3s), _u16(W2s)
            Fs = W1s.shape[1]
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
        w = np.ascontiguousarray(topk_w, dtype=np.float32)
        out = np.empty((tokens.size, H), np.float64)
        if shared_scale is None:
            _check(self.lib.oracle_layer_rows(T, H, F, E, k, Fs, _ptr(tokens), tokens.size, _ptr(idx),
                                              _ptr(w), _ptr(x), _ptr(W1), _ptr(W3), _ptr(W2),
                                              _ptr(W1s), _ptr(W3s), _ptr(W2s), _ptr(out)),
                   "layer_rows")
        else:
            sc = np.ascontiguousarray(shared_scale, dtype=np.float64)
            _check(self.lib.oracle_layer_rows_gated(T, H, F, E, k, Fs, _ptr(tokens), tokens.size,
                                                    _ptr(idx), _ptr(w), _ptr(x), _ptr(W1), _ptr(W3),
                                                    _ptr(W2), _ptr(W1s), _ptr(W3s), _ptr(W2s),
                                                    _ptr(sc), _ptr(out)),
                   "layer_rows_gated")
        return out

    def layer_forward(self, x, Wg, W1, W3, W2, k: int, bias=None, W1s=None, W3s=None, W2s=None,
                      tokens=None, renormalize=True, wsg=None):
        """Route, then the output rows for ``tokens`` (all tokens by default).
        renormalize=False takes the weights over all E (reading R3'); wsg gates
        the shared expert with sigmoid(x . wsg) (reading R5').

        Returns a dict with logits, topk_idx, topk_w, counts, offsets, src_row,
        inv_pos, tokens and out (fp64)."""
        logits, idx, w = self.route(x, Wg, k, bias)
        if not renormalize:
            w = self.gate_weights_full(logits, idx)
        scale = None if wsg is None else self.shared_gate(x, wsg)
        E = Wg.shape[1]
        counts, offsets, src_row, inv_pos = self.permute(idx, E)
        if tokens is None:
            tokens = np.arange(x.shape[0], dtype=np.int64)
        out = self.layer_rows(tokens, idx, w, x, W1, W3, W2, W1s, W3s, W2s, shared_scale=scale)
        return dict(logits=logits, topk_idx=idx, topk_w=w, counts=counts, offsets=offsets,
                    src_row=src_row, inv_pos=inv_pos, tokens=np.asarray(tokens), out=out)
