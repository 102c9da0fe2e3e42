"""ctypes wrapper of the float64 C oracle (``oracle.c``).

TEST INFRASTRUCTURE: used by the test suite, the smoke check and the benchmark's CPU legs
only. Shares no code with the CUDA path. Inputs are numpy arrays on the host: logits as
``float32`` or as ``uint16`` holding bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, BF16 = 0, 1
DRAFT_POINT, DRAFT_PROBS_F32, DRAFT_LOGITS = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")


def compile_oracle(src: str = SOURCE, out: str = LIBRARY, force: bool = False) -> str:
    """Compile an oracle source into a shared library with gcc. No contraction and no
    fast-math, so x86 and Arm hosts round identically."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


class Oracle:
    """One loaded oracle library (the default build, or a planted-mistake build in tests)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_build_mask.argtypes = [P, i32, i32, P, P, P]
        lib.oracle_row_stats.argtypes = [P, i32, i64, f64, P, P, P, P]
        lib.oracle_row_softmax.argtypes = [P, i32, i64, f64, P]
        lib.oracle_inv_cdf.argtypes = [P, i64, f64, P, P]
        lib.oracle_inv_cdf.restype = i64
        lib.oracle_verify_greedy.argtypes = [P, i32, i32, i32, i64, P, P, P, P, P, P, P, i32]
        lib.oracle_verify_sample.argtypes = [P, i32, i32, i32, i64, P, P, P, i32, i32, f64,
                                             P, P, P, P, P, P, P, P, P, P, P, i32]
        lib.oracle_max_threads.restype = i32
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def build_mask(self, parent: np.ndarray):
        """parent int32 [B, N] -> (anc uint64 [B, N], depth int32 [B, N], status int32 [B])."""
        parent = np.ascontiguousarray(parent, dtype=np.int32)
        B, N = parent.shape
        anc = np.zeros((B, N), np.uint64)
        depth = np.zeros((B, N), np.int32)
        status = np.zeros(B, np.int32)
        rc = self.lib.oracle_build_mask(_ptr(parent), B, N, _ptr(anc), _ptr(depth),
                                        _ptr(status))
        if rc != 0:
            raise ValueError("oracle_build_mask rejected its arguments")
        return anc, depth, status

    def row_stats(self, row: np.ndarray, T: float):
        """One row -> (m, S, argmax, bad) with S = sum exp((z - m)/T) (0 when T == 0)."""
        row = np.ascontiguousarray(row)
        m, S = ctypes.c_double(), ctypes.c_double()
        a, bad = ctypes.c_int64(), ctypes.c_int32()
        rc = self.lib.oracle_row_stats(_ptr(row), _dtype_code(row), row.shape[-1], float(T),
                                       ctypes.byref(m), ctypes.byref(S), ctypes.byref(a),
                                       ctypes.byref(bad))
        if rc != 0:
            raise ValueError("oracle_row_stats rejected its arguments")
        return m.value, S.value, a.value, bad.value

    def row_softmax(self, row: np.ndarray, T: float) -> np.ndarray:
        row = np.ascontiguousarray(row)
        p = np.empty(row.shape[-1], np.float64)
        if self.lib.oracle_row_softmax(_ptr(row), _dtype_code(row), row.shape[-1], float(T),
                                       _ptr(p)) != 0:
            raise ValueError("oracle_row_softmax rejected its arguments")
        return p

    def inv_cdf(self, r: np.ndarray, u: float, window: bool = False):
        """-> (token, margin), or (token, margin, (first, last token of the draw window))."""
        r = np.ascontiguousarray(r, dtype=np.float64)
        margin = ctypes.c_double()
        win = np.zeros(2, np.int64)
        v = self.lib.oracle_inv_cdf(_ptr(r), r.shape[0], float(u), ctypes.byref(margin),
                                    _ptr(win))
        if window:
            return int(v), margin.value, (int(win[0]), int(win[1]))
        return int(v), margin.value

    @staticmethod
    def _outputs(B, N):
        return (np.zeros(B, np.int32), np.zeros((B, N), np.int32), np.zeros((B, N), np.int32),
                np.zeros(B, np.int32), np.zeros(B, np.int32))

    def verify_greedy(self, logits: np.ndarray, draft_token: np.ndarray, parent: np.ndarray,
                      nthreads: int = 1) -> dict:
        """logits [B, N, V] float32 or bf16 bits (uint16); draft_token, parent int32 [B, N]."""
        logits = np.ascontiguousarray(logits)
        B, N, V = logits.shape
        tok = np.ascontiguousarray(draft_token, dtype=np.int32)
        par = np.ascontiguousarray(parent, dtype=np.int32)
        al, ot, kv, bo, st = self._outputs(B, N)
        rc = self.lib.oracle_verify_greedy(_ptr(logits), _dtype_code(logits), B, N, V,
                                           _ptr(tok), _ptr(par), _ptr(al), _ptr(ot), _ptr(kv),
                                           _ptr(bo), _ptr(st), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_verify_greedy rejected its arguments")
        return dict(accept_len=al, out_tokens=ot, kv_commit=kv, bonus=bo, status=st)

    def verify_sample(self, logits: np.ndarray, draft_token: np.ndarray, parent: np.ndarray,
                      temperature: float, uniforms: np.ndarray, draft: np.ndarray | None = None,
                      draft_kind: int = DRAFT_POINT, nthreads: int = 1) -> dict:
        """Sampling verify. uniforms float32 [B, N+1]. ``draft`` is None (point-mass drafts),
        float32 probabilities [B, N, V] (``DRAFT_PROBS_F32``) or logits (``DRAFT_LOGITS``,
        float32 or bf16 bits)."""
        logits = np.ascontiguousarray(logits)
        B, N, V = logits.shape
        tok = np.ascontiguousarray(draft_token, dtype=np.int32)
        par = np.ascontiguousarray(parent, dtype=np.int32)
        u = np.ascontiguousarray(uniforms, dtype=np.float32)
        assert u.shape == (B, N + 1), (u.shape, B, N)
        ddt = 0
        if draft is not None:
            draft = np.ascontiguousarray(draft)
            assert draft.shape == (B, N, V)
            ddt = _dtype_code(draft)
        al, ot, kv, bo, st = self._outputs(B, N)
        dm = np.zeros(B, np.float64)
        cm = np.zeros(B, np.float64)
        ca = np.zeros(B, np.int32)
        cw = np.zeros((B, 2), np.int32)
        dg = np.zeros(B, np.int32)
        rc = self.lib.oracle_verify_sample(_ptr(logits), _dtype_code(logits), B, N, V,
                                           _ptr(tok), _ptr(par), _ptr(draft), int(draft_kind),
                                           ddt, float(temperature), _ptr(u), _ptr(al), _ptr(ot),
                                           _ptr(kv), _ptr(bo), _ptr(st), _ptr(dm), _ptr(cm),
                                           _ptr(ca), _ptr(cw), _ptr(dg), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_verify_sample rejected its arguments")
        return dict(accept_len=al, out_tokens=ot, kv_commit=kv, bonus=bo, status=st,
                    decision_margin=dm, cdf_margin=cm, cdf_alt=ca, cdf_lo=cw[:, 0].copy(),
                    cdf_hi=cw[:, 1].copy(), degenerate=dg)


_default: Oracle | None = None
_lock = threading.Lock()


def default() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(compile_oracle())
    return _default


def build(force: bool = False) -> str:
    return compile_oracle(force=force)
