"""CPU oracle for closed-form GDN tree verification -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
and its Python binding) never imports, links or calls it, and the two share
no code: the only common module is the seeded input generator, which holds
none of the method's arithmetic.

The arithmetic lives in `bole_oracle.c` (plain C, double precision, one
snapshot per node).  This wrapper compiles it with gcc on first use, upcasts
inputs to float64 and runs it on `nthreads` host threads.

Pins (tests under `tests/test_oracle_*.py`, all CPU): a hand-derived worked
example (`tests/golden/`), dense Theorem 1 via a library linear solve,
nilpotency G^(d+1) = 0, the Neumann sum equal to the inverse, the single-chain
reduction to token-order GDN, star and beta = 0 special cases, sibling
relabelling and prefix causality invariants, brute-force transitive closure
for the ancestor masks, and planted mistakes that every pin set must catch.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bole_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libbole_oracle.so")

OK = 0
BAD_TOPOLOGY = 3
DEPTH = 4

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library (plain gcc, portable flags)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _needs_build(path: str, src: str) -> bool:
    return (not os.path.exists(path)) or os.path.getmtime(path) < os.path.getmtime(src)


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building if needed) an oracle library; `path` selects another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build(_LIB_PATH, _SRC):
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_pack.argtypes = [I, P, P, I, P, P, P]
    lib.oracle_pack.restype = I
    lib.oracle_verify.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, I, I, I]
    lib.oracle_verify.restype = I
    lib.oracle_commit.argtypes = [I, I, I, I, P, P, P, P, P, P, P, P, P, I, I, I]
    lib.oracle_commit.restype = I
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def pack(offsets, parent, max_depth: int, lib=None):
    """Depth, ancestor-or-self masks [N,4] uint32, per-request depth, status."""
    lib = lib or load()
    offsets, parent = _i32(offsets), _i32(parent)
    B = len(offsets) - 1
    N = int(offsets[-1]) if B >= 0 else 0
    depth = np.zeros(max(N, 1), dtype=np.int32)
    anc = np.zeros((max(N, 1), 4), dtype=np.uint32)
    req = np.zeros(max(B, 1), dtype=np.int32)
    st = lib.oracle_pack(B, _ptr(offsets), _ptr(parent), int(max_depth), _ptr(depth), _ptr(anc),
                         _ptr(req))
    return depth[:N], anc[:N], req[:B], int(st)


def verify(batch, nthreads: Optional[int] = None, unit_begin: int = 0, unit_end: int = -1,
           lib=None):
    """Sequential tree execution.  Returns (O, U, logP) as float64 arrays with
    layouts [N,H,dv], [N,H,dv], [N,H]."""
    lib = lib or load()
    b = batch
    offsets, parent = _i32(b.offsets), _i32(b.parent)
    S, q, k, v = _f64(b.S_pre), _f64(b.q), _f64(b.k), _f64(b.v)
    g, bt = _f64(b.gamma), _f64(b.beta)
    N = b.N
    O = np.zeros((N, b.H, b.dv))
    U = np.zeros((N, b.H, b.dv))
    logP = np.zeros((N, b.H))
    st = lib.oracle_verify(b.B, b.H, b.dk, b.dv, _ptr(offsets), _ptr(parent), _ptr(S), _ptr(q),
                           _ptr(k), _ptr(v), _ptr(g), _ptr(bt), _ptr(O), _ptr(U), _ptr(logP),
                           int(unit_begin), int(unit_end), int(nthreads or default_threads()))
    if st != OK:
        raise ValueError(f"oracle_verify status {st}")
    return O, U, logP


class Prepared:
    """A batch converted once (float64 copies, output arrays allocated once)
    for repeated calls over ranges of (request, head) units: the same C
    routines and arguments as verify() and commit(), without re-marshalling
    the whole batch on every call.  The benchmark's reference arm times the
    oracle this way; outputs are overwritten by each call."""

    def __init__(self, batch, nthreads: Optional[int] = None, lib=None):
        self.lib = lib or load()
        b = self.b = batch
        self.nthreads = int(nthreads or default_threads())
        self.offsets, self.parent = _i32(b.offsets), _i32(b.parent)
        self.acc = _i32(b.accepted)
        self.S, self.q, self.k, self.v = _f64(b.S_pre), _f64(b.q), _f64(b.k), _f64(b.v)
        self.g, self.bt = _f64(b.gamma), _f64(b.beta)
        self.O = np.zeros((b.N, b.H, b.dv))
        self.U = np.zeros((b.N, b.H, b.dv))
        self.logP = np.zeros((b.N, b.H))
        self.S_new = np.zeros((b.B, b.H, b.dk, b.dv))

    def verify(self, unit_begin: int, unit_end: int) -> None:
        b = self.b
        st = self.lib.oracle_verify(b.B, b.H, b.dk, b.dv, _ptr(self.offsets), _ptr(self.parent),
                                    _ptr(self.S), _ptr(self.q), _ptr(self.k), _ptr(self.v),
                                    _ptr(self.g), _ptr(self.bt), _ptr(self.O), _ptr(self.U),
                                    _ptr(self.logP), int(unit_begin), int(unit_end),
                                    self.nthreads)
        if st != OK:
            raise ValueError(f"oracle_verify status {st}")

    def commit(self, unit_begin: int, unit_end: int) -> None:
        b = self.b
        st = self.lib.oracle_commit(b.B, b.H, b.dk, b.dv, _ptr(self.offsets), _ptr(self.parent),
                                    _ptr(self.acc), _ptr(self.S), _ptr(self.k), _ptr(self.v),
                                    _ptr(self.g), _ptr(self.bt), _ptr(self.S_new),
                                    int(unit_begin), int(unit_end), self.nthreads)
        if st != OK:
            raise ValueError(f"oracle_commit status {st}")


def commit(batch, accepted=None, nthreads: Optional[int] = None, unit_begin: int = 0,
           unit_end: int = -1, lib=None):
    """Committed state [B,H,dk,dv] float64 after replaying each accepted path
    (units outside [unit_begin, unit_end) are left zero)."""
    lib = lib or load()
    b = batch
    acc = _i32(b.accepted if accepted is None else accepted)
    offsets, parent = _i32(b.offsets), _i32(b.parent)
    S, k, v = _f64(b.S_pre), _f64(b.k), _f64(b.v)
    g, bt = _f64(b.gamma), _f64(b.beta)
    S_new = np.zeros((b.B, b.H, b.dk, b.dv))
    st = lib.oracle_commit(b.B, b.H, b.dk, b.dv, _ptr(offsets), _ptr(parent), _ptr(acc), _ptr(S),
                           _ptr(k), _ptr(v), _ptr(g), _ptr(bt), _ptr(S_new), int(unit_begin),
                           int(unit_end), int(nthreads or default_threads()))
    if st != OK:
        raise ValueError(f"oracle_commit status {st}")
    return S_new


def commit_layers(batches, accepted=None, state_layout: str = "kv",
                  nthreads: Optional[int] = None, lib=None):
    """Unified cross-layer commit (Section IV-D, state lifecycle; the SGLang
    integration's single batched launch of Eq. (10) over every recurrent
    layer's P, K, U): the layers of one round share the forest and the
    accepted nodes, and layer l's committed state is that layer's own commit
    (each layer's recurrence involves only its own S_pre and operands).

    Returns [L, B, H, dk, dv], or with state_layout="vk" the serving runtime's
    canonical slot layout [L, B, H, dv, dk] (Section IV-D: slots stored
    [H, dv, dk])."""
    if state_layout not in ("kv", "vk"):
        raise ValueError(state_layout)
    b0 = batches[0]
    for b in batches[1:]:
        if not (np.array_equal(b.offsets, b0.offsets) and np.array_equal(b.parent, b0.parent)):
            raise ValueError("the layers of one round share the packed forest")
    acc = b0.accepted if accepted is None else accepted
    out = np.stack([commit(b, acc, nthreads, lib=lib) for b in batches])
    if state_layout == "vk":
        out = np.ascontiguousarray(out.transpose(0, 1, 2, 4, 3))
    return out


__all__ = ["build", "load", "pack", "verify", "commit", "commit_layers", "default_threads", "OK",
           "BAD_TOPOLOGY", "DEPTH"]
