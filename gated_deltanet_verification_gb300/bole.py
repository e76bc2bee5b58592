"""Python binding of libbole.so: argument marshalling only.

Every step of the verification runs in the library's CUDA kernels; this
module turns torch tensors into device pointers, picks the current CUDA
stream and allocates outputs with torch (device memory plumbing).  It never
falls back to a CPU or PyTorch implementation: if the library is missing the
import of any entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_BAD_TOPOLOGY = 3
ERR_DEPTH = 4
ERR_WORKSPACE = 5
ERR_CUDA = 6
ERR_TIMEOUT = 7

F32 = 0
BF16 = 1
FLAG_FORCE_SIMT = 0x1
FLAG_OVERLAP_LAUNCH = 0x2  # see bole.h: overlap with the previous library call on the stream
FLAG_STATE_VK = 0x4  # state slots stored [B, H, dv, dk] (the serving runtime's slot layout)
FLAG_ONE_TILE_PER_HEAD = 0x8  # small trees: one CTA per (request, head), not two value tiles
FLAG_VALUE_TILES = 0x10  # small trees: two value-tile CTAs per (request, head)
FLAG_INLINE_TOPOLOGY = 0x20  # tree_verify forms the topology itself (no pack_forest first)
MAX_TREE_NODES = 128
STATUS_WORDS = 4

_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


class BoleError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = int(code)
        msg = f"{what}: {status_string(code)} ({code})"
        if self.code == ERR_CUDA:
            msg += f" [CUDA error {last_cuda_error()}: {last_cuda_error_string()}]"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """The loaded libbole.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with "
                    "`python -m gated_deltanet_verification_gb300.build`")
            L = ctypes.CDLL(path)
            P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            U = ctypes.c_uint
            L.bole_status_string.argtypes = [I]
            L.bole_status_string.restype = ctypes.c_char_p
            L.bole_version.argtypes = []
            L.bole_version.restype = I
            L.bole_last_cuda_error.argtypes = []
            L.bole_last_cuda_error.restype = I
            L.bole_last_cuda_error_string.argtypes = []
            L.bole_last_cuda_error_string.restype = ctypes.c_char_p
            L.bole_workspace_size.argtypes = [I, I, I, I, I, I, I, U]
            L.bole_workspace_size.restype = S
            L.bole_pack_forest.argtypes = [P, P, I, I, I, P, P, P, P, P]
            L.bole_pack_forest.restype = I
            L.bole_tree_verify.argtypes = [P, P, P, P, I, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                           I, P, P, P, P, S, P, U, P]
            L.bole_tree_verify.restype = I
            L.bole_tree_verify_noalloc.argtypes = [P, P, P, P, I, P, P, P, P, P, P, P, I, I, I,
                                                   I, I, I, I, P, P, P, P, P]
            L.bole_tree_verify_noalloc.restype = I
            L.bole_commit.argtypes = [P, P, I, P, P, P, P, P, I, I, I, I, I, P, U, P]
            L.bole_commit.restype = I
            I64 = ctypes.c_int64
            L.bole_commit_layers.argtypes = [P, I64, P, I64, I, P, I64, P, I64, P, P, P, I, I, I,
                                             I, I, I, P, U, P]
            L.bole_commit_layers.restype = I
            L.bole_commit_verify.argtypes = [P, P, P, P, P, P, P, I, P, P, P, I, P, P, P, P, I, I,
                                             I, I, I, I, I, P, P, P, P, U, P]
            L.bole_commit_verify.restype = I
            L.bole_conv_gates.argtypes = [P, P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I,
                                          P, P, P, P, P, P, U, P]
            L.bole_conv_gates.restype = I
            L.bole_conv_commit.argtypes = [P, P, I, P, P, P, I, I, I, I, P, U, P]
            L.bole_conv_commit.restype = I
            L.bole_select_workspace_size.argtypes = [I]
            L.bole_select_workspace_size.restype = S
            L.bole_select_forest.argtypes = [P, P, P, P, I, I, I, P, P, P, P, P, S, P, U, P]
            L.bole_select_forest.restype = I
            L.bole_selftest_wait.argtypes = [P, ctypes.c_uint64, P]
            L.bole_selftest_wait.restype = I
            _lib = L
    return _lib


SELFTEST_MAX_WAIT_NS = 1_000_000_000


def selftest_wait(limit_ns: int, *, status=None, stream=None) -> torch.Tensor:
    """bole_selftest_wait: one device thread waits on a barrier nothing
    arrives on, for at most limit_ns; returns the status block, which then
    holds (ERR_TIMEOUT, -1, -1, microseconds waited)."""
    status = new_status() if status is None else status
    _check(lib().bole_selftest_wait(_ptr(status), int(limit_ns), _stream(stream)),
           "bole_selftest_wait")
    return status


def status_string(code: int) -> str:
    return lib().bole_status_string(int(code)).decode()


def version() -> int:
    return lib().bole_version()


def last_cuda_error() -> int:
    """cudaError_t behind this thread's last ERR_CUDA (0 if none)."""
    return lib().bole_last_cuda_error()


def last_cuda_error_string() -> str:
    return lib().bole_last_cuda_error_string().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libbole must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(code: int, what: str) -> None:
    if code != OK:
        raise BoleError(code, what)


def new_status(device="cuda") -> torch.Tensor:
    return torch.zeros(STATUS_WORDS, dtype=torch.int32, device=device)


def check_status(status: torch.Tensor, what: str = "device status") -> None:
    """Synchronising read of a device status block; raises on a recorded fault."""
    st = status.cpu().tolist()
    if st[0] != OK:
        raise BoleError(st[0], f"{what} (request {st[1]}, node {st[2]}, detail {st[3]})")


def workspace_size(B: int, H: int, dk: int, dv: int, max_T: int, max_depth: int,
                   dtype=torch.bfloat16, flags: int = 0) -> int:
    code = BF16 if dtype == torch.bfloat16 else F32
    return int(lib().bole_workspace_size(B, H, dk, dv, max_T, max_depth, code, flags))


def pack_forest(offsets: torch.Tensor, parent: torch.Tensor, max_depth: int, *,
                depth: Optional[torch.Tensor] = None, anc: Optional[torch.Tensor] = None,
                req_depth: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """bole_pack_forest: returns (depth [N], anc [N,4], req_depth [B], status [4])."""
    B = offsets.numel() - 1
    N = parent.numel()
    dev = offsets.device
    depth = torch.empty(N, dtype=torch.int32, device=dev) if depth is None else depth
    anc = torch.empty((N, 4), dtype=torch.int32, device=dev) if anc is None else anc
    req_depth = torch.empty(max(B, 0), dtype=torch.int32, device=dev) if req_depth is None \
        else req_depth
    status = new_status(dev) if status is None else status
    _check(lib().bole_pack_forest(_ptr(offsets), _ptr(parent), B, N, int(max_depth), _ptr(depth),
                                  _ptr(anc), _ptr(req_depth), _ptr(status), _stream(stream)),
           "bole_pack_forest")
    return depth, anc, req_depth, status


def tree_verify(S_pre, q, k, v, gamma, beta, offsets, parent, depth, anc, req_depth, max_T: int,
                max_depth: int, *, O=None, U=None, logP=None, workspace=None, status=None,
                flags: int = 0, stream=None):
    """bole_tree_verify: returns (O, U, logP).  With FLAG_INLINE_TOPOLOGY,
    depth, anc and req_depth may be None."""
    B = offsets.numel() - 1
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    code = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    O = torch.empty((N, H, dv), dtype=q.dtype, device=dev) if O is None else O
    U = torch.empty((N, H, dv), dtype=torch.float32, device=dev) if U is None else U
    logP = torch.empty((N, H), dtype=torch.float32, device=dev) if logP is None else logP
    if workspace is None:
        nbytes = lib().bole_workspace_size(B, H, dk, dv, int(max_T), int(max_depth), code, flags)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    if status is None:
        status = new_status(dev)
    _check(lib().bole_tree_verify(
        _ptr(S_pre), _ptr(q), _ptr(k), _ptr(v), code, _ptr(gamma), _ptr(beta), _ptr(offsets),
        _ptr(parent), _ptr(depth), _ptr(anc), _ptr(req_depth), B, H, dk, dv, N, int(max_T),
        int(max_depth), _ptr(O), _ptr(U), _ptr(logP), _ptr(workspace),
        workspace.numel() * workspace.element_size(),
        _ptr(status), int(flags), _stream(stream)), "bole_tree_verify")
    return O, U, logP


NOALLOC_MAX_FACTOR_ELEMS = 1 << 20


def tree_verify_noalloc(S_pre, q, k, v, gamma, beta, offsets, parent, depth, anc, req_depth,
                        max_T: int, max_depth: int, *, O=None, U=None, logP=None, status=None,
                        stream=None):
    """bole_tree_verify_noalloc: the CUDA-core verification with library-owned
    scratch, for callers that cannot allocate device memory when they verify.
    Returns (O, U, logP); the caller may pass preallocated outputs."""
    B = offsets.numel() - 1
    N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    code = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    O = torch.empty((N, H, dv), dtype=q.dtype, device=dev) if O is None else O
    U = torch.empty((N, H, dv), dtype=torch.float32, device=dev) if U is None else U
    logP = torch.empty((N, H), dtype=torch.float32, device=dev) if logP is None else logP
    if status is None:
        status = new_status(dev)
    _check(lib().bole_tree_verify_noalloc(
        _ptr(S_pre), _ptr(q), _ptr(k), _ptr(v), code, _ptr(gamma), _ptr(beta), _ptr(offsets),
        _ptr(parent), _ptr(depth), _ptr(anc), _ptr(req_depth), B, H, dk, dv, N, int(max_T),
        int(max_depth), _ptr(O), _ptr(U), _ptr(logP), _ptr(status), _stream(stream)),
        "bole_tree_verify_noalloc")
    return O, U, logP


def commit(S, k, U, logP, offsets, parent, accepted, *, status=None, flags: int = 0,
           stream=None) -> torch.Tensor:
    """bole_commit: overwrites S in place with the accepted paths' states; returns S."""
    B = offsets.numel() - 1
    N, H, dk = k.shape
    dv = U.shape[-1]
    if status is None:
        status = new_status(k.device)
    _check(lib().bole_commit(_ptr(S), _ptr(k), _dtype_code(k), _ptr(U), _ptr(logP),
                             _ptr(offsets), _ptr(parent), _ptr(accepted), B, H, dk, dv, N,
                             _ptr(status), int(flags), _stream(stream)), "bole_commit")
    return S


def commit_verify(S, k_prev, U_prev, logP_prev, offsets_prev, parent_prev, accepted_prev, q, k,
                  v, gamma, beta, offsets, parent, max_T: int, max_depth: int, *, O=None, U=None,
                  logP=None, status=None, flags: int = 0, stream=None):
    """bole_commit_verify: the previous round's commit applied to S in place,
    then this round's verification from the committed state (its topology
    formed in the kernel).  Returns (O, U, logP); U and logP must be other
    buffers than U_prev and logP_prev."""
    B = offsets.numel() - 1
    N, H, dk = q.shape
    dv = v.shape[-1]
    N_prev = k_prev.shape[0]
    dev = q.device
    code = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype or k_prev.dtype != q.dtype:
        raise TypeError("q, k, v and k_prev must share one dtype")
    O = torch.empty((N, H, dv), dtype=q.dtype, device=dev) if O is None else O
    U = torch.empty((N, H, dv), dtype=torch.float32, device=dev) if U is None else U
    logP = torch.empty((N, H), dtype=torch.float32, device=dev) if logP is None else logP
    if status is None:
        status = new_status(dev)
    _check(lib().bole_commit_verify(
        _ptr(S), _ptr(k_prev), _ptr(U_prev), _ptr(logP_prev), _ptr(offsets_prev),
        _ptr(parent_prev), _ptr(accepted_prev), N_prev, _ptr(q), _ptr(k), _ptr(v), code,
        _ptr(gamma), _ptr(beta), _ptr(offsets), _ptr(parent), B, H, dk, dv, N, int(max_T),
        int(max_depth), _ptr(O), _ptr(U), _ptr(logP), _ptr(status), int(flags), _stream(stream)),
        "bole_commit_verify")
    return O, U, logP


MAX_CONV_WIDTH = 8
MAX_CANDIDATES = 1024
SELECT_MAX_REQUESTS = 4096


def select_forest(p, cand_offsets, cand_parent, budget: int, *, caps=None, offsets=None,
                  parent=None, src=None, rho=None, workspace=None, status=None, flags: int = 0,
                  stream=None):
    """bole_select_forest: the round's proposal selection and forest build on
    the device.  p [M] float32, cand_offsets [B+1], cand_parent [M] int32,
    caps [B] int32 or None.  Returns (offsets [B+1], parent [budget],
    src [budget], rho [M], status); offsets[B] (on the device) is the node
    count -- the forest feeds pack_forest with N = budget."""
    B = cand_offsets.numel() - 1
    M = p.numel()
    dev = p.device
    i32 = torch.int32
    offsets = torch.empty(B + 1, dtype=i32, device=dev) if offsets is None else offsets
    parent = torch.empty(max(budget, 1), dtype=i32, device=dev) if parent is None else parent
    src = torch.empty(max(budget, 1), dtype=i32, device=dev) if src is None else src
    rho = torch.empty(max(M, 1), dtype=torch.float32, device=dev) if rho is None else rho
    if workspace is None:
        n = int(lib().bole_select_workspace_size(B))
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    status = new_status(dev) if status is None else status
    _check(lib().bole_select_forest(
        _ptr(p), _ptr(cand_offsets), _ptr(cand_parent), _ptr(caps), B, M, int(budget),
        _ptr(offsets), _ptr(parent), _ptr(src), _ptr(rho), _ptr(workspace),
        workspace.numel() * workspace.element_size(),
        _ptr(status), int(flags), _stream(stream)), "bole_select_forest")
    return offsets, parent, src, rho, status


def conv_gates(x, conv_state, conv_w, conv_b, a, b, offsets, parent, H: int, dk: int, dv: int,
               max_T: int, *, gate_scale=None, gate_bias=None, q=None, k=None, v=None, gamma=None,
               beta=None, status=None, flags: int = 0, stream=None):
    """bole_conv_gates: stage 1 of a GDN layer on a packed forest.

    x [N, C] (C = H (2 dk + dv); q channels, then k, then v), conv_state
    [B, W-1, C] (same dtype), conv_w [C, W] float32, conv_b [C] float32 or
    None, a, b [N, H] float32; max_T bounds the tree sizes.  Returns (q, k, v, gamma, beta) in the layouts
    bole_tree_verify takes."""
    B = offsets.numel() - 1
    N, C = x.shape
    W = conv_w.shape[1]
    dev = x.device
    code = _dtype_code(x)
    if C != H * (2 * dk + dv):
        raise ValueError("x must hold H (2 dk + dv) channels per node")
    if conv_state is not None and conv_state.dtype != x.dtype:
        raise TypeError("conv_state must have x's dtype")
    q = torch.empty((N, H, dk), dtype=x.dtype, device=dev) if q is None else q
    k = torch.empty((N, H, dk), dtype=x.dtype, device=dev) if k is None else k
    v = torch.empty((N, H, dv), dtype=x.dtype, device=dev) if v is None else v
    gamma = torch.empty((N, H), dtype=torch.float32, device=dev) if gamma is None else gamma
    beta = torch.empty((N, H), dtype=torch.float32, device=dev) if beta is None else beta
    if status is None:
        status = new_status(dev)
    _check(lib().bole_conv_gates(
        _ptr(x), _ptr(conv_state), _ptr(conv_w), _ptr(conv_b), _ptr(a), _ptr(b),
        _ptr(gate_scale), _ptr(gate_bias), code, _ptr(offsets), _ptr(parent), B, H, dk, dv, N,
        int(max_T), W,
        _ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(beta), _ptr(status), int(flags),
        _stream(stream)), "bole_conv_gates")
    return q, k, v, gamma, beta


def conv_commit(conv_state, x, offsets, parent, accepted, *, status=None, flags: int = 0,
                stream=None):
    """bole_conv_commit: conv_state [B, W-1, C] becomes, in place, the last
    W-1 tokens ending at each request's accepted node.  Returns conv_state."""
    B = offsets.numel() - 1
    N, C = x.shape
    W = conv_state.shape[1] + 1
    if status is None:
        status = new_status(x.device)
    _check(lib().bole_conv_commit(_ptr(conv_state), _ptr(x), _dtype_code(x), _ptr(offsets),
                                  _ptr(parent), _ptr(accepted), B, C, W, N, _ptr(status),
                                  int(flags), _stream(stream)), "bole_conv_commit")
    return conv_state


def _layer_stride(t: torch.Tensor, n_layers: int) -> int:
    """Element stride between the layers of a [layers, ...] tensor whose
    per-layer slices are contiguous."""
    if t.dim() < 2 or t.shape[0] != n_layers or not t[0].is_contiguous():
        raise ValueError("expected a [layers, ...] tensor with contiguous layer slices")
    return int(t.stride(0)) if n_layers > 1 else 0


def commit_layers(S, k, U, logP, offsets, parent, accepted, *, status=None, flags: int = 0,
                  stream=None) -> torch.Tensor:
    """bole_commit_layers: one launch commits every layer of a round.

    S [layers, B, H, dk, dv] (or [layers, B, H, dv, dk] with FLAG_STATE_VK),
    k [layers, N, H, dk], U [layers, N, H, dv], logP [layers, N, H]; each
    layer's slice contiguous, the layer strides taken from the tensors (a
    slice of a larger preallocated pool works).  Overwrites S in place and
    returns it."""
    n_layers = S.shape[0]
    B = offsets.numel() - 1
    _, N, H, dk = k.shape
    dv = U.shape[-1]
    if status is None:
        status = new_status(k.device)
    _check(lib().bole_commit_layers(
        S.data_ptr(), _layer_stride(S, n_layers), k.data_ptr(), _layer_stride(k, n_layers),
        _dtype_code(k), U.data_ptr(), _layer_stride(U, n_layers), logP.data_ptr(),
        _layer_stride(logP, n_layers), _ptr(offsets), _ptr(parent), _ptr(accepted), n_layers, B,
        H, dk, dv, N, _ptr(status), int(flags), _stream(stream)), "bole_commit_layers")
    return S


__all__ = ["selftest_wait", "SELFTEST_MAX_WAIT_NS", "select_forest", "MAX_CANDIDATES", "SELECT_MAX_REQUESTS", "conv_gates", "conv_commit", "MAX_CONV_WIDTH", "commit_layers", "FLAG_STATE_VK", "lib", "library_path", "status_string", "version", "workspace_size", "pack_forest",
           "tree_verify", "tree_verify_noalloc", "commit", "new_status", "check_status", "BoleError", "OK",
           "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_BAD_TOPOLOGY", "ERR_DEPTH",
           "ERR_WORKSPACE", "ERR_CUDA", "ERR_TIMEOUT", "F32", "BF16", "FLAG_FORCE_SIMT",
           "FLAG_OVERLAP_LAUNCH"]
