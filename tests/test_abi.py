"""The C ABI library: it builds, loads without a GPU, exports every entry
point include/*.h declares, and rejects host-checkable argument errors
before touching CUDA.  CPU only (no compute calls)."""
import ctypes
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(bole_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from gated_deltanet_verification_gb300 import build
    path = build.build()
    from gated_deltanet_verification_gb300 import bole
    return bole.lib()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert {"bole_pack_forest", "bole_tree_verify", "bole_commit", "bole_workspace_size",
            "bole_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), name


def test_selftest_wait_host_validation(lib):
    """Bad arguments are refused before anything is launched."""
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    f = lib.bole_selftest_wait
    assert f(None, 1000, None) == bole.ERR_INVALID_ARG               # no status block
    assert f(c((1 << 20) + 4), 1000, None) == bole.ERR_INVALID_ARG   # misaligned status
    assert f(c(1 << 20), bole.SELFTEST_MAX_WAIT_NS + 1, None) == bole.ERR_INVALID_ARG


def test_status_strings(lib):
    from gated_deltanet_verification_gb300 import bole
    assert bole.status_string(0) == "ok"
    for code in range(1, 8):
        assert bole.status_string(code) not in ("ok", "unknown status")
    assert bole.status_string(99) == "unknown status"


def test_workspace_size_rules(lib):
    f = lib.bole_workspace_size
    f.restype = ctypes.c_size_t
    # fp32 inputs use the CUDA-core path: two dense T x T factors per unit
    assert f(2, 3, 16, 16, 8, 3, 0, 0) == 2 * 4 * 2 * 3 * 8 * 8
    # bf16, dk = dv = 128, trees <= 64 nodes of depth <= 15: tensor-core kernel, every
    # intermediate on chip, no workspace
    assert f(2, 3, 128, 128, 64, 15, 1, 0) == 0
    # deeper or larger trees (up to 128 nodes): the large-tree tensor-core kernel keeps
    # [M; W] in tensor memory, no workspace either
    assert f(2, 3, 128, 128, 64, 16, 1, 0) == 0
    assert f(2, 3, 128, 128, 128, 127, 1, 0) == 0
    # forced CUDA-core path: two dense T x T factors per unit
    assert f(2, 3, 128, 128, 64, 8, 1, 1) == 2 * 4 * 2 * 3 * 64 * 64
    # invalid sizes report 0
    assert f(2, 3, 12, 16, 8, 3, 0, 0) == 0
    assert f(2, 3, 16, 16, 129, 3, 0, 0) == 0
    assert f(2, 0, 16, 16, 8, 3, 0, 0) == 0
    assert f(2, 3, 16, 16, 8, 128, 0, 0) == 0


def test_host_validation_without_gpu(lib):
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake = c(1 << 20)  # never dereferenced: validation fails first
    # pack: null offsets
    assert lib.bole_pack_forest(None, fake, 1, 4, 3, fake, fake, fake, fake, None) == \
        bole.ERR_INVALID_ARG
    # pack: max_depth out of range
    assert lib.bole_pack_forest(fake, fake, 1, 4, 200, fake, fake, fake, fake, None) == \
        bole.ERR_INVALID_ARG
    args = [fake, fake, fake, fake, 1, fake, fake, fake, fake, fake, fake, fake]
    # dk not a multiple of 16
    assert lib.bole_tree_verify(*args, 1, 1, 24, 128, 4, 8, 3, fake, fake, fake, fake, 0, fake,
                                0, None) == bole.ERR_INVALID_ARG
    # N larger than B * max_T
    assert lib.bole_tree_verify(*args, 1, 1, 128, 128, 65, 64, 3, fake, fake, fake, fake, 0, fake,
                                0, None) == bole.ERR_INVALID_ARG
    # misaligned state pointer
    args_mis = [c((1 << 20) + 4)] + args[1:]
    assert lib.bole_tree_verify(*args_mis, 1, 1, 128, 128, 4, 8, 3, fake, fake, fake, fake, 0,
                                fake, 0, None) == bole.ERR_INVALID_ARG
    # CUDA-core path needs a workspace
    assert lib.bole_tree_verify(*args, 1, 1, 128, 128, 4, 8, 3, fake, fake, fake, None, 0, fake,
                                bole.FLAG_FORCE_SIMT, None) == bole.ERR_WORKSPACE
    # commit: null accepted
    assert lib.bole_commit(fake, fake, 1, fake, fake, fake, fake, None, 1, 1, 128, 128, 4, fake,
                           0, None) == bole.ERR_INVALID_ARG


def test_commit_layers_host_validation_without_gpu(lib):
    """bole_commit_layers rejects layer strides that would overlap or misalign
    the per-layer slices, before any launch."""
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake = c(1 << 20)
    B, H, dk, dv, N = 2, 3, 128, 128, 8
    slice_ = B * H * dk * dv

    def call(n_layers, s_ls=slice_, k_ls=N * H * dk, u_ls=N * H * dv, lp_ls=N * H, S=fake,
             flags=0):
        return lib.bole_commit_layers(S, s_ls, fake, k_ls, 1, fake, u_ls, fake, lp_ls, fake,
                                      fake, fake, n_layers, B, H, dk, dv, N, fake, flags, None)

    assert call(2, s_ls=slice_ - 4) == bole.ERR_INVALID_ARG      # state slices overlap
    assert call(2, s_ls=slice_ + 2) == bole.ERR_INVALID_ARG      # 8-byte layer stride step
    assert call(2, k_ls=N * H * dk + 4) == bole.ERR_INVALID_ARG  # bf16 keys: 8 bytes
    assert call(2, u_ls=-(N * H * dv)) == bole.ERR_INVALID_ARG   # negative stride
    assert call(-1) == bole.ERR_INVALID_ARG
    assert call(65536) == bole.ERR_INVALID_ARG
    assert call(2, S=None) == bole.ERR_INVALID_ARG
    # zero layers: valid, nothing launched
    assert call(0) == bole.OK


def test_commit_verify_host_validation_without_gpu(lib):
    """bole_commit_verify rejects bad arguments and unsupported shapes before
    any launch: the previous round's factors may not be this round's output
    buffers; fp32, other head sizes and trees beyond 64 nodes or depth 15
    are the two-call sequence's (BOLE_ERR_UNSUPPORTED)."""
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake, fake2, fake3 = c(1 << 20), c(2 << 20), c(3 << 20)
    B, H, N, N_prev = 2, 3, 40, 30

    def call(S=fake, U_prev=fake2, U=fake3, logP_prev=fake2, logP=fake3, dtype=1, dk=128,
             dv=128, max_T=32, max_depth=8, flags=0, N=N, N_prev=N_prev, acc=fake):
        return lib.bole_commit_verify(S, fake, U_prev, logP_prev, fake, fake, acc, N_prev,
                                      fake, fake, fake, dtype, fake, fake, fake, fake, B, H, dk,
                                      dv, N, max_T, max_depth, fake, U, logP, fake, flags, None)

    assert call(S=None) == bole.ERR_INVALID_ARG
    assert call(acc=None) == bole.ERR_INVALID_ARG
    assert call(U=fake2) == bole.ERR_INVALID_ARG          # U aliases U_prev
    assert call(logP=fake2) == bole.ERR_INVALID_ARG       # logP aliases logP_prev
    assert call(flags=bole.FLAG_STATE_VK) == bole.ERR_INVALID_ARG
    assert call(N=B * 32 + 1) == bole.ERR_INVALID_ARG     # more nodes than B * max_T
    assert call(S=c((1 << 20) + 8)) == bole.ERR_INVALID_ARG  # 16-byte alignment
    assert call(dtype=0) == bole.ERR_UNSUPPORTED          # fp32 q/k/v
    assert call(dk=64) == bole.ERR_UNSUPPORTED
    assert call(max_T=65) == bole.ERR_UNSUPPORTED
    assert call(max_depth=16) == bole.ERR_UNSUPPORTED
    assert call(N=0, N_prev=0) == bole.OK                 # nothing to commit or verify


def test_state_layout_flag_keeps_the_workspace(lib):
    f = lib.bole_workspace_size
    f.restype = ctypes.c_size_t
    from gated_deltanet_verification_gb300 import bole
    vk = bole.FLAG_STATE_VK
    for args in [(2, 3, 16, 16, 8, 3, 0), (2, 3, 128, 128, 64, 15, 1), (2, 3, 128, 128, 128, 127, 1)]:
        assert f(*args, vk) == f(*args, 0)


def test_stage1_host_validation_without_gpu(lib):
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake = c(1 << 20)
    B, H, dk, dv, N = 2, 3, 128, 128, 8

    def gates(W=4, state=fake, dk=dk, x=fake, N=N, max_T=64):
        return lib.bole_conv_gates(x, state, fake, None, fake, fake, None, None, 1, fake, fake,
                                   B, H, dk, dv, N, max_T, W, fake, fake, fake, fake, fake, fake,
                                   0, None)

    assert gates(W=0) == bole.ERR_INVALID_ARG
    assert gates(W=bole.MAX_CONV_WIDTH + 1) == bole.ERR_INVALID_ARG
    assert gates(state=None) == bole.ERR_INVALID_ARG          # W > 1 needs the state
    assert gates(dk=24) == bole.ERR_INVALID_ARG
    assert gates(x=c((1 << 20) + 8)) == bole.ERR_INVALID_ARG  # 16-byte alignment
    assert gates(N=B * 64 + 1) == bole.ERR_INVALID_ARG        # more nodes than B * max_T
    assert gates(max_T=129) == bole.ERR_INVALID_ARG
    assert gates(max_T=0) == bole.ERR_INVALID_ARG
    assert gates(N=0) == bole.OK                              # nothing to launch

    def commit(W=4, acc=fake, N=N):
        return lib.bole_conv_commit(fake, fake, 1, fake, fake, acc, B, H * 384, W, N, fake, 0,
                                    None)

    assert commit(acc=None) == bole.ERR_INVALID_ARG
    assert commit(W=9) == bole.ERR_INVALID_ARG
    assert commit(W=1, acc=None) == bole.OK                   # no state to commit
    assert commit(N=0) == bole.OK


def test_select_host_validation_without_gpu(lib):
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake = c(1 << 20)
    ws = lib.bole_select_workspace_size
    ws.restype = ctypes.c_size_t
    assert ws(64) == 64 * 128 * 8 + 2 * 64 * 4
    assert ws(bole.SELECT_MAX_REQUESTS + 1) == 0

    def sel(B=4, M=40, budget=16, work=fake, nbytes=1 << 20, offsets=fake):
        return lib.bole_select_forest(fake, fake, fake, None, B, M, budget, offsets, fake, fake,
                                      None, work, nbytes, fake, 0, None)

    assert sel(B=bole.SELECT_MAX_REQUESTS + 1) == bole.ERR_INVALID_ARG
    assert sel(budget=-1) == bole.ERR_INVALID_ARG
    assert sel(offsets=None) == bole.ERR_INVALID_ARG
    assert sel(work=None) == bole.ERR_WORKSPACE
    assert sel(nbytes=16) == bole.ERR_WORKSPACE


def test_stage1_commit_rejects_bad_sizes_without_gpu(lib):
    from gated_deltanet_verification_gb300 import bole
    c = ctypes.c_void_p
    fake = c(1 << 20)
    assert lib.bole_conv_commit(fake, fake, 1, fake, fake, fake, 70000, 384, 4, 8, fake, 0,
                                None) == bole.ERR_INVALID_ARG      # B above the grid limit
    assert lib.bole_conv_commit(fake, fake, 1, fake, fake, fake, 2, 100, 4, 8, fake, 0,
                                None) == bole.ERR_INVALID_ARG      # C not a multiple of 16


def test_binding_constants_match_the_header():
    """Every numeric constant the binding mirrors has the header's value (the
    #defines and the bole_status codes), so the two cannot drift apart."""
    import re
    from gated_deltanet_verification_gb300 import bole
    text = open(os.path.join(os.path.dirname(__file__), "..", "include", "bole.h")).read()
    defines = {}
    for name, val in re.findall(r"#define BOLE_([A-Z_]+)\s+([0-9x()<u l]+)", text):
        defines[name] = eval(val.replace("ull", "").replace("u", "").strip())
    codes = dict((n, int(v)) for n, v in re.findall(r"BOLE_(OK|ERR_[A-Z_]+)\s*=\s*(\d+)", text))
    pairs = {"MAX_TREE_NODES": bole.MAX_TREE_NODES, "STATUS_WORDS": bole.STATUS_WORDS,
             "FLAG_FORCE_SIMT": bole.FLAG_FORCE_SIMT,
             "FLAG_OVERLAP_LAUNCH": bole.FLAG_OVERLAP_LAUNCH,
             "FLAG_STATE_VK": bole.FLAG_STATE_VK,
             "FLAG_ONE_TILE_PER_HEAD": bole.FLAG_ONE_TILE_PER_HEAD,
             "FLAG_VALUE_TILES": bole.FLAG_VALUE_TILES,
             "FLAG_INLINE_TOPOLOGY": bole.FLAG_INLINE_TOPOLOGY,
             "SELFTEST_MAX_WAIT_NS": bole.SELFTEST_MAX_WAIT_NS,
             "NOALLOC_MAX_FACTOR_ELEMS": bole.NOALLOC_MAX_FACTOR_ELEMS,
             "MAX_CANDIDATES": bole.MAX_CANDIDATES,
             "SELECT_MAX_REQUESTS": bole.SELECT_MAX_REQUESTS,
             "MAX_CONV_WIDTH": bole.MAX_CONV_WIDTH}
    for name, value in pairs.items():
        assert defines[name] == value, name
    assert codes and all(getattr(bole, n) == v for n, v in codes.items()), codes
