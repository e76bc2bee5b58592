"""Device-resident copies of a packed forest and one verify + commit round
through the C ABI (the call sequence a serving loop makes each round)."""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import bole


@dataclasses.dataclass
class DeviceBatch:
    B: int
    H: int
    dk: int
    dv: int
    N: int
    max_T: int
    max_depth: int
    offsets: torch.Tensor
    parent: torch.Tensor
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    gamma: torch.Tensor
    beta: torch.Tensor
    S: torch.Tensor          # state slots: S_pre before commit, S_new after
    accepted: torch.Tensor


def to_device(batch, device="cuda", dtype: Optional[torch.dtype] = None) -> DeviceBatch:
    """Copy a TreeBatch (numpy) to the device; q/k/v in the batch's dtype."""
    if dtype is None:
        dtype = torch.bfloat16 if batch.dtype == "bf16" else torch.float32

    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dt)

    return DeviceBatch(
        batch.B, batch.H, batch.dk, batch.dv, batch.N, max(batch.max_T, 1), batch.max_depth,
        t(batch.offsets, torch.int32), t(batch.parent, torch.int32), t(batch.q, dtype),
        t(batch.k, dtype), t(batch.v, dtype), t(batch.gamma, torch.float32),
        t(batch.beta, torch.float32), t(batch.S_pre, torch.float32),
        t(batch.accepted, torch.int32))


@dataclasses.dataclass
class RoundBuffers:
    depth: torch.Tensor
    anc: torch.Tensor
    req_depth: torch.Tensor
    status: torch.Tensor
    O: torch.Tensor
    U: torch.Tensor
    logP: torch.Tensor
    workspace: torch.Tensor
    # the other round's U and logP for bole_commit_verify (alloc_alt)
    U_alt: Optional[torch.Tensor] = None
    logP_alt: Optional[torch.Tensor] = None


def alloc_round(db: DeviceBatch, flags: int = 0) -> RoundBuffers:
    dev = db.q.device
    ws = bole.workspace_size(db.B, db.H, db.dk, db.dv, db.max_T, db.max_depth, db.q.dtype, flags)
    return RoundBuffers(
        depth=torch.empty(db.N, dtype=torch.int32, device=dev),
        anc=torch.empty((db.N, 4), dtype=torch.int32, device=dev),
        req_depth=torch.empty(max(db.B, 1), dtype=torch.int32, device=dev),
        status=bole.new_status(dev),
        O=torch.empty((db.N, db.H, db.dv), dtype=db.q.dtype, device=dev),
        U=torch.empty((db.N, db.H, db.dv), dtype=torch.float32, device=dev),
        logP=torch.empty((db.N, db.H), dtype=torch.float32, device=dev),
        workspace=torch.empty(max(ws, 16), dtype=torch.uint8, device=dev),
    )


def pack(db: DeviceBatch, rb: RoundBuffers, stream=None) -> None:
    bole.pack_forest(db.offsets, db.parent, db.max_depth, depth=rb.depth, anc=rb.anc,
                     req_depth=rb.req_depth[:db.B], status=rb.status, stream=stream)


def verify(db: DeviceBatch, rb: RoundBuffers, flags: int = 0, stream=None) -> None:
    bole.tree_verify(db.S, db.q, db.k, db.v, db.gamma, db.beta, db.offsets, db.parent, rb.depth,
                     rb.anc, rb.req_depth[:db.B], db.max_T, db.max_depth, O=rb.O, U=rb.U,
                     logP=rb.logP, workspace=rb.workspace, status=rb.status, flags=flags,
                     stream=stream)


def commit(db: DeviceBatch, rb: RoundBuffers, flags: int = 0, stream=None) -> None:
    bole.commit(db.S, db.k, rb.U, rb.logP, db.offsets, db.parent, db.accepted,
                status=rb.status, flags=flags, stream=stream)


def inline_topology_supported(db: DeviceBatch, flags: int = 0) -> bool:
    """Whether the verification can form the round's topology itself
    (bole.FLAG_INLINE_TOPOLOGY): the tensor-core kernels for dk = dv = 128,
    depth <= 15 and the default state layout -- bf16 trees of up to 64 nodes,
    fp32 trees of up to 32 (the value-tiled kernel)."""
    if (db.dk != 128 or db.dv != 128 or db.max_depth > 15
            or flags & (bole.FLAG_FORCE_SIMT | bole.FLAG_STATE_VK)):
        return False
    if db.q.dtype == torch.bfloat16:
        return db.max_T <= 64
    return (db.q.dtype == torch.float32 and db.max_T <= 32
            and not flags & bole.FLAG_ONE_TILE_PER_HEAD)


def commit_verify_supported(db: DeviceBatch, flags: int = 0) -> bool:
    """Whether bole_commit_verify applies: bf16 q/k/v, dk = dv = 128, trees of
    up to 64 nodes of depth <= 15, the default state layout."""
    return (db.dk == 128 and db.dv == 128 and db.max_T <= 64 and db.max_depth <= 15
            and db.q.dtype == torch.bfloat16
            and not flags & (bole.FLAG_FORCE_SIMT | bole.FLAG_STATE_VK))


def alloc_alt(db: DeviceBatch, rb: RoundBuffers) -> RoundBuffers:
    """A second U / logP pair, so that consecutive bole_commit_verify rounds
    alternate between them (a round's outputs may not overwrite the factors
    it commits)."""
    rb.U_alt = torch.empty_like(rb.U)
    rb.logP_alt = torch.empty_like(rb.logP)
    return rb


def commit_verify_round(db: DeviceBatch, rb: RoundBuffers, parity: int, stream=None) -> None:
    """One round of a repeated workload with the previous round's commit
    fused into this round's verification (bole_commit_verify): the same
    forest and inputs every round, parity 0 committing the factors in
    (U, logP) and writing this round's into (U_alt, logP_alt), parity 1 the
    other way round.  The first round of a sequence is a plain verification
    (verify with FLAG_INLINE_TOPOLOGY into U, logP)."""
    Up, Lp, Uo, Lo = ((rb.U, rb.logP, rb.U_alt, rb.logP_alt) if parity == 0
                      else (rb.U_alt, rb.logP_alt, rb.U, rb.logP))
    bole.commit_verify(db.S, db.k, Up, Lp, db.offsets, db.parent, db.accepted, db.q, db.k, db.v,
                       db.gamma, db.beta, db.offsets, db.parent, db.max_T, db.max_depth, O=rb.O,
                       U=Uo, logP=Lo, status=rb.status, stream=stream)


def run_round(db: DeviceBatch, rb: RoundBuffers, flags: int = 0, stream=None) -> None:
    """One round, asynchronous on one stream.  With bole.FLAG_INLINE_TOPOLOGY
    in `flags`: verify (which forms the topology itself) -> commit, the status
    block left as the previous round left it (sticky: zeroed once by the
    caller).  Otherwise pack -> verify -> commit, pack clearing the status
    block.  Each call directly follows the one it depends on, so verify and
    commit may overlap their predecessor's tail (bole.FLAG_OVERLAP_LAUNCH)."""
    if not flags & bole.FLAG_INLINE_TOPOLOGY:
        pack(db, rb, stream)
    verify(db, rb, flags | bole.FLAG_OVERLAP_LAUNCH, stream)
    commit(db, rb, (flags & ~bole.FLAG_INLINE_TOPOLOGY) | bole.FLAG_OVERLAP_LAUNCH, stream)
