"""Row-sharded BitDelta compression across ranks (torch.distributed).

A linear's rows split across ranks need no exchange for the linear itself or
for a per-row alpha: every rank compresses and applies its own rows
(section "Sunum mimarisi" of the BitDelta post: one fused kernel per shard).
A per-matrix alpha (section "Matematiksel temel", eq. (3): the mean |Delta|
over the whole matrix) is the one exchange: each rank compresses its row
block with BD_ALPHA_PER_MATRIX, which gives the mean over its own rows,
alpha_r = sum_r |Delta| / (rows_r * d_in), and the matrix's alpha is
sum_r rows_r * alpha_r / d_out -- one all-reduce of an fp64 scalar.  The sign
bits never depend on alpha, so they need no exchange.

Each alpha_r is already rounded to fp32, so the combined alpha is within a
few fp32 roundings (about 1e-7 relative) of the unsharded one, inside the
1e-6 relative bound alpha is held to.

A rank that holds no rows (d_out < world) adds exactly 0, whatever its
alpha tensor holds (bd_compress writes nothing for zero rows).

Failure: with the gloo backend a rank that never reaches the all-reduce
makes the others' all_reduce raise after the process group's timeout, which
is turned into BD_ERR_TIMEOUT (BitDeltaError).  With NCCL a collective that
times out is normally handled by NCCL's asynchronous watchdog, which aborts
the communicator (and, by default, the process) rather than raising here;
that path is not mapped to BD_ERR_TIMEOUT.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import bitdelta as bd


def row_bounds(d_out: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [r0, r1) of rank `rank` when d_out rows are split in `world`
    contiguous blocks whose sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world or d_out < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, d_out >= 0")
    return d_out * rank // world, d_out * (rank + 1) // world


def alpha_share(alpha_local: torch.Tensor, rows_local: int) -> torch.Tensor:
    """This rank's term of the per-matrix alpha sum: rows_local * alpha_local
    in fp64 (= the rank's sum of |Delta| / d_in), and exactly 0 for a rank
    without rows, whose alpha tensor may hold anything (NaN included)."""
    if alpha_local.numel() != 1 or alpha_local.dtype != torch.float32:
        raise ValueError("alpha_local must be one fp32 element")
    if rows_local < 0:
        raise ValueError("need rows_local >= 0")
    if rows_local == 0:
        return torch.zeros(1, dtype=torch.float64, device=alpha_local.device)
    return alpha_local.reshape(1).double() * float(rows_local)


def combine_alpha(shares: torch.Tensor, d_out: int) -> torch.Tensor:
    """The matrix's alpha (fp32, one element) from the summed shares."""
    if d_out <= 0:
        raise ValueError("need d_out > 0")
    return (shares.reshape(1) / float(d_out)).float()


def per_matrix_alpha_allreduce(alpha_local: torch.Tensor, rows_local: int, d_out: int, group=None) -> torch.Tensor:
    """The matrix's per-matrix alpha from each rank's alpha over its own rows.

    alpha_local: fp32 tensor of one element (this rank's bd_compress output
    in BD_ALPHA_PER_MATRIX mode; ignored when rows_local is 0), on the device
    the group's backend uses (CPU for gloo, CUDA for nccl).  Returns an fp32
    tensor of one element on the same device, equal on every rank.
    """
    if d_out <= 0:
        raise ValueError("need rows_local >= 0 and d_out > 0")
    weighted = alpha_share(alpha_local, rows_local)
    try:
        dist.all_reduce(weighted, op=dist.ReduceOp.SUM, group=group)
    except RuntimeError as e:  # gloo: the collective gave up waiting for a rank
        if "timeout" in str(e).lower() or "timed out" in str(e).lower():
            raise bd.BitDeltaError(bd.BD_ERR_TIMEOUT, "per_matrix_alpha_allreduce") from e
        raise
    return combine_alpha(weighted, d_out)
