"""The gated map split across GPUs, one process per GPU.

The page "Technical summary: Gated Subspace Inference for transformer
acceleration" sets GSI beside methods that shorten the token axis, because
GSI works on the hidden axis (section 3).  The map splits two ways:

- Rows (one token, T = 1): rank r holds rows [r0, r1) of W and of
  M = W V_k, and all of V_k.  Every rank computes g = V_k^T x, rho and the
  gate itself; the library's one-token kernel reduces g exactly (fixed-point
  integers), so ranks with the same x, V_k and SM count take the same gate,
  bit for bit, and need no collective to agree.  The ranks' rows of y are then
  gathered.
- Tokens (T > 1): every rank holds the whole linear and takes a contiguous
  block of the T tokens; the blocks of y are gathered.  Tokens are
  independent, so no collective touches the computation itself.

The functions here are the partition and the gather only.  The computation
of a rank's part is a callable ``local_forward(x) -> (y, gate, rho)`` (on
a GPU, the rank's GatedLinear; the tests pass other implementations), and
the gather is torch.distributed's all_gather on the given process group
(NCCL between GPUs).
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

ROW_ALIGN = 8  # rows per unit: the library needs d_out % 8 == 0 for every part


def row_ranges(d_out: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous row blocks [r0, r1) of d_out rows for `world` ranks, in
    units of 8 rows, as equal as the units allow (earlier ranks never get
    fewer rows than later ones)."""
    if d_out % ROW_ALIGN != 0:
        raise ValueError("d_out must be a multiple of 8")
    if world < 1 or world * ROW_ALIGN > d_out:
        raise ValueError("every rank needs at least 8 rows")
    units = d_out // ROW_ALIGN
    out = []
    for r in range(world):
        u0 = (r * units) // world
        u1 = ((r + 1) * units) // world
        out.append((u0 * ROW_ALIGN, u1 * ROW_ALIGN))
    return out


def token_ranges(T: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous token blocks [t0, t1) of T tokens for `world` ranks (a
    rank may get none when T < world)."""
    if world < 1 or T < 0:
        raise ValueError("world >= 1 and T >= 0")
    return [((r * T) // world, ((r + 1) * T) // world) for r in range(world)]


def _gather_padded(part, parts: Sequence[Tuple[int, int]], dim: int, group=None):
    """All-gather `part` (this rank's block along `dim`, blocks of sizes given
    by `parts`) into the full tensor: blocks are padded to the largest size for
    the collective, then cut and concatenated in rank order."""
    import torch
    import torch.distributed as dist
    sizes = [b - a for (a, b) in parts]
    width = max(sizes)
    shape = list(part.shape)
    pad = list(shape)
    pad[dim] = width
    buf = torch.zeros(pad, dtype=part.dtype, device=part.device)
    buf.narrow(dim, 0, shape[dim]).copy_(part)
    bufs = [torch.empty_like(buf) for _ in parts]
    dist.all_gather(bufs, buf, group=group)
    return torch.cat([b.narrow(dim, 0, n) for b, n in zip(bufs, sizes)], dim=dim)


def row_sharded_forward(local_forward: Callable, x, d_out: int, rank: int, world: int,
                        group=None, check_gates: bool = False):
    """One call of the row-split map: this rank's rows, then the gather.

    local_forward(x) -> (y_part, gate, rho) computes rows row_ranges(d_out,
    world)[rank] of y (T x rows) for the tokens x, with gate and rho (T,).
    Returns (y, gate, rho) with y = T x d_out.  With check_gates, the ranks'
    gates and rho are gathered too and must agree bit for bit (they do when
    every rank reduces g the same way); a disagreement raises."""
    import torch
    import torch.distributed as dist
    parts = row_ranges(d_out, world)
    y_part, gate, rho = local_forward(x)
    if y_part.dim() == 1:
        y_part = y_part.unsqueeze(0)
    y = _gather_padded(y_part, parts, dim=1, group=group) if world > 1 else y_part
    if check_gates and world > 1:
        g_all = [torch.empty_like(gate) for _ in range(world)]
        r_all = [torch.empty_like(rho) for _ in range(world)]
        dist.all_gather(g_all, gate, group=group)
        dist.all_gather(r_all, rho, group=group)
        for r in range(world):
            if not torch.equal(g_all[r], gate) or not torch.equal(
                    r_all[r].view(torch.uint8), rho.view(torch.uint8)):
                raise RuntimeError(f"rank {r} took a different gate or rho than rank {rank}")
    return y, gate, rho


def token_sharded_forward(local_forward: Callable, x, T: int, rank: int, world: int,
                          group=None):
    """One call of the token-split map: this rank's block of tokens, then the
    gather.  x is the full T x d input; local_forward(x_block) -> (y_block,
    gate_block, rho_block) for the rows token_ranges(T, world)[rank] of x.
    Returns the full (y, gate, rho) in token order."""
    parts = token_ranges(T, world)
    t0, t1 = parts[rank]
    y_b, g_b, r_b = local_forward(x[t0:t1])
    if world == 1:
        return y_b, g_b, r_b
    return (_gather_padded(y_b, parts, dim=0, group=group),
            _gather_padded(g_b, parts, dim=0, group=group),
            _gather_padded(r_b, parts, dim=0, group=group))


class RowShard:
    """This rank's part of a row-split gated linear on the GPU: a libgsi
    handle on rows [r0, r1) of W and M (views, no copy) with the full V_k."""

    def __init__(self, W, V_k, M, eps: float, rank: int, world: int):
        from . import lib
        self.d_out = W.shape[0]
        self.r0, self.r1 = row_ranges(self.d_out, world)[rank]
        self.rank, self.world = rank, world
        self.lin = lib.GatedLinear(W[self.r0:self.r1], V_k, M[self.r0:self.r1], eps)

    def local_forward(self, x, stream=None):
        import torch
        T = x.shape[0]
        y = torch.empty((T, self.r1 - self.r0), dtype=torch.float32, device=x.device)
        gate = torch.empty((T,), dtype=torch.uint8, device=x.device)
        rho = torch.empty((T,), dtype=torch.float32, device=x.device)
        self.lin.forward(x, y, gate, rho, stream)
        return y, gate, rho

    def forward(self, x, group=None, stream=None, check_gates: bool = False):
        return row_sharded_forward(lambda xx: self.local_forward(xx, stream), x, self.d_out,
                                   self.rank, self.world, group, check_gates)

    def close(self):
        self.lin.close()


class TokenShard:
    """This rank's part of a token-split gated linear on the GPU: the whole
    linear (a libgsi handle), applied to this rank's block of the tokens."""

    def __init__(self, W, V_k, M, eps: float, rank: int, world: int, max_T: Optional[int] = None):
        from . import lib
        self.rank, self.world = rank, world
        self.d_out = W.shape[0]
        self.lin = lib.GatedLinear(W, V_k, M, eps, max_T=max_T or 0)

    def local_forward(self, x, stream=None):
        import torch
        T = x.shape[0]
        y = torch.empty((T, self.d_out), dtype=torch.float32, device=x.device)
        gate = torch.empty((T,), dtype=torch.uint8, device=x.device)
        rho = torch.empty((T,), dtype=torch.float32, device=x.device)
        if T > 0:
            self.lin.forward(x, y, gate, rho, stream)
        return y, gate, rho

    def forward(self, x, group=None, stream=None):
        return token_sharded_forward(lambda xx: self.local_forward(xx, stream), x, x.shape[0],
                                     self.rank, self.world, group)

    def close(self):
        self.lin.close()
