"""The multi-GPU split of the gated map, on CPU: the partition of rows and
tokens, and two gloo ranks that each run the fp64 oracle on their part and
gather, against the oracle on the whole linear.

Row split (one token): rank r holds rows row_ranges(d_out, 2)[r] of W and M
and all of V_k, computes g, rho and the gate itself, and the y parts are
gathered.  Token split (T > 1): each rank takes a block of tokens.  The
gathered y, gate and rho must equal the unsplit oracle bit for bit (the oracle
computes each row and token independently), and with check_gates the ranks'
gates must agree."""
import os
import socket

import numpy as np
import pytest

from gated_rank_subspace_gsi_gb300 import shard


def test_row_ranges_cover_and_align():
    for d_out in (8, 16, 24, 4096, 4104, 28672):
        for world in (1, 2, 3, 4, 7, 8):
            if world * 8 > d_out:
                with pytest.raises(ValueError):
                    shard.row_ranges(d_out, world)
                continue
            parts = shard.row_ranges(d_out, world)
            assert parts[0][0] == 0 and parts[-1][1] == d_out
            for (a, b), (c, _) in zip(parts, parts[1:]):
                assert b == c
            sizes = [b - a for a, b in parts]
            assert all(s % 8 == 0 and s >= 8 for s in sizes)
            assert max(sizes) - min(sizes) <= 8
    with pytest.raises(ValueError):
        shard.row_ranges(100, 2)


def test_token_ranges_cover():
    for T in (0, 1, 2, 5, 64, 511):
        for world in (1, 2, 3, 8):
            parts = shard.token_ranges(T, world)
            assert parts[0][0] == 0 and parts[-1][1] == T
            assert all(b >= a for a, b in parts)
            assert sum(b - a for a, b in parts) == T
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import gsi_inputs as gi
    spec = gi.LinearSpec("shard", 200, 256, 64, 0.1, 0.05, 0.3)
    inp = gi.make_linear_inputs(spec, 6, 2, seed=123)
    return inp


def _bits(a):
    """bf16 bit patterns (uint16) as a torch int16 tensor: the token rows
    travel through the split as raw bits, untouched."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16))


def _oracle_forward(orc, W, Vb, M, eps):
    """local_forward over rows of W and M on the fp64 oracle."""
    import torch

    def fwd(xb):
        ref = orc.forward_bf16(W, Vb, M, eps, xb.numpy().view(np.uint16))
        return (torch.from_numpy(ref["y"]), torch.from_numpy(ref["gate"].astype(np.uint8)),
                torch.from_numpy(ref["rho"]))
    return fwd


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    try:
        import torch.distributed as dist

        import oracle
        dist.init_process_group("gloo", rank=rank, world_size=world)
        orc = oracle.default()
        inp = _case()
        W, Vb, X, eps = inp.W, inp.basis.V_bits, inp.X_bits, 0.1
        d_out = W.shape[0]
        M = orc.precompute_M_bf16(W, Vb)
        r0, r1 = shard.row_ranges(d_out, world)[rank]
        rows_fwd = _oracle_forward(orc, W[r0:r1], Vb, M[r0:r1], eps)
        rows = []
        for t in range(X.shape[0]):  # one token per call, as the row split is used
            y, g, r = shard.row_sharded_forward(rows_fwd, _bits(X[t:t + 1]), d_out, rank, world,
                                                check_gates=True)
            rows.append((y.numpy(), g.numpy(), r.numpy()))
        tok_fwd = _oracle_forward(orc, W, Vb, M, eps)
        ty, tg, tr = shard.token_sharded_forward(tok_fwd, _bits(X), X.shape[0], rank, world)
        dist.destroy_process_group()
        q.put((rank, rows, (ty.numpy(), tg.numpy(), tr.numpy()), None))
    except Exception:  # reported to the parent, which fails the test
        import traceback
        q.put((rank, None, None, traceback.format_exc()))


def test_split_two_gloo_ranks_reproduce_the_oracle(orc):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(q.get(timeout=240))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    errors = [e for (*_, e) in results if e]
    assert not errors, errors[0]
    inp = _case()
    M = orc.precompute_M_bf16(inp.W, inp.basis.V_bits)
    ref = orc.forward_bf16(inp.W, inp.basis.V_bits, M, 0.1, inp.X_bits)
    assert set(ref["gate"].tolist()) == {0, 1}
    for rank, rows, (ty, tg, tr), _ in results:
        # row split: every rank gathers the whole y of each token
        for t, (y, g, r) in enumerate(rows):
            assert np.array_equal(y[0], ref["y"][t]), (rank, t)
            assert int(g[0]) == int(ref["gate"][t]) and r[0] == ref["rho"][t]
        # token split
        assert np.array_equal(ty, ref["y"]) and np.array_equal(tg, ref["gate"])
        assert np.array_equal(tr, ref["rho"])


def _mismatch_worker(rank: int, world: int, port: int, q):
    """Rank 1 plants a different rho: check_gates must refuse the split."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        import torch
        import torch.distributed as dist
        dist.init_process_group("gloo", rank=rank, world_size=world)

        def fwd(xb):
            rho = torch.tensor([0.25 + 1e-7 * rank], dtype=torch.float64)
            return torch.zeros((1, 8)), torch.zeros((1,), dtype=torch.uint8), rho
        try:
            shard.row_sharded_forward(fwd, None, 16, rank, world, check_gates=True)
            q.put((rank, "no error"))
        except RuntimeError as e:
            q.put((rank, "refused" if "different gate" in str(e) else repr(e)))
        dist.destroy_process_group()
    except Exception:
        import traceback
        q.put((rank, traceback.format_exc()))


def test_split_refuses_ranks_that_disagree():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_mismatch_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(q.get(timeout=120))
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.kill()
    assert sorted(results) == [(0, "refused"), (1, "refused")], results
