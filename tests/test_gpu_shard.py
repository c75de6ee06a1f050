"""The multi-GPU split of the gated map, on one GPU: the parts that ranks
would compute, computed here one after another, against the whole linear.

Row split (T = 1): handles on rows [r0, r1) of W and M with the full V_k give
exactly the full handle's rows of y, and the same gate and rho, bit for bit
(the one-token kernel reduces g as exact integers, so every part takes the
same g; the split is 3 unequal parts).  Tokens include some close to eps, whose
gate the kernel takes from its gate CTA.  Token split (T > 1): the batched
path on blocks of tokens gives exactly the rows of the whole batch."""
import numpy as np
import pytest

import gsi_inputs as gi
from gsi_testlib import GpuLinear, check_against_oracle, to_dev

pytestmark = pytest.mark.gpu


def _tokens(basis, eps, seed):
    rng = np.random.default_rng(seed)
    rs = np.concatenate([np.full(5, 0.05), np.full(3, 0.3),
                         eps + rng.uniform(-3e-3, 3e-3, size=6)])
    return gi.tokens(basis, rs, seed)


def test_row_parts_reproduce_the_whole_linear(gsi, orc):
    import torch
    from gated_rank_subspace_gsi_gb300 import shard
    d_out, d, k, eps = 4096, 4096, 256, 0.1
    W = gi.gaussian_weights(d_out, d, 301)
    basis = gi.random_basis(d, k, 301)
    X = _tokens(basis, eps, 301)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(X, one_by_one=True)
    check_against_oracle(orc, lin, X, y, g, r, what="whole linear")
    assert 0 < g.sum() < len(X)
    parts = [shard.RowShard(lin.W_dev, lin.V_dev, lin.M_dev, eps, rank, 3) for rank in range(3)]
    x = to_dev(X)
    for t in range(len(X)):
        for p in parts:
            yp, gp, rp = p.local_forward(x[t:t + 1])
            torch.cuda.synchronize()
            assert np.array_equal(yp.cpu().numpy()[0], y[t, p.r0:p.r1]), (t, p.rank)
            assert int(gp.item()) == int(g[t]), (t, p.rank)
            assert np.float32(rp.item()).view(np.int32) == np.float32(r[t]).view(np.int32)
    for p in parts:
        assert gsi.gsi_device_status(p.lin.h) == 0
        p.close()
    lin.close()


@pytest.mark.parametrize("k", [128, 256])
def test_token_blocks_reproduce_the_whole_batch(gsi, orc, k):
    from gated_rank_subspace_gsi_gb300 import shard
    d_out, d, eps, T = 2048, 4096, 0.1, 96
    W = gi.gaussian_weights(d_out, d, 302 + k)
    basis = gi.random_basis(d, k, 302 + k)
    rs = np.where(np.arange(T) % 3 == 0, 0.3, 0.05)
    X = gi.tokens(basis, rs, 302 + k)
    lin = GpuLinear(gsi, orc, W, basis.V_bits, eps)
    y, g, r = lin.forward(X)
    check_against_oracle(orc, lin, X, y, g, r, what="whole batch")
    for (t0, t1) in shard.token_ranges(T, 3):
        yb, gb, rb = lin.forward(X[t0:t1])
        assert np.array_equal(yb, y[t0:t1]), (t0, t1)
        assert np.array_equal(gb, g[t0:t1]) and np.array_equal(rb.view(np.int32),
                                                                r[t0:t1].view(np.int32))
    lin.close()
