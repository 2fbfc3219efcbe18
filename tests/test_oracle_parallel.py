"""The oracle's row-block process pool gives the serial oracle's results bit
for bit (it only splits the output rows of the unchanged GEMM functions)."""

import numpy as np

from oracle import gemm, parallel


def layer(M, N, K, seed):
    rng = np.random.default_rng(seed)
    bf = lambda a: (np.asarray(a, np.float32).view(np.uint32) + 0x8000 >> 16 << 16).astype(np.uint32).view(np.float32)
    X = bf(rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, (M, 1))))
    W = bf(rng.standard_normal((N, K)) * 0.02)
    dY = bf(rng.standard_normal((M, N)) * 1e-3)
    return X, W, dY


def test_pool_matches_serial_oracle_bit_for_bit():
    X, W, dY = layer(384, 256, 512, 3)
    try:
        for mode in ("amax448", "pow2"):
            Y1, s1 = gemm.linear_fwd(X, W, scale_mode=mode)
            Y2, s2 = parallel.linear_fwd(X, W, scale_mode=mode)
            assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
            for k in s1:
                assert np.array_equal(np.asarray(s1[k]), np.asarray(s2[k])), k
            dX1, dW1 = gemm.linear_bwd(dY, s1, scale_mode=mode)
            dX2, dW2 = parallel.linear_bwd(dY, s2, scale_mode=mode)
            assert np.array_equal(dX1.view(np.uint32), dX2.view(np.uint32))
            assert np.array_equal(dW1.view(np.uint32), dW2.view(np.uint32))
        acc1, _ = gemm.fprop(*[s1[k] for k in ("Xq", "sX", "Wq", "sW")])
        acc2, _ = parallel.gemm_rows("fprop", *[s1[k] for k in ("Xq", "sX", "Wq", "sW")])
        assert np.array_equal(acc1.view(np.uint32), acc2.view(np.uint32))
        # subsets of rows and columns (the tile samples of the oracle timing plan), split either way
        for rows, cols in ((np.arange(128, 384), np.arange(0, 128)), (np.arange(0, 128), np.arange(0, 256))):
            a1, o1 = gemm.fprop(*[s1[k] for k in ("Xq", "sX", "Wq", "sW")], rows=rows, cols=cols)
            a2, o2 = parallel.gemm_rows("fprop", *[s1[k] for k in ("Xq", "sX", "Wq", "sW")], rows=rows, cols=cols)
            assert np.array_equal(a1.view(np.uint32), a2.view(np.uint32))
            assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    finally:
        parallel.shutdown()
