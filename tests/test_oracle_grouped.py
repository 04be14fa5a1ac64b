"""The oracle's grouped (MoE) product is the plain W4A16 product applied per
group: one group reproduces the plain product, and empty groups contribute
nothing."""
import numpy as np

import oracle
import synth


def test_grouped_is_the_plain_product_per_group():
    K, N = 256, 96
    Ws = [synth.quant_weight(N=N, K=K, seed=10 + e) for e in range(3)]
    qs = [oracle.quantize(W) for W in Ws]
    x = synth.decode_x(11, K=K)
    offs = [0, 4, 4, 11]  # the middle group is empty
    got = oracle.grouped_logits(x, offs, [q[0] for q in qs], [q[1] for q in qs], [q[2] for q in qs])
    assert np.array_equal(got[:4], oracle.logits(x[:4], *qs[0]))
    assert np.array_equal(got[4:], oracle.logits(x[4:], *qs[2]))
    one = oracle.grouped_logits(x, [0, 11], [qs[1][0]], [qs[1][1]], [qs[1][2]])
    assert np.array_equal(one, oracle.logits(x, *qs[1]))
