"""The bench's work accounting (CPU): the FLOPs behind every TFLOP/s figure
and the bytes behind every HBM fraction, checked against the oracle's own
FLOP count, hand arithmetic on the workload shapes, and the visibility sums
of the layouts."""
import numpy as np
import pytest

import bench
from oracle import qi21_oracle as O
from synthetic import qi21_inputs as S


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
def test_pass_flops_equal_the_oracle_count(name):
    w = S.WORKLOADS[name]
    n = w.n_target
    for vis in (n * n, 123456):
        assert bench.pass_flops(w, n, vis) == O.step_flops(w.dim, w.mlp_hidden, w.layers, n, vis)


def test_bench_workload_totals_by_hand():
    # 32 blocks, dim 4096, mlp 12288, 4096 target rows against a 4114-row
    # prefix: every target row sees 4114 + 4096 keys
    w = S.WORKLOADS["step32_cond4114_n4096"]
    H, I, L, M = 4096, 12288, 32, 4096
    assert (w.dim, w.mlp_hidden, w.layers, w.n_target) == (H, I, L, M)
    vis = M * (4114 + 4096)
    g, a = bench.pass_flops(w, M, vis)
    assert g == 2 * M * (3 * H * H + H * H + 2 * H * I + H * I) * L
    assert a == 4 * H * M * 8210 * L
    assert round(g / 1e12, 2) == 57.17 and round(a / 1e12, 2) == 17.63
    work = bench.class_work(w, M, vis)
    total = sum(work[k][1] for k in ("qkv", "o", "gateup", "down")) * L
    assert total == g
    assert work["attention"][1] * L == a
    # the row kernel: x read in f32, xn written in f16
    assert work["rowop"] == ("byte", M * H * 6.0)


def test_visibility_sum_of_a_prefill_matches_the_layout():
    # prefill rows see a leading run given by the oracle's visibility
    segs = [(O.TEXT, 18, 0), (O.IMAGE, 4, 6), (O.IMAGE, 2, 2)]
    vis = O.prefix_visibility(segs)
    assert len(vis) == 18 + 24
    # text rows are causal, image rows see their whole block
    assert list(vis[:18]) == list(range(1, 19))
    assert np.all(vis[18:] == 18 + 24)
