"""bench.py's host-side bookkeeping, without a GPU: the kernel-launch counts
it reports as gpu_launches, pinned to the launch lists ncu recorded for the
same steps (30 kernels per forward step and 49 per backward step of the
DeepSeek-V3-shaped layer, whose Zipf routing overflows into 4 chunks)."""
import bench


def chunks(n, T=8192):
    c = T // n
    return [(i * c, (i + 1) * c, False) for i in range(n)]


def test_forward_launches():
    # route + check, then per chunk: block counts, expert scan, assign,
    # scatter, GEMM1, GEMM2, combine
    assert bench.launches_per_step(chunks(4), "fallback") == 30
    assert bench.launches_per_step([(0, 8192, True)], "fallback") == 9
    assert bench.launches_per_step([(0, 8192, False)], "dropless") == 8
    # the routing/permute sweep: no expert FFN
    assert bench.launches_per_step(chunks(8), "fallback",
                                   dispatch_only=True) == 2 + 8 * 5
    # the duplication plan adds one launch
    assert bench.launches_per_step([(0, 8192, True)], "fallback",
                                   planned=1) == 10
    # an empty pass launches nothing
    assert bench.launches_per_step([(0, 0, False)], "fallback") == 2


def test_backward_launches():
    # route + check; per chunk 4 permute kernels, GEMM1 keeping g/u, GEMM2,
    # combine backward, two dgrad GEMMs, permute backward; route backward;
    # regrouping (2); the two weight-gradient GEMMs; two zero fills
    assert bench.backward_launches(chunks(4), "fallback", True) == 49
    # without regrouping the segments go in batches of 16 passes
    assert bench.backward_launches(chunks(20), "fallback", False) == \
        2 + 20 * 10 + 1 + 2 * 2 + 2
    # with duplicate slots (one capped pass over the plan's groups): the
    # plan adds a launch; the zero fills stay (ncu saw two per step there)
    assert bench.backward_launches([(0, 8192, True)], "fallback", True,
                                   planned=True) == 3 + 10 + 1 + 2 + 2 + 2
