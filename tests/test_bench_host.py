"""bench.py's host-side bookkeeping, without a GPU: the kernel-launch counts
it reports as gpu_launches, pinned to the launch lists ncu recorded for the
same steps (31 kernels per forward step -- the router GEMM and 30 -- and
49 per backward step of the DeepSeek-V3-shaped layer, whose Zipf routing
overflows into 4 chunks of 2048 tokens; 8 shards)."""
import bench


def chunks(n, T=8192):
    c = T // n
    return [(i * c, (i + 1) * c, False) for i in range(n)]


def test_table_launches():
    # block counts, expert scan, assign; the dedup scan only above 1024
    # block x shard counts
    assert bench.table_launches(2048, 8) == 3      # 16 blocks x 8 shards
    assert bench.table_launches(8192, 16) == 3     # 64 x 16 = 1024
    assert bench.table_launches(8193, 16) == 4
    assert bench.table_launches(65536, 8) == 4     # 512 x 8
    assert bench.table_launches(0, 8) == 1         # the expert scan alone


def test_forward_launches():
    # router + route + check, then per chunk: 3 table kernels, scatter,
    # GEMM1, GEMM2, combine
    assert bench.launches_per_step(chunks(4), "fallback", shards=8) == 31
    # no overflow: the capped pass (Llama4-Maverick: 16 shards, 64 blocks)
    assert bench.launches_per_step([(0, 8192, True)], "fallback",
                                   shards=16) == 3 + 7
    assert bench.launches_per_step([(0, 8192, False)], "dropless",
                                   shards=8) == 9
    # the routing/permute sweep: no expert FFN; 64K tokens in one capped
    # pass take the dedup scan kernel
    assert bench.launches_per_step(chunks(8, 65536), "fallback",
                                   dispatch_only=True, shards=8) == 3 + 8 * 5
    assert bench.launches_per_step([(0, 65536, True)], "capped",
                                   dispatch_only=True, shards=8) == 2 + 6
    # the duplication plan adds one launch
    assert bench.launches_per_step([(0, 8192, True)], "fallback", planned=1,
                                   shards=8) == 4 + 7


def test_backward_launches():
    # route + check; per chunk 3 table kernels, scatter, GEMM1 keeping g/u,
    # GEMM2, combine backward, two dgrad GEMMs, permute backward; route
    # backward; regrouping (2); two weight-gradient GEMMs; two zero fills
    assert bench.backward_launches(chunks(4), "fallback", True,
                                   shards=8) == 49
    # without regrouping the segments go in batches of 16 passes
    assert bench.backward_launches(chunks(20, 20480), "fallback", False,
                                   shards=8) == \
        2 + 20 * 10 + 1 + 2 * 2 + 2
    # duplicate slots, one capped pass over the plan's groups: the plan
    # adds a launch; the zero fills stay (ncu saw two per step there)
    assert bench.backward_launches([(0, 8192, True)], "fallback", True,
                                   planned=True, shards=8) == \
        3 + 10 + 1 + 2 + 2 + 2


def test_traced_graph_launches():
    # DeepSeek-V3 layer, 4 chunks of 2048 tokens: router, route, check,
    # branch select, 23 stamps; side branches: the capped pass's tables (64
    # blocks x 8 shards: 3 kernels) and chunk 0's (3); per chunk scatter,
    # GEMM1, GEMM2, combine; chunks 1-3 their tables (3 each)
    assert bench.graph_launches(chunks(4), 8192, 8, 0, 2048, 4) == \
        1 + 3 + 23 + 3 + 3 + 16 + 9
    # Llama4-Maverick, no overflow: the capped pass only (its tables and
    # chunk 0's of the 8-chunk fallback ran before the branch)
    assert bench.graph_launches([(0, 8192, True)], 8192, 16, 0, 1024, 8) == \
        1 + 3 + 8 + 3 + 3 + 4
    # with a duplication plan the capped pass computes its own tables
    assert bench.graph_launches([(0, 8192, True)], 8192, 8, 1, 2048, 4) == \
        1 + 3 + 1 + 8 + 3 + 4 + 3
