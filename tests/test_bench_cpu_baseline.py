"""CPU: the bench's oracle baseline pieces -- the host CPU name and the
row-sharded oracle pass over every core (the same arithmetic as the
single-thread pass: row_begin keeps each shard's noise counters)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle as orc  # noqa: E402
from semi_structured_sparsity_gb300 import workloads as W  # noqa: E402


def test_cpu_model_names_the_host():
    name = bench.cpu_model()
    assert isinstance(name, str) and name


def test_sharded_pass_runs_and_shards_reproduce_the_whole():
    wl = W.WORKLOADS["llama2_7b_block"]
    sample = bench.oracle_sample_step(wl, 6)
    bench.oracle_step_sharded(wl, sample, 0, 4)   # every matrix in 4 row shards
    Wb, L, _, tid = sample[4]
    whole = orc.forward(Wb, L, wl.tau, wl.kappa, 0, 0, tid)[0]
    parts = [orc.forward(Wb[a:b], L[a:b], wl.tau, wl.kappa, 0, 0, tid, row_begin=a)[0]
             for a, b in ((0, 2), (2, 5), (5, 6))]
    assert np.array_equal(np.concatenate(parts), whole)


def test_source_digest_follows_code_not_comments():
    """A stored DRAM-traffic figure stays valid while only comments or
    whitespace of the stream-kernel sources change, and no longer once the
    code does."""
    a = "int f(int x) {  // the count\n  return x + 1; /* one\n more */ }\n"
    b = "int f(int x) {\n\n  return x + 1;   }  // comments differ\n"
    c = "int f(int x) { return x + 2; }\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert len(bench.kernel_source_digest()) == 12


def test_traffic_table_reads_the_committed_summary():
    tt = bench.traffic_table()
    for k in bench.KERNELS:
        bytes_, digest = tt[(k, "llama2_7b_block")]
        # DRAM bytes of one launch within 5% of the algorithmic bytes
        alg = bench.BYTES_PER_WEIGHT[k] * W.WORKLOADS["llama2_7b_block"].weights
        assert 0.95 * alg <= bytes_ <= 1.01 * alg
        assert len(digest) == 12
