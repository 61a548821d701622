"""The multi-core CPU comparison program (oracle/parallel_baseline.c, used by bench.py only) must move
exactly what the oracle moves, so that its timing line measures the same work."""
import numpy as np
import pytest

import oracle
import workloads
from oracle import parallel_baseline as pb


@pytest.mark.parametrize("case", ["c1", "skew", "int64_scatter", "e8m0"])
def test_parallel_baseline_matches_oracle(case):
    rng = np.random.default_rng(11)
    if case == "c1":
        p = workloads.config(1)
    elif case == "skew":
        counts = np.ones((4, 4), np.int32)
        counts[-1, -1] = 3000 - 15
        p = workloads.make_problem(rng, A=3000, H=96, N=4, E=4, token_dtype="int8", counts=counts,
                                   scale_layout="f32_a", scale_cols=1, has_topk=False)
    elif case == "int64_scatter":
        p = workloads.make_problem(rng, A=2000, H=64, N=8, E=16, token_dtype="bfloat16",
                                   count_dtype=np.int64, scale_layout="f32_as", scale_cols=4, idx_type=1)
    else:
        p = workloads.make_problem(rng, A=1500, H=256, N=16, E=8, token_dtype="float8_e4m3fn",
                                   scale_layout="e8m0", scale_cols=8)
    ref = oracle.run_problem(p)
    lib = pb.load()
    outs = {"tokens": np.empty(p.A * p.row_bytes, np.uint8),
            "scales": None if p.scales is None else np.empty(p.A * p.scale_row_bytes, np.uint8),
            "idx": np.empty(p.A, np.int32), "etn": np.empty(p.E, p.counts.dtype),
            "topk": None if p.topk is None else np.empty(p.A, np.float32)}
    pb.run(lib, p, outs, threads=4)
    assert np.array_equal(outs["tokens"].reshape(p.A, p.row_bytes), ref["permute_tokens"])
    assert np.array_equal(outs["idx"], ref["permute_token_idx"])
    assert np.array_equal(outs["etn"], ref["expert_token_num"])
    if p.scales is not None:
        assert np.array_equal(outs["scales"].reshape(p.A, p.scale_row_bytes), ref["permute_scales"])
    if p.topk is not None:
        assert np.array_equal(outs["topk"].view(np.uint32), ref["permute_topk_weight"].view(np.uint32))
