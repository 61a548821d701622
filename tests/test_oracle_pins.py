"""Pins for the CPU oracle, checked against facts that do not come from the oracle itself.

* hand-worked examples (tests/golden/hand_examples.json), derived by hand from the
  MoeReRoutingV2 article, section 计算公式;
* brute force: the expert-major order is a stable sort of the source rows by
  (expert, rank) -- checked exhaustively on every count matrix with N, E <= 3 and counts 1..3;
* a closed form: for the all-ones N x E matrix the gather index is the transpose of the
  N x E index grid (numpy transpose);
* identities: N = 1 or E = 1 leaves the rows in place (the GEIR sample's A=11, H=79, N=11,
  E=1 shape among them);
* invariants on seeded random problems: idx is a permutation, gather and scatter are
  inverse, permute_tokens == tokens[gather] (numpy fancy indexing), expert_token_num equals
  numpy's column sums, each (rank, expert) segment lands contiguously;
* validation: counts <= 0 and Sum(counts) != A are rejected and nothing is written;
* planted mistakes: mutated copies of the oracle source (a transposed walk, an inclusive
  prefix, a swapped index, row sums for column sums) must each fail one of these pins.
"""
import ctypes
import itertools
import json
import os
import re
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


# ----------------------------------------------------------------------------- independent references

def brute_force_gather(counts: np.ndarray) -> np.ndarray:
    """Label each source row with its (rank, expert) by walking the rank-major layout, then
    stable-sort the rows by (expert, rank)."""
    N, E = counts.shape
    labels = []
    for i in range(N):
        for j in range(E):
            labels += [(j, i)] * int(counts[i, j])
    return np.array(sorted(range(len(labels)), key=lambda s: labels[s]), dtype=np.int32)


def inverse(perm: np.ndarray) -> np.ndarray:
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm), dtype=perm.dtype)
    return inv


def row_payload(A: int, rb: int) -> np.ndarray:
    """Byte rows that encode their own row number (so a moved row is identifiable)."""
    s = np.arange(A, dtype=np.int64)
    cols = np.arange(rb, dtype=np.int64)
    return ((s[:, None] * 131 + cols[None, :] * 7 + (s[:, None] >> 8)) & 0xFF).astype(np.uint8)


# ----------------------------------------------------------------------------- pin checks (lib-parametrised)

def check_hand_examples(lib):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        for dt in (np.int32, np.int64):
            c = np.array(case["counts"], dtype=dt)
            A = case["A"]
            src, dst = oracle.offsets(c, lib=lib)
            assert src.tolist() == case["src_offset"], case["name"]
            assert dst.tolist() == case["dst_offset"], case["name"]
            tok = row_payload(A, 5)
            g = oracle.run(tok, c, idx_type=0, lib=lib)
            s = oracle.run(tok, c, idx_type=1, lib=lib)
            assert g["permute_token_idx"].tolist() == case["gather"], case["name"]
            assert s["permute_token_idx"].tolist() == case["scatter"], case["name"]
            assert g["expert_token_num"].tolist() == case["expert_token_num"], case["name"]
            assert g["expert_token_num"].dtype == dt
            assert np.array_equal(g["permute_tokens"], tok[np.array(case["gather"])])


def check_brute_force(lib, max_dim=3, max_count=3):
    for N in range(1, max_dim + 1):
        for E in range(1, max_dim + 1):
            for flat in itertools.product(range(1, max_count + 1), repeat=N * E):
                c = np.array(flat, dtype=np.int32).reshape(N, E)
                A = int(c.sum())
                tok = row_payload(A, 3)
                w = np.arange(A, dtype=np.float32) * 0.5
                out = oracle.run(tok, c, topk=w, idx_type=0, lib=lib)
                ref = brute_force_gather(c)
                assert np.array_equal(out["permute_token_idx"], ref), c
                assert np.array_equal(out["permute_tokens"], tok[ref]), c
                assert np.array_equal(out["permute_topk_weight"], w[ref]), c
                sc = oracle.run(tok, c, idx_type=1, lib=lib)["permute_token_idx"]
                assert np.array_equal(sc, inverse(ref)), c


def check_transpose_closed_form(lib):
    for N, E in [(1, 1), (2, 3), (3, 2), (16, 16), (5, 7), (64, 3)]:
        c = np.ones((N, E), np.int32)
        out = oracle.run(row_payload(N * E, 4), c, idx_type=0, lib=lib)
        expect = np.arange(N * E, dtype=np.int32).reshape(N, E).T.ravel()
        assert np.array_equal(out["permute_token_idx"], expect), (N, E)


def check_identity(lib):
    rng = np.random.default_rng(7)
    for N, E, A, rb in [(11, 1, 11, 158), (1, 9, 40, 33), (1, 1, 5, 16), (4, 1, 50, 3)]:
        c = workloads.counts_uniform(rng, N, E, A)
        tok = rng.integers(0, 256, size=(A, rb), dtype=np.uint16).astype(np.uint8)
        for it in (0, 1):
            out = oracle.run(tok, c, idx_type=it, lib=lib)
            assert np.array_equal(out["permute_token_idx"], np.arange(A, dtype=np.int32))
            assert np.array_equal(out["permute_tokens"], tok)


def check_invariants(lib, problem):
    p = problem
    g = oracle.run(p.tokens, p.counts, scales=p.scales, topk=p.topk, idx_type=0, lib=lib)
    s = oracle.run(p.tokens, p.counts, scales=p.scales, topk=p.topk, idx_type=1, lib=lib)
    gather, scatter = g["permute_token_idx"], s["permute_token_idx"]
    A = p.A
    assert np.array_equal(np.sort(gather), np.arange(A, dtype=np.int32))
    assert np.array_equal(gather[scatter], np.arange(A, dtype=np.int32))
    assert np.array_equal(scatter[gather], np.arange(A, dtype=np.int32))
    assert np.array_equal(g["permute_tokens"], p.tokens[gather])
    assert np.array_equal(s["permute_tokens"], g["permute_tokens"])
    if p.scales is not None:
        assert np.array_equal(g["permute_scales"], p.scales[gather])
    if p.topk is not None:
        assert np.array_equal(g["permute_topk_weight"].view(np.uint32), p.topk[gather].view(np.uint32))
    assert np.array_equal(g["expert_token_num"], p.counts.sum(axis=0).astype(p.counts.dtype))
    assert int(g["expert_token_num"].sum()) == A
    # each (rank, expert) segment of the source lands as one contiguous run, ranks ascending
    N, E = p.counts.shape
    starts = np.concatenate([[0], np.cumsum(p.counts.ravel())])  # row-major segment starts
    seg_of_src = np.repeat(np.arange(N * E), p.counts.ravel())
    seg_at_dst = seg_of_src[gather]
    order = [i * E + j for j in range(E) for i in range(N)]     # expert-major visiting order
    runs = [k for k, _ in itertools.groupby(seg_at_dst.tolist())]
    assert runs == order
    for q in range(N * E):
        pos = np.nonzero(seg_at_dst == q)[0]
        assert np.array_equal(gather[pos], np.arange(starts[q], starts[q + 1]))


def check_unroute_hand_examples(lib):
    """Inverse move: rank-major row s takes expert-major row scatter[s] (hand-derived scatter)."""
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        c = np.array(case["counts"], dtype=np.int32)
        y = row_payload(case["A"], 6)                      # an expert-major buffer
        out = oracle.unroute(y, c, permute_topk=np.arange(case["A"], dtype=np.float32), lib=lib)
        sc = np.array(case["scatter"])
        assert np.array_equal(out["tokens"], y[sc]), case["name"]
        assert np.array_equal(out["topk_weight"], sc.astype(np.float32)), case["name"]


def check_unroute_brute_force(lib, max_dim=3, max_count=2):
    for N in range(1, max_dim + 1):
        for E in range(1, max_dim + 1):
            for flat in itertools.product(range(1, max_count + 1), repeat=N * E):
                c = np.array(flat, dtype=np.int64).reshape(N, E)
                A = int(c.sum())
                y = row_payload(A, 3)
                sc = inverse(brute_force_gather(c))
                out = oracle.unroute(y, c, permute_scales=y[:, :2], lib=lib)
                assert np.array_equal(out["tokens"], y[sc]), c
                assert np.array_equal(out["scales"], y[sc][:, :2]), c


# ----------------------------------------------------------------------------- tests on the real oracle

def test_hand_examples(oracle_lib):
    check_hand_examples(oracle_lib)


def test_brute_force_exhaustive(oracle_lib):
    check_brute_force(oracle_lib)


def test_transpose_closed_form(oracle_lib):
    check_transpose_closed_form(oracle_lib)


def test_identity_cases(oracle_lib):
    check_identity(oracle_lib)


@pytest.mark.parametrize("seed,N,E,A,dtype,layout,cols", [
    (1, 4, 4, 64, "bfloat16", "f32_a", 1),
    (2, 8, 32, 700, "int8", "f32_as", 4),
    (3, 32, 8, 900, "float8_e4m3fn", "e8m0", 8),
    (4, 23, 2, 52, "float16", "none", 0),
    (5, 14, 1, 35, "float4_e2m1", "f32_a", 1),
    (6, 64, 64, 5000, "float16", "f32_a", 1),
])
def test_invariants_random(oracle_lib, seed, N, E, A, dtype, layout, cols):
    rng = np.random.default_rng(seed)
    p = workloads.make_problem(rng, A=A, H=22, N=N, E=E, token_dtype=dtype,
                               count_dtype=np.int64 if seed % 2 else np.int32,
                               scale_layout=layout, scale_cols=cols, has_topk=True)
    check_invariants(oracle_lib, p)


def test_unroute_hand_examples(oracle_lib):
    check_unroute_hand_examples(oracle_lib)


def test_unroute_brute_force(oracle_lib):
    check_unroute_brute_force(oracle_lib, max_dim=3, max_count=3)


@pytest.mark.parametrize("seed,N,E,A", [(11, 4, 4, 64), (12, 8, 32, 900), (13, 64, 64, 5000), (14, 1, 7, 30),
                                        (15, 9, 1, 40)])
def test_unroute_inverts_the_forward_move(oracle_lib, seed, N, E, A):
    rng = np.random.default_rng(seed)
    p = workloads.make_problem(rng, A=A, H=40, N=N, E=E, token_dtype="bfloat16",
                               count_dtype=np.int64 if seed % 2 else np.int32,
                               scale_layout="e8m0", scale_cols=6, has_topk=True)
    fwd = oracle.run_problem(p, lib=oracle_lib)
    back = oracle.unroute(fwd["permute_tokens"], p.counts, permute_scales=fwd["permute_scales"],
                          permute_topk=fwd["permute_topk_weight"], lib=oracle_lib)
    assert np.array_equal(back["tokens"], p.tokens)
    assert np.array_equal(back["scales"], p.scales)
    assert np.array_equal(back["topk_weight"].view(np.uint32), p.topk.view(np.uint32))
    # and the other way round: route(unroute(y)) == y
    y = rng.integers(0, 256, size=(A, 17), dtype=np.uint16).astype(np.uint8)
    again = oracle.run(oracle.unroute(y, p.counts, lib=oracle_lib)["tokens"], p.counts, lib=oracle_lib)
    assert np.array_equal(again["permute_tokens"], y)


def test_unroute_rejects_invalid_counts():
    c = np.array([[1, 0], [2, 3]], np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.unroute(row_payload(6, 4), c)
    assert e.value.code == oracle.ORC_ERR_COUNT_NONPOS
    with pytest.raises(oracle.OracleError) as e:
        oracle.unroute(row_payload(7, 4), np.array([[1, 1], [2, 2]], np.int32))
    assert e.value.code == oracle.ORC_ERR_COUNT_SUM


@pytest.mark.parametrize("seed,N,E,dt", [(21, 4, 4, np.int32), (22, 8, 32, np.int64), (23, 1, 9, np.int32),
                                         (24, 13, 1, np.int64)])
def test_expert_token_num_modes(oracle_lib, seed, N, E, dt):
    """Count mode = numpy column sums; cumsum mode = numpy's (inclusive) cumsum of them, last = A."""
    c = workloads.counts_uniform(np.random.default_rng(seed), N, E, N * E * 5, dt)
    count = oracle.expert_token_num(c, 1, lib=oracle_lib)
    cum = oracle.expert_token_num(c, 0, lib=oracle_lib)
    assert count.dtype == dt and cum.dtype == dt
    assert np.array_equal(count, c.sum(axis=0))
    assert np.array_equal(cum, np.cumsum(c.sum(axis=0)))
    assert int(cum[-1]) == N * E * 5
    run0 = oracle.run(row_payload(N * E * 5, 2), c, expert_token_num_type=0, lib=oracle_lib)
    assert np.array_equal(run0["expert_token_num"], cum)
    with pytest.raises(oracle.OracleError):
        oracle.expert_token_num(c, 2, lib=oracle_lib)


def check_cumsum_mode(lib):
    c = np.array([[1, 2], [3, 1]], np.int32)          # hand example: column sums 4, 3
    assert oracle.expert_token_num(c, 0, lib=lib).tolist() == [4, 7]
    assert oracle.expert_token_num(c, 1, lib=lib).tolist() == [4, 3]


def test_workload_c1_invariants(oracle_lib):
    check_invariants(oracle_lib, workloads.config(1))


def test_empty_problem(oracle_lib):
    """N = 0 (no ranks) is the empty problem: A = 0 and expert_token_num all zero."""
    out = oracle.run(np.zeros((0, 8), np.uint8), np.zeros((0, 3), np.int32), lib=oracle_lib)
    assert out["permute_token_idx"].shape == (0,)
    assert out["expert_token_num"].tolist() == [0, 0, 0]


@pytest.mark.parametrize("counts,A,code", [
    ([[1, 0], [2, 3]], 6, oracle.ORC_ERR_COUNT_NONPOS),
    ([[1, -2], [2, 3]], 4, oracle.ORC_ERR_COUNT_NONPOS),
    ([[1, 1], [2, 3]], 8, oracle.ORC_ERR_COUNT_SUM),
    ([[1, 1], [2, 3]], 6, oracle.ORC_ERR_COUNT_SUM),
])
def test_rejects_invalid_counts_and_writes_nothing(oracle_lib, counts, A, code):
    for dt in (np.int32, np.int64):
        c = np.array(counts, dtype=dt)
        assert oracle.validate(c, A, lib=oracle_lib) == code
        tok = row_payload(A, 4)
        out_tok = np.full_like(tok, 0xA5)
        idx = np.full(A, -7, np.int32)
        etn = np.full(2, -9, dt)
        rc = oracle_lib.mrr_oracle_run(
            tok.ctypes.data, A, 4, c.ctypes.data, int(dt == np.int64), 2, 2, None, 0, None,
            out_tok.ctypes.data, None, idx.ctypes.data, etn.ctypes.data, None, 0)
        assert rc == code
        assert (out_tok == 0xA5).all() and (idx == -7).all() and (etn == -9).all()


def test_rejects_int64_count_beyond_int32():
    c = np.array([[2**33, 1]], dtype=np.int64)
    assert oracle.validate(c, 2**33 + 1) == oracle.ORC_ERR_ARG      # A beyond the int32 index
    assert oracle.validate(c, 5) == oracle.ORC_ERR_COUNT_SUM
    c = np.array([[2**62, 2**62, 2**62, 2**62, 3]], dtype=np.int64)  # sum wraps in int64
    assert oracle.validate(c, 3) == oracle.ORC_ERR_COUNT_SUM


# ----------------------------------------------------------------------------- planted mistakes

MUTANTS = {
    # destination walk made rank-outer (a transposed DstOffset)
    "dst_walk_rank_outer": (
        "    for (int64_t j = 0; j < E; ++j)         /* cur_expert outer */\n"
        "        for (int64_t i = 0; i < N; ++i) {   /* cur_rank inner   */\n"
        "            dst_off[i * E + j] = run;",
        "    for (int64_t i = 0; i < N; ++i)\n"
        "        for (int64_t j = 0; j < E; ++j) {\n"
        "            dst_off[i * E + j] = run;"),
    # source walk made expert-outer
    "src_walk_expert_outer": (
        "    for (int64_t i = 0; i < N; ++i)         /* cur_rank outer   */\n"
        "        for (int64_t j = 0; j < E; ++j) {   /* cur_expert inner */\n"
        "            src_off[i * E + j] = run;",
        "    for (int64_t j = 0; j < E; ++j)\n"
        "        for (int64_t i = 0; i < N; ++i) {\n"
        "            src_off[i * E + j] = run;"),
    # inclusive instead of exclusive prefix on the source side
    "src_inclusive_prefix": (
        "            src_off[i * E + j] = run;\n"
        "            run += count_at(counts, count_is_i64, E, i, j);",
        "            run += count_at(counts, count_is_i64, E, i, j);\n"
        "            src_off[i * E + j] = run - 1;"),
    # gather index written with the destination row
    "gather_writes_dst": (
        "permute_token_idx[d] = (int32_t)s;", "permute_token_idx[d] = (int32_t)d;"),
    # scatter index written at the destination position
    "scatter_swapped": (
        "permute_token_idx[s] = (int32_t)d;", "permute_token_idx[d] = (int32_t)s;"),
    # expert_token_num as row sums (a transposed operand)
    "etn_row_sums": (
        "total += count_at(counts, count_is_i64, E, i, j);\n        if (count_is_i64)",
        "total += count_at(counts, count_is_i64, E, j < N ? j : 0, i < E ? i : 0);\n        if (count_is_i64)"),
    # the same transposition in the two-mode expert_token_num
    "etn_modes_row_sums": (
        "total += count_at(counts, count_is_i64, E, i, j);\n        running += total;",
        "total += count_at(counts, count_is_i64, E, j < N ? j : 0, i < E ? i : 0);\n        running += total;"),
    # the move reads the destination offset on the source side
    "move_src_from_dst": (
        "int64_t s = src_off[i * E + j] + k;\n                int64_t d = dst_off[i * E + j] + k;\n"
        "                memcpy(permute_tokens",
        "int64_t s = dst_off[i * E + j] + k;\n                int64_t d = dst_off[i * E + j] + k;\n"
        "                memcpy(permute_tokens"),
    # the zero-count check dropped
    "no_nonpos_check": ("            if (c <= 0)\n                return ORC_ERR_COUNT_NONPOS;\n", ""),
    # inverse move: source and destination positions swapped
    "unroute_swapped": (
        "memcpy(tokens + s * row_bytes, permute_tokens + d * row_bytes, (size_t)row_bytes);",
        "memcpy(tokens + d * row_bytes, permute_tokens + s * row_bytes, (size_t)row_bytes);"),
    # inverse move: top-k weights taken from the rank-major position
    "unroute_topk_from_src": ("topk_w[s] = permute_topk_w[d];", "topk_w[s] = permute_topk_w[s];"),
    # inverse move: scale rows moved with the token row size
    # cumsum mode made exclusive (the running total taken before adding the expert's count)
    "cumsum_exclusive": ("        running += total;\n        const int64_t v = expert_token_num_type == 1 ? total : running;",
                         "        const int64_t v = expert_token_num_type == 1 ? total : running;\n        running += total;"),
    "unroute_scale_stride": ("scales + s * scale_row_bytes, permute_scales + d * scale_row_bytes,",
                             "scales + s * scale_row_bytes, permute_scales + d * row_bytes,"),
}

PINS = [check_hand_examples, check_transpose_closed_form,
        lambda lib: check_brute_force(lib, max_dim=2, max_count=2),
        check_unroute_hand_examples, lambda lib: check_unroute_brute_force(lib, max_dim=2, max_count=2),
        check_cumsum_mode]


def _nonpos_pin(lib):
    c = np.array([[1, 0], [2, 3]], np.int32)
    assert oracle.validate(c, 6, lib=lib) == oracle.ORC_ERR_COUNT_NONPOS


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = open(oracle.SOURCE, encoding="utf-8").read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found in the oracle source"
    mutant = tmp_path / f"{name}.c"
    mutant.write_text(src.replace(old, new), encoding="utf-8")
    lib = oracle.load(oracle.build(str(mutant), str(tmp_path / f"lib{name}.so")))
    caught = False
    for pin in PINS + [_nonpos_pin]:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError):
            caught = True
            break
    assert caught, f"planted mistake {name} passed every pin"
