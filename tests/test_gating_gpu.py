"""GPU parity of the MoE gating top-k op (mrr_gating_topk_run) against the CPU oracle.

Integer results (expert_idx) must equal the oracle's wherever the choice is unique.  Both sides
decide on float32 scores, but the GPU computes the normalisation with float32 exp/log while the
oracle rounds a float64 result, so two scores within a few float32 ulps may order differently.
In such rows the GPU's experts must still be a valid top-k under the oracle's scores within
that margin: for groups, kept groups that score among the best and no unchosen expert of a kept
group above a chosen one; y_out must equal the weight formula applied to the oracle's scores of
the GPU's own experts; and each kind of stress row has its own bound on such rows.  Floating
outputs: y_out within the rounding of its dtype (float16 2^-10, bfloat16 2^-7, float32 1e-5,
relative) plus 1e-6; norm_out (float32) within 2e-5 relative.

Source: "CANN 自定义算子详解：npu_moe_gating_top_k" (m.qwbw.cn/news/316089), sections 归一化公式,
分组排序公式, 专家选择公式, 路由权重缩放公式 and 调用示例 (the shapes of its test cases).
"""
import numpy as np
import pytest

from oracle import gating
import moe_expert_token_gb300.mrr_v2 as m
from harness import DevBuf

pytestmark = pytest.mark.gpu

RTOL = {"float16": 2.0 ** -10, "bfloat16": 2.0 ** -7, "float32": 1e-5}
CODE = {"float16": m.MRR_GATE_F16, "bfloat16": m.MRR_GATE_BF16, "float32": m.MRR_GATE_F32}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_token_gb300 import build

    build.build()
    m.load_library()


def as_dtype(a: np.ndarray, dt: str) -> np.ndarray:
    """Round float32 values to dt and return them as float32 (what both sides read)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(getattr(torch, dt)).to(torch.float32).numpy()


def raw(a: np.ndarray, dt: str) -> np.ndarray:
    import torch

    if a.size == 0:
        return np.zeros(0, np.uint8)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(getattr(torch, dt)).view(torch.uint8).numpy()


def run_gpu_gating(x32, dt, k, *, bias=None, input_ids=None, tid2eid=None, extra_bias=None, mask=None,
                   out_flag=True, expect=m.MRR_OK, x_offset=0, out_offset=0, **kw):
    import torch

    d = torch.device("cuda:0")
    T, e = x32.shape
    xb = DevBuf.of(raw(x32, dt), d, offset=x_offset)
    bb = None if bias is None else DevBuf.of(raw(bias, dt), d)
    eb = None if extra_bias is None else DevBuf.of(raw(extra_bias, dt), d)
    mb = None if mask is None else DevBuf.of(np.asarray(mask, np.uint8), d)
    ib = None if input_ids is None else DevBuf.of(np.asarray(input_ids, np.int64), d)
    tb = None if tid2eid is None else DevBuf.of(np.asarray(tid2eid, np.int32), d)
    esz = {"float16": 2, "bfloat16": 2, "float32": 4}[dt]
    y = DevBuf(T * k * esz, d)
    idx = DevBuf(T * k * 4, d)
    out = DevBuf(T * e * 4, d, offset=out_offset) if out_flag else None
    ws = DevBuf(4096, d, fill=0x5A)
    args = dict(k_group=1, group_count=1, routed_scaling_factor=1.0, eps=1e-20, group_select_mode=0,
                renorm=0, norm_type=0)
    args.update(kw)
    s = torch.cuda.current_stream().cuda_stream
    P = lambda b: None if b is None else b.ptr
    st = m.mrr_gating_topk_run(xb.ptr, CODE[dt], T, e, k, P(bb), P(ib), P(tb),
                               0 if tid2eid is None else len(tid2eid), P(eb), P(mb), args["k_group"],
                               args["group_count"], args["routed_scaling_factor"], args["eps"],
                               args["group_select_mode"], args["renorm"], args["norm_type"], y.ptr,
                               idx.ptr, P(out), ws.ptr, ws.n, s)
    assert st == expect, m.mrr_status_str(st)
    if st != m.MRR_OK:
        return None
    res = {"status": m.mrr_v2_read_status(ws.ptr, ws.n, s)}
    torch.cuda.synchronize()
    if T == 0:
        res["guards"] = all(b.guards_intact() for b in (y, idx, out) if b is not None)
        return res
    yh = y.host()
    res["y_out"] = (torch.from_numpy(yh.copy()).view(getattr(torch, dt)).float().numpy().reshape(T, k))
    res["expert_idx"] = idx.host().view(np.int32).reshape(T, k)
    res["norm_out"] = None if out is None else out.host().view(np.float32).reshape(T, e)
    res["guards"] = all(b.guards_intact() for b in (y, idx, out) if b is not None)
    return res


def _group_scores(row: np.ndarray, G: int, mode: int) -> np.ndarray:
    """Group scores as the oracle forms them from float32 scores: the maximum (mode 0) or the
    float32 sum of the two largest (mode 1)."""
    g = np.sort(row.astype(np.float32).reshape(G, -1), axis=1)[:, ::-1]
    return g[:, 0].astype(np.float64) if mode == 0 else (g[:, 0] + g[:, 1]).astype(np.float32).astype(np.float64)


def _grouped_choice_problem(row, gi, G, kg, mode, margin):
    """None if the experts gi are a valid grouped top-k under the float32 scores ``row`` with
    every comparison allowed ``margin`` of slack; else why not.  Valid means: some set K of kg
    groups, each scoring at least the kg-th best group score minus the margin, holds every chosen
    expert, and no unchosen expert of K scores more than the lowest chosen one plus the margin
    (the page's 分组排序公式 then 专家选择公式, decided within the margin)."""
    from itertools import combinations, islice

    e = row.size
    gsize = e // G
    gs = _group_scores(row, G, mode)
    order = sorted(range(G), key=lambda g: (-gs[g], g))
    kth = gs[order[kg - 1]]
    used = sorted({int(j) // gsize for j in gi})
    if len(used) > kg:
        return f"experts from {len(used)} groups, k_group is {kg}"
    for g in used:
        if gs[g] < kth - margin:
            return f"group {g} scores {gs[g]!r}, below the kept groups' {kth!r}"
    chosen = set(int(j) for j in gi)
    lo = min(float(row[j]) for j in gi)

    def unchosen_ok(groups):
        return all(float(row[j]) <= lo + margin
                   for g in groups for j in range(g * gsize, (g + 1) * gsize) if j not in chosen)

    if not unchosen_ok(used):
        return "an unchosen expert of a kept group outscores a chosen one"
    spare = [g for g in order if g not in used and gs[g] >= kth - margin]
    for extra in islice(combinations(spare, kg - len(used)), 5000):
        if unchosen_ok(extra):
            return None
    return "no set of kept groups completes the choice"


def _decisive_near_tie(s, x, k, G, kg, mode):
    """True when the oracle's float32 scores ``s`` of one row hold a near-tie that decides the
    result: two scores within 16 float32 ulps of the larger one (a few ulps of float32 exp / log
    on the GPU against a correctly rounded oracle can swap them) at the kept-group boundary, or
    between consecutive experts of the top k + 1 among the kept groups (the order of the picks,
    and the boundary of the choice).  Two experts with equal logits (``x``) and equal scores
    are an exact tie, which both sides break the same way (lower index), not a near-tie."""
    eps = float(np.finfo(np.float32).eps)

    def close(a, b):
        return abs(a - b) <= 16 * eps * max(abs(a), abs(b))

    e = s.size
    cand = list(range(e))
    if G > 1:
        gs = _group_scores(s, G, mode)
        order = sorted(range(G), key=lambda g: (-gs[g], g))
        if kg < G and close(gs[order[kg - 1]], gs[order[kg]]):
            return True
        gsize = e // G
        cand = [j for g in order[:kg] for j in range(g * gsize, (g + 1) * gsize)]
    top = sorted(cand, key=lambda j: (-float(s[j]), j))[:k + 1]
    for a, b in zip(top, top[1:]):
        exact = x is not None and x[a] == x[b] and s[a] == s[b]
        if close(float(s[a]), float(s[b])) and not exact:
            return True
    return False


def check_against_oracle(gpu, ref, dt, params, max_tie_rows=0.02, x=None):
    """The GPU's outputs against the oracle's.  Rows with the oracle's experts: y_out within RTOL.
    Other rows (near-ties: scores within a few float32 ulps, which the GPU's float32 exp / log may
    order differently from the oracle's rounded float64) must hold a valid choice under the
    oracle's float32 scores: distinct in-range experts in descending score order; ungrouped, the
    same multiset of scores as the oracle's choice; grouped, a valid group-then-expert choice
    (_grouped_choice_problem); and y_out equal to the oracle's weight formula (路由权重缩放公式)
    applied to the oracle's scores of the GPU's own experts.  A differing row must also hold a
    decisive near-tie in the oracle's own scores (_decisive_near_tie; ``x`` gives the logits, so
    that exact ties of equal logits do not count).  At most max_tie_rows (a fraction of the rows,
    at least one row if > 0) may differ.  Returns the number of differing rows."""
    assert gpu["status"] == m.MRR_OK
    assert gpu["guards"]
    T, k = ref["expert_idx"].shape
    s = ref["norm_out"].astype(np.float64)
    e = s.shape[1]
    G = params.get("group_count", 1)
    kg = params.get("k_group", 1)
    mode = params.get("group_select_mode", 0)
    scale = params.get("routed_scaling_factor", 1.0)
    eps = params.get("eps", 1e-20)
    tie_rows = 0
    for t in range(T):
        gi, ri = gpu["expert_idx"][t], ref["expert_idx"][t]
        if np.array_equal(gi, ri):
            assert np.allclose(gpu["y_out"][t], ref["y_out"][t], rtol=RTOL[dt], atol=1e-6), t
            continue
        tie_rows += 1
        assert _decisive_near_tie(ref["norm_out"][t], None if x is None else x[t], k, G, kg, mode), \
            (t, "differs from the oracle with no near-tie in the oracle's scores")
        assert len(set(gi.tolist())) == k and gi.min() >= 0 and gi.max() < e, t
        margin = 8 * np.finfo(np.float32).eps * max(1.0, np.abs(s[t]).max())
        assert np.all(np.diff(s[t, gi]) <= margin), (t, "experts not in descending score order")
        if G == 1:
            assert np.allclose(np.sort(s[t, gi]), np.sort(s[t, ri]), atol=margin), t
        else:
            why = _grouped_choice_problem(ref["norm_out"][t], gi, G, kg, mode, margin)
            assert why is None, (t, why)
        y = s[t, gi]
        y_ref = y / (y.sum() + eps) * scale
        assert np.allclose(gpu["y_out"][t], y_ref, rtol=RTOL[dt], atol=1e-6), (t, "y_out of the chosen set")
    bound = 0 if max_tie_rows == 0 else max(1, int(round(max_tie_rows * T)))
    assert tie_rows <= bound, f"{tie_rows} of {T} rows differ (at most {bound})"
    if gpu["norm_out"] is not None:
        assert np.allclose(gpu["norm_out"], ref["norm_out"], rtol=2e-5, atol=1e-6)
    return tie_rows


def test_page_example_384_experts_top6():
    """The page's basic case: 16 tokens, 384 experts, top-6, sigmoid, float16, no groups."""
    rng = np.random.default_rng(1)
    x = as_dtype(rng.standard_normal((16, 384)), "float16")
    kw = dict(norm_type=1, eps=1e-6)
    ref = gating.gating_topk(x, 6, **kw)
    check_against_oracle(run_gpu_gating(x, "float16", 6, **kw), ref, "float16", kw)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("norm_type", [0, 1, 2])
@pytest.mark.parametrize("mode", [0, 1])
def test_grouped_with_bias(dt, norm_type, mode):
    """Grouped ranking (256 experts, 8 groups, keep 4, top-8) with a bias, all norms and dtypes."""
    rng = np.random.default_rng(10 * norm_type + mode)
    T, e = 512, 256
    x = as_dtype(rng.standard_normal((T, e)) * 2, dt)
    bias = as_dtype(rng.standard_normal(e) * 0.05, dt)
    kw = dict(k_group=4, group_count=8, group_select_mode=mode, norm_type=norm_type,
              routed_scaling_factor=2.5, eps=1e-20)
    ref = gating.gating_topk(x, 8, bias=bias, **kw)
    check_against_oracle(run_gpu_gating(x, dt, 8, bias=bias, **kw), ref, dt, kw)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("e", [128, 256, 384, 512])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("k_group", [1, 3, 4, 7])
def test_grouped_sigmoid_instance_matches_general(dt, e, mode, k_group):
    """Sigmoid with a bias and lane-aligned groups (8 groups of e / 8, keep k_group, top-8), no
    norm_out: the specialised kernel instance runs.  Asking for norm_out runs the general one.  The
    two must agree bit for bit (same arithmetic, same order), and both against the oracle."""
    rng = np.random.default_rng(e + mode + 10 * k_group)
    T = 1024
    x = as_dtype(rng.standard_normal((T, e)) * 2, dt)
    bias = as_dtype(rng.standard_normal(e) * 0.05, dt)
    kw = dict(k_group=k_group, group_count=8, group_select_mode=mode, norm_type=1, routed_scaling_factor=2.5,
              eps=1e-20)
    fast = run_gpu_gating(x, dt, 8, bias=bias, out_flag=False, **kw)
    full = run_gpu_gating(x, dt, 8, bias=bias, out_flag=True, **kw)
    assert fast["status"] == m.MRR_OK and fast["guards"]
    assert np.array_equal(fast["expert_idx"], full["expert_idx"])
    assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
    ref = gating.gating_topk(x, 8, bias=bias, **kw)
    check_against_oracle(fast, ref, dt, kw)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("e", [256, 512])
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("k_group", [1, 4, 7])
def test_grouped_sigmoid_instance_ties(dt, e, mode, k_group):
    """The specialised grouped instance on rows full of exact ties: logits 0 or 2 (every 5th row
    all 1) and, for group maxima, a bias of 0 or 1/2 leave at most four distinct scores per row.
    Equal scores and equal group scores go to the lower expert and group, exactly as the oracle's
    stable order has them, and the instance agrees with the general one bit for bit.  (For group
    sums the bias is 0: with more distinct scores two different pairs can have the same exact sum,
    which float32 rounding may order either way.)"""
    rng = np.random.default_rng(e + 3 * mode + k_group)
    T = 320
    x = rng.choice(np.array([0.0, 2.0], np.float32), size=(T, e))
    x[::5] = 1.0
    bias = (rng.integers(0, 2, size=e) * 0.5 if mode == 0 else np.zeros(e)).astype(np.float32)
    kw = dict(k_group=k_group, group_count=8, group_select_mode=mode, norm_type=1, routed_scaling_factor=2.5,
              eps=1e-20)
    fast = run_gpu_gating(x, dt, 8, bias=bias, out_flag=False, **kw)
    full = run_gpu_gating(x, dt, 8, bias=bias, out_flag=True, **kw)
    assert np.array_equal(fast["expert_idx"], full["expert_idx"])
    assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
    ref = gating.gating_topk(x, 8, bias=bias, **kw)
    assert np.array_equal(fast["expert_idx"], ref["expert_idx"])
    check_against_oracle(fast, ref, dt, kw, max_tie_rows=0)


@pytest.mark.parametrize("norm_type", [0, 1, 2])
def test_additional_bias_rows(norm_type):
    """The page's additional_bias case: every other token uses additional_bias instead of bias."""
    rng = np.random.default_rng(20 + norm_type)
    T, e = 64, 384
    x = as_dtype(rng.standard_normal((T, e)), "float16")
    bias = as_dtype(rng.random(e), "float16")
    extra = as_dtype(rng.random(e), "float16")
    mask = np.zeros(T, bool)
    mask[::2] = True
    ref = gating.gating_topk(x, 6, bias=bias, additional_bias=extra, additional_token_mask=mask,
                             norm_type=norm_type, eps=1e-6)
    gpu = run_gpu_gating(x, "float16", 6, bias=bias, extra_bias=extra, mask=mask, norm_type=norm_type, eps=1e-6)
    check_against_oracle(gpu, ref, "float16", dict(norm_type=norm_type, eps=1e-6))


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
def test_hash_routing(dt):
    """The page's hash case: 100-entry vocabulary, tid2eid [100, k]."""
    rng = np.random.default_rng(30)
    T, e, k, n = 128, 384, 6, 100
    x = as_dtype(rng.standard_normal((T, e)), dt)
    ids = rng.integers(0, n, size=T)
    tab = rng.integers(0, e, size=(n, k)).astype(np.int32)
    ref = gating.gating_topk(x, k, input_ids=ids, tid2eid=tab, norm_type=1, eps=1e-6)
    gpu = run_gpu_gating(x, dt, k, input_ids=ids, tid2eid=tab, norm_type=1, eps=1e-6)
    assert np.array_equal(gpu["expert_idx"], ref["expert_idx"])
    check_against_oracle(gpu, ref, dt, dict(norm_type=1, eps=1e-6), max_tie_rows=0)


def test_hash_index_out_of_range_is_reported():
    rng = np.random.default_rng(31)
    x = as_dtype(rng.standard_normal((8, 64)), "float32")
    ids = np.array([0, 1, 2, 5, 0, 1, 2, 3])                 # 5 is outside a 4-entry table
    tab = rng.integers(0, 64, size=(4, 4)).astype(np.int32)
    tab[2, 1] = 64                                           # an expert id outside [0, e)
    gpu = run_gpu_gating(x, "float32", 4, input_ids=ids, tid2eid=tab, norm_type=1)
    assert gpu["status"] == m.MRR_ERR_INDEX
    assert gpu["guards"]


@pytest.mark.parametrize("T,e,k,G,kg", [(3, 1024, 64, 1, 1), (257, 33, 5, 1, 1), (40, 1024, 16, 32, 8),
                                        (100, 64, 64, 1, 1), (16384, 256, 8, 8, 4), (5, 2, 2, 2, 2),
                                        (64, 160, 5, 5, 2), (64, 1000, 16, 40, 7), (32, 1024, 8, 1024, 9),
                                        (64, 384, 8, 8, 4), (64, 64, 4, 2, 1), (50, 96, 10, 6, 3),
                                        (64, 200, 7, 10, 4), (64, 100, 5, 4, 2), (70, 512, 20, 16, 5)])
def test_shapes(T, e, k, G, kg):
    rng = np.random.default_rng(T + e)
    x = as_dtype(rng.standard_normal((T, e)), "bfloat16")
    kw = dict(k_group=kg, group_count=G, norm_type=0, eps=1e-9)
    ref = gating.gating_topk(x, k, **kw)
    gpu = run_gpu_gating(x, "bfloat16", k, out_flag=(T * e <= 1 << 20), **kw)
    check_against_oracle(gpu, ref, "bfloat16", kw)


def test_no_tokens():
    gpu = run_gpu_gating(np.zeros((0, 16), np.float32), "float32", 2, norm_type=1)
    assert gpu["status"] == m.MRR_OK and gpu["guards"]


def test_torch_level_call_3d_input():
    import torch

    rng = np.random.default_rng(40)
    x = as_dtype(rng.standard_normal((2, 8, 256)), "float32")
    xt = torch.from_numpy(x).cuda()
    y, idx, out = m.moe_gating_top_k(xt, 8, k_group=4, group_count=8, group_select_mode=1, norm_type=1,
                                     out_flag=True, check_status=True)
    assert tuple(y.shape) == (2, 8, 8) and tuple(idx.shape) == (2, 8, 8) and tuple(out.shape) == (2, 8, 256)
    ref = gating.gating_topk(x.reshape(16, 256), 8, k_group=4, group_count=8, group_select_mode=1, norm_type=1)
    check_against_oracle({"status": m.MRR_OK, "guards": True, "y_out": y.reshape(16, 8).cpu().numpy(),
                          "expert_idx": idx.reshape(16, 8).cpu().numpy(),
                          "norm_out": out.reshape(16, 256).cpu().numpy()}, ref, "float32",
                         dict(k_group=4, group_count=8, group_select_mode=1, norm_type=1))


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("e,k,G,kg,mode", [(384, 6, 1, 1, 0), (256, 8, 8, 4, 1), (160, 5, 5, 2, 1),
                                            (1000, 16, 40, 7, 0), (64, 64, 1, 1, 0), (96, 10, 6, 3, 1)])
def test_ties_go_to_the_lower_index(dt, e, k, G, kg, mode):
    """Integer logits (many equal scores) and constant rows: equal scores must go to the lower
    group / expert index, exactly as the oracle orders them."""
    rng = np.random.default_rng(e + k + G)
    x = rng.integers(-2, 3, size=(48, e)).astype(np.float32)
    x[::7] = 0.5                                              # whole rows of equal scores
    kw = dict(k_group=kg, group_count=G, group_select_mode=mode, norm_type=1, eps=1e-9)
    ref = gating.gating_topk(x, k, **kw)
    gpu = run_gpu_gating(x, dt, k, **kw)
    assert np.array_equal(gpu["expert_idx"], ref["expert_idx"])
    check_against_oracle(gpu, ref, dt, kw, max_tie_rows=0)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("e", [256, 384, 96, 33])
def test_misaligned_rows_use_narrower_loads(dt, e):
    """x and norm_out at odd byte offsets: the kernel must fall back to narrower loads and stores."""
    rng = np.random.default_rng(50 + e)
    x = as_dtype(rng.standard_normal((40, e)), dt)
    esz = 4 if dt == "float32" else 2
    kw = dict(k_group=1, group_count=1, norm_type=0, eps=1e-9)
    ref = gating.gating_topk(x, 6, **kw)
    for x_off, o_off in [(esz, 4), (2 * esz, 8), (4 * esz, 12)]:
        gpu = run_gpu_gating(x, dt, 6, x_offset=x_off, out_offset=o_off, **kw)
        check_against_oracle(gpu, ref, dt, kw)


def test_grouped_additional_bias_and_norm_out():
    """additional_bias rows together with grouped ranking (both group paths) and norm_out."""
    rng = np.random.default_rng(60)
    for e, G, kg, k in [(256, 8, 3, 6), (160, 5, 2, 4)]:
        x = as_dtype(rng.standard_normal((64, e)), "bfloat16")
        bias = as_dtype(rng.random(e) * 0.2, "bfloat16")
        extra = as_dtype(rng.random(e) * 0.2, "bfloat16")
        mask = rng.random(64) < 0.5
        kw = dict(k_group=kg, group_count=G, group_select_mode=1, norm_type=2, routed_scaling_factor=1.5, eps=1e-9)
        ref = gating.gating_topk(x, k, bias=bias, additional_bias=extra, additional_token_mask=mask, **kw)
        gpu = run_gpu_gating(x, "bfloat16", k, bias=bias, extra_bias=extra, mask=mask, **kw)
        check_against_oracle(gpu, ref, "bfloat16", kw)


# Kinds of _logit_rows with no decisive near-tie by construction: 16-bit N(0,1) logits and ramp
# logits leave gaps far above a float32 ulp between the scores around the k-th pick (distinct
# 16-bit logits differ by at least 2^-11 relative), and small-integer and +-0 logits tie exactly
# (equal logits, equal scores, lower index first on both sides).  Their rows must match the
# oracle exactly.  (Float32 N(0,1) logits can fall arbitrarily close: about one row in 800 of
# them holds a near-tie, so for float32 x that kind gets only the per-row rule below.)  N(0,16) logits reach the range where sigmoid is within
# 1e-5 of 1, and logits in [10, 20] saturate it: there, rows may differ, but only rows whose
# oracle scores hold a decisive near-tie, and each such row must still be a valid choice.
TIE_FREE_KINDS = (0, 2, 3, 4)


def _logit_rows(rng, T_each, e, dt):
    """Rows of several kinds: N(0,1), N(0,16), small integers (many equal logits), an ascending
    ramp (every pick from the last lanes), +-0 only, and logits in [10, 20] where float32 sigmoid
    saturates (different logits, equal scores)."""
    kinds = [rng.standard_normal((T_each, e)),
             rng.standard_normal((T_each, e)) * 4,
             rng.integers(-2, 3, size=(T_each, e)).astype(np.float64),
             np.tile(np.linspace(-3, 3, e), (T_each, 1)),
             np.where(rng.random((T_each, e)) < 0.5, 0.0, -0.0),
             rng.uniform(10, 20, size=(T_each, e))]
    return as_dtype(np.concatenate(kinds), dt), len(kinds)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("norm_type", [0, 1, 2])
@pytest.mark.parametrize("e,k", [(384, 6), (256, 8), (1, 1), (7, 7), (33, 5), (64, 32), (100, 7), (160, 5),
                                 (512, 20), (1000, 16), (1024, 32)])
def test_rank_by_logit_matches_full_evaluation(dt, norm_type, e, k):
    """With no bias, groups, hash table or norm_out, the kernel ranks by logit and scores only the
    chosen experts (softmax still sums exp over the row).  Asking for norm_out makes it evaluate every
    score instead: the two runs must agree bit for bit, on rows that stress equal logits, saturated
    scores and picks crowded into one lane, and match the oracle."""
    rng = np.random.default_rng(e * 100 + k + 7 * norm_type)
    T_each = 24
    x, n_kinds = _logit_rows(rng, T_each, e, dt)
    kw = dict(norm_type=norm_type, eps=1e-9, routed_scaling_factor=1.7)
    fast = run_gpu_gating(x, dt, k, out_flag=False, **kw)
    full = run_gpu_gating(x, dt, k, out_flag=True, **kw)
    assert fast["status"] == m.MRR_OK and fast["guards"]
    assert np.array_equal(fast["expert_idx"], full["expert_idx"])
    assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
    ref = gating.gating_topk(x, k, **kw)
    for kind in range(n_kinds):
        rows = slice(kind * T_each, (kind + 1) * T_each)
        near = sum(_decisive_near_tie(ref["norm_out"][t], x[t], k, 1, 1, 0)
                   for t in range(rows.start, rows.stop))
        if kind in TIE_FREE_KINDS and not (kind == 0 and dt == "float32"):
            assert near == 0, (kind, near)
        # at most the kind's near-tie rows may differ (each is also checked to be one of them)
        check_against_oracle({**fast, "expert_idx": fast["expert_idx"][rows], "y_out": fast["y_out"][rows]},
                             {key: v[rows] for key, v in ref.items()}, dt, kw,
                             max_tie_rows=near / T_each, x=x[rows])


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("norm_type", [0, 1, 2])
@pytest.mark.parametrize("e", [128, 256, 384, 512])
@pytest.mark.parametrize("k", [2, 4, 6, 8])
def test_fixed_shape_logit_instances(dt, norm_type, e, k):
    """e = 32 x experts-per-lane (128 to 512) and k in {2, 4, 6, 8}, 16-byte rows, no norm_out:
    the fixed-shape rank-by-logit instances run (the pick loop unrolled).  They must agree bit for
    bit with the full evaluation (norm_out asked for) on the stress rows, and with the oracle."""
    rng = np.random.default_rng(e * 10 + k + 1000 * norm_type)
    T_each = 8
    x, n_kinds = _logit_rows(rng, T_each, e, dt)
    kw = dict(norm_type=norm_type, eps=1e-9, routed_scaling_factor=1.3)
    fast = run_gpu_gating(x, dt, k, out_flag=False, **kw)
    full = run_gpu_gating(x, dt, k, out_flag=True, **kw)
    assert fast["status"] == m.MRR_OK and fast["guards"]
    assert np.array_equal(fast["expert_idx"], full["expert_idx"])
    assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
    ref = gating.gating_topk(x, k, **kw)
    for kind in range(n_kinds):
        rows = slice(kind * T_each, (kind + 1) * T_each)
        near = sum(_decisive_near_tie(ref["norm_out"][t], x[t], k, 1, 1, 0)
                   for t in range(rows.start, rows.stop))
        check_against_oracle({**fast, "expert_idx": fast["expert_idx"][rows], "y_out": fast["y_out"][rows]},
                             {key: v[rows] for key, v in ref.items()}, dt, kw,
                             max_tie_rows=near / T_each, x=x[rows])


@pytest.mark.parametrize("dt,T,e,k,norm_type", [("float16", 16384, 384, 6, 1), ("bfloat16", 20000, 256, 8, 2),
                                                ("float16", 7001, 1000, 16, 1), ("bfloat16", 9000, 768, 32, 1),
                                                ("float32", 16384, 384, 6, 1), ("float32", 10000, 160, 9, 2),
                                                ("bfloat16", 16384, 256, 8, 0), ("float32", 8000, 64, 4, 0)])
def test_rank_by_logit_many_rows(dt, T, e, k, norm_type):
    """Full-size batches: each warp ranks several rows, loading the next row while it works on the
    current one.  Bit for bit against the full evaluation, and against the oracle."""
    rng = np.random.default_rng(T + e + k)
    x = as_dtype(rng.standard_normal((T, e)), dt)
    kw = dict(norm_type=norm_type, eps=1e-6, routed_scaling_factor=2.5)
    fast = run_gpu_gating(x, dt, k, out_flag=False, **kw)
    full = run_gpu_gating(x, dt, k, out_flag=True, **kw)
    assert np.array_equal(fast["expert_idx"], full["expert_idx"])
    assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
    ref = gating.gating_topk(x, k, **kw)
    check_against_oracle(fast, ref, dt, kw)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("e", [384, 100, 33, 1024])
def test_rank_by_logit_misaligned_rows(dt, e):
    """x at offsets of 1, 2 and 4 elements: the rank-by-logit loads fall back to narrower words
    or single elements."""
    rng = np.random.default_rng(70 + e)
    x = as_dtype(rng.standard_normal((300, e)), dt)
    kw = dict(norm_type=1, eps=1e-6)
    ref = gating.gating_topk(x, 6, **kw)
    esz = 4 if dt == "float32" else 2
    for x_off in (esz, 2 * esz, 4 * esz):
        fast = run_gpu_gating(x, dt, 6, out_flag=False, x_offset=x_off, **kw)
        full = run_gpu_gating(x, dt, 6, out_flag=True, x_offset=x_off, **kw)
        assert np.array_equal(fast["expert_idx"], full["expert_idx"])
        assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
        check_against_oracle(fast, ref, dt, kw)


def _ordered(f32: np.ndarray) -> np.ndarray:
    """float32 values as integers that step by one per representable float (-0 and +0 equal)."""
    b = f32.astype(np.float32).view(np.int32).astype(np.int64)
    return np.where(b < 0, -(b & 0x7FFFFFFF), b)


@pytest.mark.parametrize("dt", ["float16", "bfloat16", "float32"])
@pytest.mark.parametrize("grouped", [False, True])
def test_infinite_logits_with_sigmoid(dt, grouped):
    """Logits of +inf and -inf among finite ones, sigmoid scores: +inf scores 1 and -inf scores 0
    (归一化公式), so the experts and weights are those of the oracle; equal scores (several +inf
    logits, or a finite logit whose sigmoid rounds to 1) go to the lower expert.  Grouped: the
    8-group top-8 shape with a bias (the specialised instance) and, with norm_out, the general
    one, which must agree bit for bit.  Ungrouped: no bias, so rows are ranked by logit."""
    rng = np.random.default_rng(7 + grouped)
    T, e = 512, 256
    x = as_dtype(rng.standard_normal((T, e)) * 3, dt)
    x[rng.random((T, e)) < 0.05] = np.inf
    x[rng.random((T, e)) < 0.05] = -np.inf
    x[::9] = -np.inf                                # rows with every score 0 (plus the bias)
    x[1::9, :40] = np.inf                           # rows whose best scores all tie at 1
    if grouped:
        bias = as_dtype(rng.random(e) * 0.1, dt)
        kw = dict(k_group=4, group_count=8, group_select_mode=1, norm_type=1, routed_scaling_factor=2.5,
                  eps=1e-20)
        fast = run_gpu_gating(x, dt, 8, bias=bias, out_flag=False, **kw)
        full = run_gpu_gating(x, dt, 8, bias=bias, out_flag=True, **kw)
        assert np.array_equal(fast["expert_idx"], full["expert_idx"])
        assert np.array_equal(fast["y_out"].view(np.uint32), full["y_out"].view(np.uint32))
        ref = gating.gating_topk(x, 8, bias=bias, **kw)
    else:
        kw = dict(norm_type=1, eps=1e-6)
        fast = run_gpu_gating(x, dt, 6, out_flag=False, **kw)
        ref = gating.gating_topk(x, 6, **kw)
    assert np.all(np.isfinite(fast["y_out"]))
    check_against_oracle(fast, ref, dt, kw, x=x)


@pytest.mark.parametrize("dt", ["float16", "bfloat16"])
@pytest.mark.parametrize("norm_type,bound", [(1, 4), (2, 3)])
def test_scores_of_every_16bit_logit(dt, norm_type, bound):
    """Sigmoid and softplus scores (norm_out, no bias) for every finite 16-bit logit, against the
    exact function rounded to float32: within `bound` float32 ulps.  Where the exact score is
    below the smallest normal float, the kernel may flush it to zero (归一化公式)."""
    import torch

    bits = np.arange(65536, dtype=np.uint16)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(getattr(torch, dt)).float().numpy()
    x[~np.isfinite(x)] = 0.0
    x = x.reshape(256, 256)
    gpu = run_gpu_gating(x, dt, 1, norm_type=norm_type)
    assert gpu["status"] == m.MRR_OK and gpu["guards"]
    xd = x.astype(np.float64)
    with np.errstate(over="ignore"):   # exp(-x) overflows to inf for x below -709: sigmoid 0
        exact = 1.0 / (1.0 + np.exp(-xd)) if norm_type == 1 else np.logaddexp(0.0, xd)
    exact32 = exact.astype(np.float32)
    got = gpu["norm_out"]
    tiny = np.abs(exact) < np.finfo(np.float32).tiny
    assert np.all(np.abs(got[tiny]) < np.finfo(np.float32).tiny)
    ulps = np.abs(_ordered(got) - _ordered(exact32))[~tiny]
    print(f"{dt} norm_type {norm_type}: max {ulps.max()} ulp, mean {ulps.mean():.3f}")
    assert ulps.max() <= bound
