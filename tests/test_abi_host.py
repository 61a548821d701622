"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
include/mrr_v2.h declares, and rejects bad arguments before touching CUDA.

Validation rules (MoeReRoutingV2 article, sections 参数说明, 参数取值细节, 约束说明 and
Torch 扩展的图转换细节): 0 < H < 16384; every count > 0 with Sum(counts) = A (so N*E <= A);
the index output is int32 (A <= INT32_MAX); expert_token_num_type and idx_type are 0 or 1, and
only expert_token_num_type = 1 is supported; expert_topk_weight and permute_topk_weight are
given together.
"""
import ctypes
import subprocess

import pytest

from moe_expert_token_gb300 import build as mbuild
import moe_expert_token_gb300.mrr_v2 as m


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return m.load_library()


def test_exports_every_header_function(lib):
    names = m.header_functions()
    assert set(names) == {"mrr_v2_plan", "mrr_v2_run", "mrr_v2_run_plan", "mrr_v2_read_status",
                          "mrr_status_str", "mrr_v2_run_noalloc", "mrr_v2_unroute_plan",
                          "mrr_v2_unroute", "mrr_v1_run", "mrr_gating_topk_run", "mrr_v2_run_multi",
                          "mrr_v2_run_plan_multi", "mrr_v2_offsets_host", "mrr_v2_push"}
    out = subprocess.run(["nm", "-D", "--defined-only", m.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_library_is_built_for_sm103a_only():
    """Every translation unit is compiled with one -gencode, for sm_103a: GPU code of no other
    architecture (and no PTX for a JIT fallback) is put into the library."""
    flags = mbuild.ARCH_FLAGS
    assert flags == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in list(range(0, 11)) + [16, 17, 18, 19, 20]:
        s = m.mrr_status_str(code)
        assert s.startswith("MRR_"), (code, s)
    assert m.mrr_status_str(12345) == "unknown mrr_status"


def plan(**kw):
    args = dict(A=16384, H=7168, dt=m.MRR_I8, N=16, E=16, count_is_i64=0, sl=m.MRR_SCALE_F32_A,
                scale_cols=1, has_topk=0, expert_token_num_type=1, idx_type=0, device=0)
    args.update(kw)
    return m.mrr_v2_plan(**args)[0]


@pytest.mark.parametrize("kw,code", [
    (dict(dt=99), m.MRR_ERR_DTYPE),
    (dict(sl=7), m.MRR_ERR_DTYPE),
    (dict(count_is_i64=2), m.MRR_ERR_DTYPE),
    (dict(H=0), m.MRR_ERR_SHAPE),
    (dict(H=-3), m.MRR_ERR_SHAPE),
    (dict(H=16384), m.MRR_ERR_SHAPE),
    (dict(H=79, dt=m.MRR_F4E2M1), m.MRR_ERR_SHAPE),          # FP4 packs two per byte
    (dict(A=-1), m.MRR_ERR_SHAPE),
    (dict(A=2**31), m.MRR_ERR_SHAPE),                        # int32 index output
    (dict(A=100, N=16, E=16), m.MRR_ERR_SHAPE),              # N*E > A: no positive counts
    (dict(A=0), m.MRR_ERR_SHAPE),                            # A = 0 needs N*E = 0
    (dict(A=10, N=0, E=4), m.MRR_ERR_SHAPE),                 # N*E = 0 needs A = 0
    (dict(N=-1), m.MRR_ERR_SHAPE),
    (dict(sl=m.MRR_SCALE_F32_A, scale_cols=2), m.MRR_ERR_SHAPE),
    (dict(sl=m.MRR_SCALE_F32_AS, scale_cols=0), m.MRR_ERR_SHAPE),
    (dict(sl=m.MRR_SCALE_E8M0_AK2, scale_cols=3), m.MRR_ERR_SHAPE),
    (dict(expert_token_num_type=2), m.MRR_ERR_ATTR),
    (dict(idx_type=2), m.MRR_ERR_ATTR),
    (dict(idx_type=-1), m.MRR_ERR_ATTR),
])
def test_plan_rejects(lib, kw, code):
    assert plan(**kw) == code


def test_plan_valid_args_reach_the_device_query(lib):
    import torch

    st = plan()
    if torch.cuda.is_available():
        assert st == m.MRR_OK
    else:
        assert st == m.MRR_ERR_CUDA


def test_plan_null_out(lib):
    assert lib.mrr_v2_plan(16, 8, 0, 4, 4, 0, 0, 0, 0, 1, 0, 0, None) == m.MRR_ERR_NULL


# fake, never-dereferenced device addresses: every error below is found before any CUDA call
T, C, S, W, O1, O2, I, X, OW, WS = (0x10000 * k for k in range(1, 11))


def run(**kw):
    a = dict(tokens=T, dt=m.MRR_BF16, A=64, H=128, counts=C, count_is_i64=0, N=4, E=4, scales=S,
             sl=m.MRR_SCALE_F32_A, scale_cols=1, topk_w=W, permute_tokens=O1, permute_scales=O2,
             permute_token_idx=I, expert_token_num=X, permute_topk_w=OW,
             expert_token_num_type=1, idx_type=0, workspace=WS, workspace_bytes=1 << 20, stream=None)
    a.update(kw)
    return m.mrr_v2_run(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(permute_topk_w=None), m.MRR_ERR_TOPK_PAIR),
    (dict(topk_w=None), m.MRR_ERR_TOPK_PAIR),
    (dict(tokens=None), m.MRR_ERR_NULL),
    (dict(counts=None), m.MRR_ERR_NULL),
    (dict(permute_tokens=None), m.MRR_ERR_NULL),
    (dict(permute_token_idx=None), m.MRR_ERR_NULL),
    (dict(expert_token_num=None), m.MRR_ERR_NULL),
    (dict(scales=None), m.MRR_ERR_NULL),
    (dict(permute_scales=None), m.MRR_ERR_NULL),
    (dict(counts=C + 2), m.MRR_ERR_ALIGN),
    (dict(counts=C + 4, count_is_i64=1), m.MRR_ERR_ALIGN),
    (dict(permute_token_idx=I + 2), m.MRR_ERR_ALIGN),
    (dict(expert_token_num=X + 1), m.MRR_ERR_ALIGN),
    (dict(workspace=None), m.MRR_ERR_WORKSPACE),
    (dict(workspace=WS + 16), m.MRR_ERR_WORKSPACE),
    (dict(workspace_bytes=1024), m.MRR_ERR_WORKSPACE),
    (dict(workspace_bytes=4096), m.MRR_ERR_WORKSPACE),                # status, but no counter
    (dict(H=16384), m.MRR_ERR_SHAPE),
    (dict(expert_token_num_type=-1), m.MRR_ERR_ATTR),
    (dict(idx_type=3), m.MRR_ERR_ATTR),
    (dict(dt=42), m.MRR_ERR_DTYPE),
])
def test_run_rejects_before_any_cuda_call(lib, kw, code):
    assert run(**kw) == code


def test_run_without_scales_ignores_scale_pointers(lib):
    import torch

    st = run(scales=None, permute_scales=None, sl=m.MRR_SCALE_NONE)
    # valid arguments: reaches CUDA (no device here -> MRR_ERR_CUDA)
    if not torch.cuda.is_available():
        assert st == m.MRR_ERR_CUDA


def test_read_status_checks_arguments(lib):
    assert m.mrr_v2_read_status(None, 4096, None) == m.MRR_ERR_NULL
    assert m.mrr_v2_read_status(WS, 100, None) == m.MRR_ERR_WORKSPACE


def test_run_plan_rejects_null_plan(lib):
    assert lib.mrr_v2_run_plan(None, T, 0, C, None, None, O1, None, I, X, None, 1, WS, 4096,
                               None) == m.MRR_ERR_NULL


def test_plan_struct_layout_matches_header(tmp_path):
    """The binding's ctypes mirror of mrr_v2_plan_t has the C compiler's size and field offsets
    (a C program built against include/mrr_v2.h prints them)."""
    fields = [name for name, _ in m.mrr_v2_plan_t._fields_]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"mrr_v2.h\"\nint main(void) {\n"
                   + '  printf("size %zu\\n", sizeof(mrr_v2_plan_t));\n'
                   + "".join(f'  printf("{f} %zu\\n", offsetof(mrr_v2_plan_t, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", mbuild.INCLUDE, "-o", str(exe), str(src)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(m.mrr_v2_plan_t)
    for f in fields:
        assert int(got[f]) == getattr(m.mrr_v2_plan_t, f).offset, f


def test_cumsum_mode_passes_the_host_checks(lib):
    import torch

    st = plan(expert_token_num_type=0)
    assert st == (m.MRR_OK if torch.cuda.is_available() else m.MRR_ERR_CUDA)


def v1(**kw):
    a = dict(tokens=T, dt=m.MRR_I8, A=64, H=128, counts=C, count_is_i64=0, N=4, E=4,
             per_token_scales=S, permute_tokens=O1, permute_per_token_scales=O2,
             permute_token_idx=I, expert_token_num=X, expert_token_num_type=1, idx_type=0,
             workspace=WS, workspace_bytes=1 << 20, stream=None)
    a.update(kw)
    return m.mrr_v1_run(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(dt=m.MRR_F8E4M3FN), m.MRR_ERR_DTYPE),      # v1: float16, bfloat16, int8 only
    (dict(dt=m.MRR_F4E2M1), m.MRR_ERR_DTYPE),
    (dict(idx_type=1), m.MRR_ERR_UNSUPPORTED),       # v1: gather index only
    (dict(expert_token_num_type=0), m.MRR_ERR_UNSUPPORTED),
    (dict(idx_type=2), m.MRR_ERR_ATTR),
    (dict(permute_token_idx=None), m.MRR_ERR_NULL),
    (dict(H=0), m.MRR_ERR_SHAPE),
])
def test_v1_rejects(lib, kw, code):
    assert v1(**kw) == code


def gate(**kw):
    a = dict(x=T, dt=m.MRR_GATE_F16, T=16, e=384, k=6, bias=None, input_ids=None, tid2eid=None,
             n_vocab=0, additional_bias=None, additional_token_mask=None, k_group=1, group_count=1,
             routed_scaling_factor=1.0, eps=1e-20, group_select_mode=0, renorm=0, norm_type=1,
             y_out=O1, expert_idx=I, norm_out=None, workspace=WS, workspace_bytes=4096, stream=None)
    a.update(kw)
    return m.mrr_gating_topk_run(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(dt=7), m.MRR_ERR_DTYPE),
    (dict(renorm=1), m.MRR_ERR_ATTR),                       # the page: renorm supports 0 only
    (dict(norm_type=3), m.MRR_ERR_ATTR),
    (dict(group_select_mode=2), m.MRR_ERR_ATTR),
    (dict(input_ids=C), m.MRR_ERR_TOPK_PAIR),               # input_ids and tid2eid together
    (dict(k=65), m.MRR_ERR_SHAPE),                          # k <= 64
    (dict(k=0), m.MRR_ERR_SHAPE),
    (dict(e=2048), m.MRR_ERR_SHAPE),                        # this implementation: e <= 1024
    (dict(group_count=5), m.MRR_ERR_SHAPE),                 # e must divide into the groups
    (dict(group_count=4, k_group=5), m.MRR_ERR_SHAPE),
    (dict(group_count=64, k_group=1, k=7), m.MRR_ERR_SHAPE),  # k <= e / group_count * k_group
    (dict(group_count=384, group_select_mode=1), m.MRR_ERR_SHAPE),
    (dict(input_ids=C, tid2eid=S, n_vocab=0), m.MRR_ERR_SHAPE),
    (dict(x=None), m.MRR_ERR_NULL),
    (dict(expert_idx=None), m.MRR_ERR_NULL),
    (dict(workspace_bytes=100), m.MRR_ERR_WORKSPACE),
])
def test_gating_rejects(lib, kw, code):
    assert gate(**kw) == code


def run_multi(**kw):
    a = dict(src_tokens=T, src_scales=S, src_topk_w=W, src_rows=None, dt=m.MRR_BF16, A=64, H=128, counts=C,
             count_is_i64=0, N=4, E=4, sl=m.MRR_SCALE_F32_A, scale_cols=1, permute_tokens=O1,
             permute_scales=O2, permute_token_idx=I, expert_token_num=X, permute_topk_w=OW,
             expert_token_num_type=1, idx_type=0, workspace=WS, workspace_bytes=1 << 20, stream=None)
    a.update(kw)
    return m.mrr_v2_run_multi(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(src_tokens=None), m.MRR_ERR_NULL),
    (dict(src_topk_w=None), m.MRR_ERR_TOPK_PAIR),                  # output given, input table not
    (dict(permute_topk_w=None), m.MRR_ERR_TOPK_PAIR),
    (dict(src_scales=None), m.MRR_ERR_NULL),                       # scales layout without a table
    (dict(permute_scales=None), m.MRR_ERR_NULL),
    (dict(H=16384), m.MRR_ERR_SHAPE),
    (dict(A=10), m.MRR_ERR_SHAPE),                                 # N*E > A
    (dict(idx_type=3), m.MRR_ERR_ATTR),
    (dict(workspace=None), m.MRR_ERR_WORKSPACE),
    (dict(src_rows=WS + 4), m.MRR_ERR_ALIGN),                      # int64 table misaligned
])
def test_run_multi_host_errors(lib, kw, code):
    assert run_multi(**kw) == code


def test_run_plan_multi_refuses_the_inverse_direction(lib):
    plan = m.mrr_v2_plan_t()
    plan.A, plan.H, plan.N, plan.E, plan.row_bytes = 64, 128, 4, 4, 256
    plan.direction = 1
    st = m.mrr_v2_run_plan_multi(plan, T, None, None, None, m.MRR_BF16, C, O1, None, I, X, None, 1, WS,
                                 1 << 20, None)
    assert st in (m.MRR_ERR_PLAN, m.MRR_ERR_CUDA)


def test_push_host_refusals(lib):
    """mrr_v2_push's argument checks run on the host before anything is enqueued (no GPU needed):
    the addresses below are never dereferenced."""
    a = 1 << 20   # a 16-byte aligned stand-in address
    bf16 = m.DTYPE_CODES["bfloat16"]
    none = m.MRR_SCALE_NONE

    def push(**kw):
        args = dict(send_tokens=a, send_scales=None, send_topk_w=None, dt=bf16, S=16, H=8, send_counts=a,
                    count_is_i64=0, R=2, E=2, sl=none, scale_cols=0, dst_offsets=a, recv_src_offsets=None,
                    out_tokens=a, out_scales=None, out_topk_w=None, idx_out=None, out_rows=None, workspace=a,
                    workspace_bytes=4096, stream=None)
        args.update(kw)
        return m.mrr_v2_push(*args.values())

    assert push(R=64, E=65, S=8192) == m.MRR_ERR_SHAPE            # more than 4096 segments
    assert push(S=3) == m.MRR_ERR_SHAPE                           # fewer rows than segments
    assert push(H=16384) == m.MRR_ERR_SHAPE
    assert push(dt=99) == m.MRR_ERR_DTYPE
    assert push(workspace_bytes=1024) == m.MRR_ERR_WORKSPACE
    assert push(workspace=a + 8) == m.MRR_ERR_WORKSPACE
    assert push(out_tokens=None) == m.MRR_ERR_NULL
    assert push(send_counts=None) == m.MRR_ERR_NULL
    assert push(sl=m.MRR_SCALE_F32_A, scale_cols=1) == m.MRR_ERR_NULL   # a scale layout without scales
    assert push(idx_out=a) == m.MRR_ERR_NULL                       # an index without source offsets
    assert push(send_topk_w=a) == m.MRR_ERR_TOPK_PAIR
    assert push(send_counts=a + 2) == m.MRR_ERR_ALIGN
    assert push(dst_offsets=a + 4) == m.MRR_ERR_ALIGN
    assert m.mrr_status_str(m.MRR_ERR_DEST).startswith("MRR_ERR_DEST")
