"""Thin ctypes binding of the C ABI in include/mrr_v2.h (argument marshalling only).

The functions keep the C names.  ``moe_re_routing`` is the torch-level convenience call with
the signature of the pages' PyTorch API (``cann_ops_transformer.moe_re_routing``, section
PyTorch API 调用单算子模式 of the "CANN ops-transformer MoeReRoutingV2" article): it
allocates the five outputs and the workspace with torch and runs the op through
``mrr_v2_run``.  Every step of the op runs in the CUDA library; there is no other code path,
and loading fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

from . import build as _build

# ---------------------------------------------------------------------------- constants (mrr_v2.h)

MRR_OK = 0
MRR_ERR_NULL = 1
MRR_ERR_SHAPE = 2
MRR_ERR_DTYPE = 3
MRR_ERR_ATTR = 4
MRR_ERR_UNSUPPORTED = 5
MRR_ERR_TOPK_PAIR = 6
MRR_ERR_WORKSPACE = 7
MRR_ERR_CUDA = 8
MRR_ERR_ALIGN = 9
MRR_ERR_PLAN = 10
MRR_ERR_COUNT_NONPOS = 16
MRR_ERR_COUNT_SUM = 17
MRR_ERR_TIMEOUT = 18
MRR_ERR_INDEX = 19
MRR_ERR_SOURCE = 20
MRR_ERR_DEST = 21
MRR_GATE_F16, MRR_GATE_BF16, MRR_GATE_F32 = 0, 1, 2
MRR_NOALLOC_MAX_SEGMENTS = 16384
MRR_NOALLOC_SCRATCH_BYTES = 137984

MRR_F16, MRR_BF16, MRR_I8, MRR_F8E5M2, MRR_F8E4M3FN, MRR_HIF8, MRR_F4E2M1, MRR_F4E1M2 = range(8)
MRR_SCALE_NONE, MRR_SCALE_F32_A, MRR_SCALE_F32_AS, MRR_SCALE_E8M0_AK2 = range(4)
MRR_PATH_AUTO, MRR_PATH_BULK, MRR_PATH_VECTOR = 0, 1, 2
MRR_HINT_LOAD_EVICT_FIRST, MRR_HINT_STORE_EVICT_FIRST = 1, 2

DTYPE_CODES = {
    "float16": MRR_F16, "bfloat16": MRR_BF16, "int8": MRR_I8, "float8_e5m2": MRR_F8E5M2,
    "float8_e4m3fn": MRR_F8E4M3FN, "hifloat8": MRR_HIF8, "float4_e2m1": MRR_F4E2M1,
    "float4_e1m2": MRR_F4E1M2,
}
SCALE_CODES = {"none": MRR_SCALE_NONE, "f32_a": MRR_SCALE_F32_A, "f32_as": MRR_SCALE_F32_AS,
               "e8m0": MRR_SCALE_E8M0_AK2}


class MrrError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        super().__init__(f"{where}: {mrr_status_str(code)}" if where else mrr_status_str(code))
        self.code = code


class mrr_v2_plan_t(ctypes.Structure):
    _fields_ = [
        ("A", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64), ("E", ctypes.c_int64),
        ("row_bytes", ctypes.c_int64), ("scale_row_bytes", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("count_is_i64", ctypes.c_int32), ("scale_layout", ctypes.c_int32),
        ("has_topk", ctypes.c_int32), ("idx_type", ctypes.c_int32),
        ("fuse_scan", ctypes.c_int32), ("path", ctypes.c_int32), ("grid", ctypes.c_int32),
        ("block", ctypes.c_int32), ("chunk_bytes", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("hints", ctypes.c_int32), ("sched", ctypes.c_int32), ("static_chunks", ctypes.c_int32),
        ("pdl", ctypes.c_int32), ("direction", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("prefetch_chunks", ctypes.c_int32), ("epoch", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


# ---------------------------------------------------------------------------- loading

_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libmrr_v2.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -m moe_expert_token_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.mrr_status_str.restype = ctypes.c_char_p
    lib.mrr_status_str.argtypes = [I32]
    lib.mrr_v2_plan.restype = I32
    lib.mrr_v2_plan.argtypes = [I64, I64, I32, I64, I64, I32, I32, I64, I32, I64, I64, I32,
                                ctypes.POINTER(mrr_v2_plan_t)]
    lib.mrr_v2_run.restype = I32
    lib.mrr_v2_run.argtypes = [P, I32, I64, I64, P, I32, I64, I64, P, I32, I64, P,
                               P, P, P, P, P, I64, I64, P, ctypes.c_size_t, P]
    lib.mrr_v2_run_plan.restype = I32
    lib.mrr_v2_run_plan.argtypes = [ctypes.POINTER(mrr_v2_plan_t), P, I32, P, P, P,
                                    P, P, P, P, P, I64, P, ctypes.c_size_t, P]
    lib.mrr_v2_read_status.restype = I32
    lib.mrr_v2_read_status.argtypes = [P, ctypes.c_size_t, P]
    lib.mrr_v2_unroute_plan.restype = I32
    lib.mrr_v2_unroute_plan.argtypes = [I64, I64, I32, I64, I64, I32, I32, I64, I32, I32,
                                        ctypes.POINTER(mrr_v2_plan_t)]
    lib.mrr_v2_unroute.restype = I32
    lib.mrr_v2_unroute.argtypes = [P, I32, I64, I64, P, I32, I64, I64, P, I32, I64, P, P, P, P, P,
                                   ctypes.c_size_t, P]
    lib.mrr_v1_run.restype = I32
    lib.mrr_v1_run.argtypes = [P, I32, I64, I64, P, I32, I64, I64, P, P, P, P, P, I64, I64, P,
                               ctypes.c_size_t, P]
    lib.mrr_gating_topk_run.restype = I32
    lib.mrr_gating_topk_run.argtypes = [P, I32, I64, I64, I64, P, P, P, I64, P, P, I64, I64,
                                        ctypes.c_float, ctypes.c_float, I64, I64, I64, P, P, P, P,
                                        ctypes.c_size_t, P]
    lib.mrr_v2_run_multi.restype = I32
    lib.mrr_v2_run_multi.argtypes = [P, P, P, P, I32, I64, I64, P, I32, I64, I64, I32, I64,
                                     P, P, P, P, P, I64, I64, P, ctypes.c_size_t, P]
    lib.mrr_v2_run_plan_multi.restype = I32
    lib.mrr_v2_run_plan_multi.argtypes = [ctypes.POINTER(mrr_v2_plan_t), P, P, P, P, I32, P,
                                          P, P, P, P, P, I64, P, ctypes.c_size_t, P]
    lib.mrr_v2_offsets_host.restype = I32
    lib.mrr_v2_offsets_host.argtypes = [P, I32, I64, I64, I64, P, P, P]
    lib.mrr_v2_push.restype = I32
    lib.mrr_v2_push.argtypes = [P, P, P, I32, I64, I64, P, I32, I64, I64, I32, I64, P, P, P, P, P, P, P,
                                P, ctypes.c_size_t, P]
    lib.mrr_v2_run_noalloc.restype = I32
    lib.mrr_v2_run_noalloc.argtypes = [P, I32, I64, I64, P, I32, I64, I64, P, I32, I64, P,
                                       P, P, P, P, P, I64, I64, I32, P]
    if path == _build.LIB_PATH:
        _lib = lib
    return lib


def header_functions() -> list:
    """Names of the functions the headers in include/ declare."""
    names = set()
    for h in sorted(os.listdir(_build.INCLUDE)):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(_build.INCLUDE, h), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s*(mrr_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


# ---------------------------------------------------------------------------- C functions, same names

def mrr_status_str(code: int) -> str:
    return load_library().mrr_status_str(int(code)).decode()


def mrr_v2_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, has_topk,
                expert_token_num_type=1, idx_type=0, device=0) -> Tuple[int, mrr_v2_plan_t]:
    plan = mrr_v2_plan_t()
    st = load_library().mrr_v2_plan(A, H, dt, N, E, int(count_is_i64), sl, scale_cols,
                                    int(has_topk), expert_token_num_type, idx_type, device,
                                    ctypes.byref(plan))
    return st, plan


def mrr_v2_run(tokens, dt, A, H, counts, count_is_i64, N, E, scales, sl, scale_cols, topk_w,
               permute_tokens, permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
               expert_token_num_type, idx_type, workspace, workspace_bytes, stream) -> int:
    """All buffers are integer device addresses (or None); stream is a cudaStream_t value."""
    return load_library().mrr_v2_run(
        tokens, dt, A, H, counts, int(count_is_i64), N, E, scales, sl, scale_cols, topk_w,
        permute_tokens, permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
        expert_token_num_type, idx_type, workspace, workspace_bytes, stream)


def mrr_v2_run_plan(plan: mrr_v2_plan_t, tokens, dt, counts, scales, topk_w, permute_tokens,
                    permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
                    expert_token_num_type, workspace, workspace_bytes, stream) -> int:
    return load_library().mrr_v2_run_plan(
        ctypes.byref(plan), tokens, dt, counts, scales, topk_w, permute_tokens, permute_scales,
        permute_token_idx, expert_token_num, permute_topk_w, expert_token_num_type, workspace,
        workspace_bytes, stream)


def mrr_v1_run(tokens, dt, A, H, counts, count_is_i64, N, E, per_token_scales, permute_tokens,
               permute_per_token_scales, permute_token_idx, expert_token_num, expert_token_num_type,
               idx_type, workspace, workspace_bytes, stream) -> int:
    """The v1 op (float16/bfloat16/int8 tokens, [A] fp32 scales, count mode, gather index)."""
    return load_library().mrr_v1_run(
        tokens, dt, A, H, counts, int(count_is_i64), N, E, per_token_scales, permute_tokens,
        permute_per_token_scales, permute_token_idx, expert_token_num, expert_token_num_type,
        idx_type, workspace, workspace_bytes, stream)


def mrr_v2_unroute_plan(A, H, dt, N, E, count_is_i64, sl, scale_cols, has_topk,
                        device=0) -> Tuple[int, mrr_v2_plan_t]:
    plan = mrr_v2_plan_t()
    st = load_library().mrr_v2_unroute_plan(A, H, dt, N, E, int(count_is_i64), sl, scale_cols,
                                            int(has_topk), device, ctypes.byref(plan))
    return st, plan


def mrr_v2_unroute(permute_tokens, dt, A, H, counts, count_is_i64, N, E, permute_scales, sl,
                   scale_cols, permute_topk_w, tokens, scales, topk_w, workspace, workspace_bytes,
                   stream) -> int:
    """The inverse move (expert-major rows back to rank-major order); integer device addresses."""
    return load_library().mrr_v2_unroute(
        permute_tokens, dt, A, H, counts, int(count_is_i64), N, E, permute_scales, sl, scale_cols,
        permute_topk_w, tokens, scales, topk_w, workspace, workspace_bytes, stream)


def mrr_v2_run_multi(src_tokens, src_scales, src_topk_w, src_rows, dt, A, H, counts, count_is_i64,
                     N, E, sl, scale_cols, permute_tokens, permute_scales, permute_token_idx,
                     expert_token_num, permute_topk_w, expert_token_num_type, idx_type, workspace,
                     workspace_bytes, stream) -> int:
    """The multi-source form: src_tokens / src_scales / src_topk_w / src_rows are device
    addresses of [N] tables (pointers, pointers, pointers, int64 rows), or None."""
    return load_library().mrr_v2_run_multi(
        src_tokens, src_scales, src_topk_w, src_rows, dt, A, H, counts, int(count_is_i64), N, E, sl,
        scale_cols, permute_tokens, permute_scales, permute_token_idx, expert_token_num,
        permute_topk_w, expert_token_num_type, idx_type, workspace, workspace_bytes, stream)


def mrr_v2_run_plan_multi(plan: mrr_v2_plan_t, src_tokens, src_scales, src_topk_w, src_rows, dt,
                          counts, permute_tokens, permute_scales, permute_token_idx,
                          expert_token_num, permute_topk_w, expert_token_num_type, workspace,
                          workspace_bytes, stream) -> int:
    return load_library().mrr_v2_run_plan_multi(
        ctypes.byref(plan), src_tokens, src_scales, src_topk_w, src_rows, dt, counts,
        permute_tokens, permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
        expert_token_num_type, workspace, workspace_bytes, stream)


def mrr_v2_offsets_host(counts, count_is_i64, N, E, A, src_offset, dst_offset, expert_token_num) -> int:
    """Host addresses: counts [N, E] (int32 / int64), int64 outputs [N, E], [N, E], [E] or None."""
    return load_library().mrr_v2_offsets_host(counts, int(count_is_i64), N, E, A, src_offset, dst_offset,
                                              expert_token_num)


def mrr_v2_push(send_tokens, send_scales, send_topk_w, dt, S, H, send_counts, count_is_i64, R, E, sl,
                scale_cols, dst_offsets, recv_src_offsets, out_tokens, out_scales, out_topk_w, idx_out,
                out_rows, workspace, workspace_bytes, stream) -> int:
    """The push form, one sender's side; out_tokens / out_scales / out_topk_w / idx_out / out_rows are
    device addresses of [R] tables (pointers, or int64 rows), or None."""
    return load_library().mrr_v2_push(
        send_tokens, send_scales, send_topk_w, dt, S, H, send_counts, int(count_is_i64), R, E, sl,
        scale_cols, dst_offsets, recv_src_offsets, out_tokens, out_scales, out_topk_w, idx_out, out_rows,
        workspace, workspace_bytes, stream)


def mrr_v2_read_status(workspace, workspace_bytes, stream) -> int:
    return load_library().mrr_v2_read_status(workspace, workspace_bytes, stream)


def mrr_v2_run_noalloc(tokens, dt, A, H, counts, count_is_i64, N, E, scales, sl, scale_cols, topk_w,
                       permute_tokens, permute_scales, permute_token_idx, expert_token_num,
                       permute_topk_w, expert_token_num_type, idx_type, wait_and_check,
                       stream) -> int:
    """mrr_v2_run without a workspace, for callers that cannot allocate device memory: the
    library's own fixed device array serves as scratch (see include/mrr_v2.h)."""
    return load_library().mrr_v2_run_noalloc(
        tokens, dt, A, H, counts, int(count_is_i64), N, E, scales, sl, scale_cols, topk_w,
        permute_tokens, permute_scales, permute_token_idx, expert_token_num, permute_topk_w,
        expert_token_num_type, idx_type, int(wait_and_check), stream)


# ---------------------------------------------------------------------------- torch-level call

def _torch_token_code(t, tokens_dtype: Optional[str]):
    """(dtype code, H) for a tokens tensor; FP4 payloads hold two elements per byte."""
    import torch

    names = {torch.float16: "float16", torch.bfloat16: "bfloat16", torch.int8: "int8",
             torch.float8_e5m2: "float8_e5m2", torch.float8_e4m3fn: "float8_e4m3fn"}
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    if tokens_dtype is not None:
        name = {"float4_e2m1fn_x2": "float4_e2m1", "float4_e1m2fn_x2": "float4_e1m2"}.get(
            tokens_dtype, tokens_dtype)
        if t.element_size() != 1 and name not in ("float16", "bfloat16"):
            raise TypeError("tokens_dtype names a 1-byte or packed type but tokens are wider")
    elif fp4 is not None and t.dtype == fp4:
        name = "float4_e2m1"
    elif t.dtype in names:
        name = names[t.dtype]
    else:
        raise TypeError(f"unsupported tokens dtype {t.dtype}; pass tokens_dtype for uint8 storage")
    code = DTYPE_CODES[name]
    H = t.shape[-1] * (2 if code in (MRR_F4E2M1, MRR_F4E1M2) else 1)
    return code, H


def _scale_layout(s):
    import torch

    if s is None:
        return MRR_SCALE_NONE, 0
    if s.dtype == torch.float32 and s.dim() == 1:
        return MRR_SCALE_F32_A, 1
    if s.dtype == torch.float32 and s.dim() == 2:
        return MRR_SCALE_F32_AS, s.shape[1]
    if s.element_size() == 1 and s.dim() == 3 and s.shape[2] == 2:
        return MRR_SCALE_E8M0_AK2, s.shape[1] * 2
    raise TypeError("per_token_scales must be [A] / [A,S] float32 or [A, K/64, 2] e8m0 bytes")


def moe_re_routing(tokens, expert_token_num_per_rank, *, per_token_scales=None,
                   expert_topk_weight=None, expert_token_num_type: int = 1, idx_type: int = 0,
                   tokens_dtype: Optional[str] = None, workspace=None, stream=None,
                   check_status: bool = False):
    """Re-route rank-major tokens to expert-major order on the GPU.

    Returns (permute_tokens, permute_per_token_scales, permute_token_idx, expert_token_num,
    permute_topk_weight) with the shapes of the pages' InferShape rules: absent scales give an
    unwritten [A] float32 tensor, absent top-k weights an empty (0,) tensor.
    ``check_status=True`` synchronises and raises on a device-detected count error.
    """
    import torch

    t, c = tokens, expert_token_num_per_rank
    if t.dim() != 2 or c.dim() != 2:
        raise ValueError("tokens and expert_token_num_per_rank must be 2-D")
    if not t.is_cuda:
        raise ValueError("tokens must be a CUDA tensor")
    if c.dtype not in (torch.int32, torch.int64):
        raise TypeError("expert_token_num_per_rank must be int32 or int64")
    dev = t.device
    code, H = _torch_token_code(t, tokens_dtype)
    A = t.shape[0]
    N, E = c.shape
    sl, scale_cols = _scale_layout(per_token_scales)
    for x in (c, per_token_scales, expert_topk_weight):
        if x is not None and (x.device != dev or not x.is_contiguous()):
            raise ValueError("all tensors must be contiguous and on the tokens' device")
    if not t.is_contiguous():
        raise ValueError("tokens must be contiguous")
    if expert_topk_weight is not None and (expert_topk_weight.dtype != torch.float32
                                           or expert_topk_weight.shape != (A, 1)):
        raise ValueError("expert_topk_weight must be float32 [A, 1]")

    st, plan = mrr_v2_plan(A, H, code, N, E, c.dtype == torch.int64, sl, scale_cols,
                           expert_topk_weight is not None, expert_token_num_type, idx_type,
                           dev.index if dev.index is not None else torch.cuda.current_device())
    if st != MRR_OK:
        raise MrrError(st, "mrr_v2_plan")

    out_tok = torch.empty_like(t)
    out_sc = (torch.empty_like(per_token_scales) if per_token_scales is not None
              else torch.empty(A, dtype=torch.float32, device=dev))
    idx = torch.empty(A, dtype=torch.int32, device=dev)
    etn = torch.empty(E, dtype=c.dtype, device=dev)
    out_tw = (torch.empty_like(expert_topk_weight) if expert_topk_weight is not None
              else torch.empty(0, dtype=torch.float32, device=dev))
    if workspace is None or workspace.numel() < plan.workspace_bytes:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)

    def ptr(x):
        return None if x is None else x.data_ptr()

    with torch.cuda.device(dev):
        st = mrr_v2_run(ptr(t), code, A, H, ptr(c), c.dtype == torch.int64, N, E,
                        ptr(per_token_scales), sl, scale_cols, ptr(expert_topk_weight),
                        ptr(out_tok), ptr(out_sc) if per_token_scales is not None else None,
                        ptr(idx), ptr(etn),
                        ptr(out_tw) if expert_topk_weight is not None else None,
                        expert_token_num_type, idx_type, workspace.data_ptr(),
                        workspace.numel(), stream.cuda_stream)
        if st != MRR_OK:
            raise MrrError(st, "mrr_v2_run")
        if check_status:
            st = mrr_v2_read_status(workspace.data_ptr(), workspace.numel(), stream.cuda_stream)
            if st != MRR_OK:
                raise MrrError(st, "device")
    return out_tok, out_sc, idx, etn, out_tw


def moe_re_routing_multi(tokens_per_rank, expert_token_num_per_rank, *, per_token_scales=None,
                         expert_topk_weight=None, expert_token_num_type: int = 1, idx_type: int = 0,
                         tokens_dtype: Optional[str] = None, workspace=None, stream=None,
                         check_status: bool = False):
    """``moe_re_routing`` with the received rows still in one tensor per source rank.

    ``tokens_per_rank[i]`` is a [rows_i, H] tensor holding rank i's rows (the rows row i of the
    count matrix describes), and so are the optional per-rank lists ``per_token_scales`` and
    ``expert_topk_weight`` ([rows_i, 1] float32).  The outputs equal ``moe_re_routing`` on the
    concatenation of the lists; each rank's capacity (rows_i) is passed along, so counts that do
    not fit a rank's tensor raise instead of reading past it (with ``check_status=True``)."""
    import torch

    ts, c = list(tokens_per_rank), expert_token_num_per_rank
    if c.dim() != 2 or len(ts) != c.shape[0]:
        raise ValueError("one tokens tensor per row of expert_token_num_per_rank")
    if c.dtype not in (torch.int32, torch.int64):
        raise TypeError("expert_token_num_per_rank must be int32 or int64")
    dev = c.device
    N, E = c.shape
    code, H = _torch_token_code(ts[0], tokens_dtype)
    lists = [ts, per_token_scales, expert_topk_weight]
    if any(lst is not None and len(lst) != N for lst in lists):
        raise ValueError("every per-rank list needs one tensor per rank")
    for i, t in enumerate(ts):
        if t.dim() != 2 or t.dtype != ts[0].dtype or _torch_token_code(t, tokens_dtype)[1] != H:
            raise ValueError("per-rank token tensors must be [rows_i, H] of one dtype")
        if not t.is_cuda or t.device != dev or not t.is_contiguous():
            raise ValueError("per-rank tensors must be contiguous CUDA tensors on the counts' device")
        for lst in lists[1:]:
            if lst is not None and (lst[i].shape[0] != t.shape[0] or lst[i].device != dev
                                    or not lst[i].is_contiguous()):
                raise ValueError("rank %d: scales / top-k weights must match its token rows" % i)
    A = sum(int(t.shape[0]) for t in ts)
    sl, scale_cols = _scale_layout(None if per_token_scales is None else per_token_scales[0])
    if per_token_scales is not None and any(_scale_layout(x) != (sl, scale_cols) for x in per_token_scales):
        raise ValueError("per-rank scales must share one layout")
    if expert_topk_weight is not None and any(x.dtype != torch.float32 or x.dim() != 2 or x.shape[1] != 1
                                              for x in expert_topk_weight):
        raise ValueError("expert_topk_weight entries must be float32 [rows_i, 1]")

    st, plan = mrr_v2_plan(A, H, code, N, E, c.dtype == torch.int64, sl, scale_cols,
                           expert_topk_weight is not None, expert_token_num_type, idx_type,
                           dev.index if dev.index is not None else torch.cuda.current_device())
    if st != MRR_OK:
        raise MrrError(st, "mrr_v2_plan")

    if stream is None:
        stream = torch.cuda.current_stream(dev)

    def table(lst):   # a device array of the tensors' addresses, uploaded on the op's stream
        if lst is None:
            return None
        return torch.tensor([x.data_ptr() for x in lst], dtype=torch.int64, device=dev)

    with torch.cuda.device(dev), torch.cuda.stream(stream):
        t_tok, t_sc, t_tw = table(ts), table(per_token_scales), table(expert_topk_weight)
        rows = torch.tensor([int(t.shape[0]) for t in ts], dtype=torch.int64, device=dev)
    out_tok = torch.empty((A,) + tuple(ts[0].shape[1:]), dtype=ts[0].dtype, device=dev)
    out_sc = (torch.empty((A,) + tuple(per_token_scales[0].shape[1:]), dtype=per_token_scales[0].dtype,
                          device=dev)
              if per_token_scales is not None else torch.empty(A, dtype=torch.float32, device=dev))
    idx = torch.empty(A, dtype=torch.int32, device=dev)
    etn = torch.empty(E, dtype=c.dtype, device=dev)
    out_tw = (torch.empty(A, 1, dtype=torch.float32, device=dev) if expert_topk_weight is not None
              else torch.empty(0, dtype=torch.float32, device=dev))
    if workspace is None or workspace.numel() < plan.workspace_bytes:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)

    def ptr(x):
        return None if x is None else x.data_ptr()

    with torch.cuda.device(dev):
        st = mrr_v2_run_multi(ptr(t_tok), ptr(t_sc), ptr(t_tw), ptr(rows), code, A, H, ptr(c),
                              c.dtype == torch.int64, N, E, sl, scale_cols, ptr(out_tok),
                              ptr(out_sc) if per_token_scales is not None else None, ptr(idx), ptr(etn),
                              ptr(out_tw) if expert_topk_weight is not None else None,
                              expert_token_num_type, idx_type, workspace.data_ptr(), workspace.numel(),
                              stream.cuda_stream)
        if st != MRR_OK:
            raise MrrError(st, "mrr_v2_run_multi")
        # the tables must outlive the enqueued work: keep them with the stream's pending work
        for x in (t_tok, t_sc, t_tw, rows):
            if x is not None:
                x.record_stream(stream)
        if check_status:
            st = mrr_v2_read_status(workspace.data_ptr(), workspace.numel(), stream.cuda_stream)
            if st != MRR_OK:
                raise MrrError(st, "device")
    return out_tok, out_sc, idx, etn, out_tw


def moe_re_routing_inverse(permute_tokens, expert_token_num_per_rank, *,
                           permute_per_token_scales=None, permute_topk_weight=None,
                           tokens_dtype: Optional[str] = None, workspace=None, stream=None,
                           check_status: bool = False):
    """Move expert-major rows back to the rank-major order they arrived in (the combine side).

    ``expert_token_num_per_rank`` is the same count matrix the forward move used.  Returns
    (tokens, per_token_scales, topk_weight); the last two are None when not given.
    """
    import torch

    t, c = permute_tokens, expert_token_num_per_rank
    if t.dim() != 2 or c.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("permute_tokens must be a contiguous 2-D CUDA tensor, counts 2-D")
    if c.dtype not in (torch.int32, torch.int64):
        raise TypeError("expert_token_num_per_rank must be int32 or int64")
    dev = t.device
    code, H = _torch_token_code(t, tokens_dtype)
    A = t.shape[0]
    N, E = c.shape
    sl, scale_cols = _scale_layout(permute_per_token_scales)
    for x in (c, permute_per_token_scales, permute_topk_weight):
        if x is not None and (x.device != dev or not x.is_contiguous()):
            raise ValueError("all tensors must be contiguous and on the tokens' device")
    st, plan = mrr_v2_unroute_plan(A, H, code, N, E, c.dtype == torch.int64, sl, scale_cols,
                                   permute_topk_weight is not None,
                                   dev.index if dev.index is not None else torch.cuda.current_device())
    if st != MRR_OK:
        raise MrrError(st, "mrr_v2_unroute_plan")
    out_tok = torch.empty_like(t)
    out_sc = None if permute_per_token_scales is None else torch.empty_like(permute_per_token_scales)
    out_tw = None if permute_topk_weight is None else torch.empty_like(permute_topk_weight)
    if workspace is None or workspace.numel() < plan.workspace_bytes:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)

    def ptr(x):
        return None if x is None else x.data_ptr()

    with torch.cuda.device(dev):
        st = mrr_v2_unroute(ptr(t), code, A, H, ptr(c), c.dtype == torch.int64, N, E,
                            ptr(permute_per_token_scales), sl, scale_cols, ptr(permute_topk_weight),
                            ptr(out_tok), ptr(out_sc), ptr(out_tw), workspace.data_ptr(),
                            workspace.numel(), stream.cuda_stream)
        if st != MRR_OK:
            raise MrrError(st, "mrr_v2_unroute")
        if check_status:
            st = mrr_v2_read_status(workspace.data_ptr(), workspace.numel(), stream.cuda_stream)
            if st != MRR_OK:
                raise MrrError(st, "device")
    return out_tok, out_sc, out_tw


def moe_re_routing_v1(tokens, expert_token_num_per_rank, *, per_token_scales=None,
                      expert_token_num_type: int = 1, idx_type: int = 0, workspace=None,
                      stream=None, check_status: bool = False):
    """The v1 call (torch_npu.npu_moe_re_routing): float16/bfloat16/int8 tokens, optional [A]
    float32 scales, count mode and a gather index only; returns (permute_tokens,
    permute_per_token_scales, permute_token_idx, expert_token_num)."""
    import torch

    t, c = tokens, expert_token_num_per_rank
    if t.dim() != 2 or c.dim() != 2 or not t.is_cuda or not t.is_contiguous():
        raise ValueError("tokens must be a contiguous 2-D CUDA tensor, counts 2-D")
    codes = {torch.float16: MRR_F16, torch.bfloat16: MRR_BF16, torch.int8: MRR_I8}
    if t.dtype not in codes:
        raise TypeError("v1 supports float16, bfloat16 and int8 tokens")
    if per_token_scales is not None and (per_token_scales.dtype != torch.float32 or per_token_scales.dim() != 1):
        raise TypeError("v1 per_token_scales are [A] float32")
    dev = t.device
    A, H = t.shape
    N, E = c.shape
    st, plan = mrr_v2_plan(A, H, codes[t.dtype], N, E, c.dtype == torch.int64,
                           MRR_SCALE_F32_A if per_token_scales is not None else MRR_SCALE_NONE,
                           1 if per_token_scales is not None else 0, False, 1, 0,
                           dev.index if dev.index is not None else torch.cuda.current_device())
    if st != MRR_OK:
        raise MrrError(st, "mrr_v2_plan")
    out_tok = torch.empty_like(t)
    out_sc = torch.empty(A, dtype=torch.float32, device=dev)
    idx = torch.empty(A, dtype=torch.int32, device=dev)
    etn = torch.empty(E, dtype=c.dtype, device=dev)
    if workspace is None or workspace.numel() < plan.workspace_bytes:
        workspace = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        st = mrr_v1_run(t.data_ptr(), codes[t.dtype], A, H, c.data_ptr(), c.dtype == torch.int64, N, E,
                        None if per_token_scales is None else per_token_scales.data_ptr(),
                        out_tok.data_ptr(), out_sc.data_ptr(), idx.data_ptr(), etn.data_ptr(),
                        expert_token_num_type, idx_type, workspace.data_ptr(), workspace.numel(),
                        stream.cuda_stream)
        if st != MRR_OK:
            raise MrrError(st, "mrr_v1_run")
        if check_status:
            st = mrr_v2_read_status(workspace.data_ptr(), workspace.numel(), stream.cuda_stream)
            if st != MRR_OK:
                raise MrrError(st, "device")
    return out_tok, out_sc, idx, etn


def mrr_gating_topk_run(x, dt, T, e, k, bias, input_ids, tid2eid, n_vocab, additional_bias,
                        additional_token_mask, k_group, group_count, routed_scaling_factor, eps,
                        group_select_mode, renorm, norm_type, y_out, expert_idx, norm_out,
                        workspace, workspace_bytes, stream) -> int:
    """MoE gating top-k (include/mrr_gating.h); integer device addresses or None."""
    return load_library().mrr_gating_topk_run(
        x, dt, T, e, k, bias, input_ids, tid2eid, n_vocab, additional_bias, additional_token_mask,
        k_group, group_count, routed_scaling_factor, eps, group_select_mode, renorm, norm_type,
        y_out, expert_idx, norm_out, workspace, workspace_bytes, stream)


def moe_gating_top_k(x, k: int, *, bias=None, input_ids=None, tid2eid=None, additional_bias=None,
                     additional_token_mask=None, k_group: int = 1, group_count: int = 1,
                     routed_scaling_factor: float = 1.0, eps: float = 1e-20,
                     group_select_mode: int = 0, renorm: int = 0, norm_type: int = 0,
                     out_flag: bool = False, workspace=None, stream=None, check_status: bool = False):
    """The torch-level call of the gating op, with the page's signature (npu_moe_gating_top_k):
    returns (y, expert_idx, out); out is the float32 normalised scores when out_flag, else None.
    x may be [T, e] or [b, s, e]; outputs keep the leading dimensions."""
    import torch

    if not x.is_cuda or not x.is_contiguous() or x.dim() not in (2, 3):
        raise ValueError("x must be a contiguous 2-D or 3-D CUDA tensor")
    codes = {torch.float16: MRR_GATE_F16, torch.bfloat16: MRR_GATE_BF16, torch.float32: MRR_GATE_F32}
    if x.dtype not in codes:
        raise TypeError("x must be float16, bfloat16 or float32")
    lead = tuple(x.shape[:-1])
    e = x.shape[-1]
    T = 1
    for d in lead:
        T *= d
    dev = x.device
    for b in (bias, additional_bias):
        if b is not None and (b.dtype != x.dtype or b.numel() != e or b.device != dev):
            raise ValueError("bias / additional_bias must be [e] in x's dtype on x's device")
    mask = None
    if additional_token_mask is not None:
        if additional_token_mask.dtype != torch.bool or additional_token_mask.numel() != T:
            raise ValueError("additional_token_mask must be [T] bool")
        mask = additional_token_mask.contiguous().view(torch.uint8)
    ids = None if input_ids is None else input_ids.to(torch.int64).contiguous()
    tab = None if tid2eid is None else tid2eid.to(torch.int32).contiguous()
    y = torch.empty(*lead, k, dtype=x.dtype, device=dev)
    idx = torch.empty(*lead, k, dtype=torch.int32, device=dev)
    out = torch.empty(*lead, e, dtype=torch.float32, device=dev) if out_flag else None
    if workspace is None:
        workspace = torch.empty(4096, dtype=torch.uint8, device=dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)

    def ptr(t):
        return None if t is None else t.data_ptr()

    with torch.cuda.device(dev):
        st = mrr_gating_topk_run(ptr(x), codes[x.dtype], T, e, k, ptr(bias), ptr(ids), ptr(tab),
                                 0 if tab is None else tab.shape[0], ptr(additional_bias), ptr(mask),
                                 k_group, group_count, routed_scaling_factor, eps, group_select_mode,
                                 renorm, norm_type, ptr(y), ptr(idx), ptr(out), workspace.data_ptr(),
                                 workspace.numel(), stream.cuda_stream)
        if st != MRR_OK:
            raise MrrError(st, "mrr_gating_topk_run")
        if check_status:
            st = mrr_v2_read_status(workspace.data_ptr(), workspace.numel(), stream.cuda_stream)
            if st != MRR_OK:
                raise MrrError(st, "device")
    return y, idx, out
