"""CPU oracle for the MoeReRoutingV2 re-routing step -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library and its Python binding never import it, and it
imports nothing from them.

``mrr_oracle.c`` is the definition of the op written as the nested loops of the
"CANN ops-transformer MoeReRoutingV2" article (m.nlpx.cn/news/59074), section 计算公式;
this module only builds it with gcc and marshals numpy arrays into it.

Every function here is pinned by tests/test_oracle_pins.py (worked example, brute-force
stable sort, transpose closed form, identity cases, invariants, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mrr_oracle.c")
LIB = os.path.join(_HERE, "_build", "liboracle.so")

ORC_OK, ORC_ERR_ARG, ORC_ERR_COUNT_NONPOS, ORC_ERR_COUNT_SUM = 0, 1, 2, 3


class OracleError(RuntimeError):
    def __init__(self, code: int):
        names = {1: "bad argument", 2: "a count is <= 0", 3: "counts do not sum to A"}
        super().__init__(f"oracle rejected the input: {names.get(code, code)}")
        self.code = code


def build(source: str = SOURCE, out: str = LIB, extra_flags=()) -> str:
    """Compile the oracle with gcc into a shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", *extra_flags, "-o", out, source]
    subprocess.run(cmd, check=True)
    return out


_lib = None


def _built_for_this_host(path: str) -> bool:
    import platform
    import struct

    with open(path, "rb") as f:
        head = f.read(20)
    want = {"x86_64": 62, "aarch64": 183}.get(platform.machine())
    return (len(head) == 20 and head[:4] == b"\x7fELF"
            and (want is None or struct.unpack_from("<H", head, 18)[0] == want))


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.mrr_oracle_run.restype = ctypes.c_int
    lib.mrr_oracle_run.argtypes = [P, I64, I64, P, ctypes.c_int, I64, I64, P, I64, P,
                                   P, P, P, P, P, I64]
    lib.mrr_oracle_validate.restype = ctypes.c_int
    lib.mrr_oracle_validate.argtypes = [P, ctypes.c_int, I64, I64, I64]
    lib.mrr_oracle_offsets.restype = None
    lib.mrr_oracle_offsets.argtypes = [P, ctypes.c_int, I64, I64, P, P]
    lib.mrr_oracle_expert_token_num.restype = ctypes.c_int
    lib.mrr_oracle_expert_token_num.argtypes = [P, ctypes.c_int, I64, I64, I64, P]
    lib.mrr_oracle_unroute.restype = ctypes.c_int
    lib.mrr_oracle_unroute.argtypes = [P, I64, I64, P, ctypes.c_int, I64, I64, P, I64, P, P, P, P]
    return lib


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SOURCE)
                or not _built_for_this_host(LIB)):
            build()
        _lib = _bind(ctypes.CDLL(LIB))
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def offsets(counts: np.ndarray, lib: Optional[ctypes.CDLL] = None):
    """(src_off, dst_off) as [N, E] int64 arrays: SrcOffset / DstOffset of every segment."""
    lib = lib or load()
    c = np.ascontiguousarray(counts)
    N, E = c.shape
    src = np.zeros(N * E + 1, np.int64)
    dst = np.zeros(N * E + 1, np.int64)
    lib.mrr_oracle_offsets(_ptr(c), int(c.dtype == np.int64), N, E, _ptr(src), _ptr(dst))
    return src[: N * E].reshape(N, E), dst[: N * E].reshape(N, E)


def validate(counts: np.ndarray, A: int, lib: Optional[ctypes.CDLL] = None) -> int:
    lib = lib or load()
    c = np.ascontiguousarray(counts)
    N, E = c.shape
    return lib.mrr_oracle_validate(_ptr(c), int(c.dtype == np.int64), N, E, A)


def expert_token_num(counts: np.ndarray, expert_token_num_type: int = 1,
                     lib: Optional[ctypes.CDLL] = None) -> np.ndarray:
    """expert_token_num in count mode (1) or inclusive cumsum mode (0), in the counts' dtype."""
    lib = lib or load()
    c = np.ascontiguousarray(counts)
    N, E = c.shape
    out = np.empty(E, c.dtype)
    rc = lib.mrr_oracle_expert_token_num(_ptr(c), int(c.dtype == np.int64), N, E,
                                         expert_token_num_type, _ptr(out))
    if rc != ORC_OK:
        raise OracleError(rc)
    return out


def run(tokens: np.ndarray, counts: np.ndarray, *, scales: Optional[np.ndarray] = None,
        topk: Optional[np.ndarray] = None, idx_type: int = 0, expert_token_num_type: int = 1,
        lib: Optional[ctypes.CDLL] = None) -> dict:
    """Run the op on byte rows.

    tokens: [A, row_bytes] uint8; counts: [N, E] int32/int64; scales: [A, scale_row_bytes]
    uint8 or None; topk: [A] float32 or None.  Returns a dict with permute_tokens,
    permute_scales (None when scales is None), permute_token_idx (int32 [A]),
    expert_token_num ([E], the counts' dtype), permute_topk_weight (None when topk is None).
    Raises OracleError when the counts are invalid.
    """
    lib = lib or load()
    tok = np.ascontiguousarray(tokens, dtype=np.uint8)
    if tok.ndim != 2:
        raise ValueError("tokens must be [A, row_bytes] bytes")
    A, rb = tok.shape
    c = np.ascontiguousarray(counts)
    if c.dtype not in (np.int32, np.int64) or c.ndim != 2:
        raise ValueError("counts must be a 2-D int32/int64 array")
    N, E = c.shape
    out_tok = np.empty_like(tok)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.uint8)
    sb = 0 if sc is None else sc.shape[1]
    out_sc = None if sc is None else np.empty_like(sc)
    tw = None if topk is None else np.ascontiguousarray(topk, dtype=np.float32).reshape(-1)
    out_tw = None if tw is None else np.empty_like(tw)
    idx = np.empty(A, np.int32)
    etn = np.empty(E, c.dtype)
    rc = lib.mrr_oracle_run(_ptr(tok), A, rb, _ptr(c), int(c.dtype == np.int64), N, E,
                            _ptr(sc), sb, _ptr(tw), _ptr(out_tok), _ptr(out_sc), _ptr(idx),
                            _ptr(etn), _ptr(out_tw), idx_type)
    if rc != ORC_OK:
        raise OracleError(rc)
    if expert_token_num_type != 1:
        etn = expert_token_num(c, expert_token_num_type, lib=lib)
    return {"permute_tokens": out_tok, "permute_scales": out_sc, "permute_token_idx": idx,
            "expert_token_num": etn, "permute_topk_weight": out_tw}


def run_problem(p, lib: Optional[ctypes.CDLL] = None) -> dict:
    """Run the oracle on a ``workloads.Problem``."""
    return run(p.tokens, p.counts, scales=p.scales, topk=p.topk, idx_type=p.idx_type,
               expert_token_num_type=p.expert_token_num_type, lib=lib)


def unroute(permute_tokens: np.ndarray, counts: np.ndarray, *, permute_scales: Optional[np.ndarray] = None,
            permute_topk: Optional[np.ndarray] = None, lib: Optional[ctypes.CDLL] = None) -> dict:
    """The inverse move: expert-major byte rows back to rank-major order.

    Returns a dict with tokens ([A, row_bytes] uint8), scales (None when permute_scales is None)
    and topk_weight ([A] float32 or None).  Raises OracleError when the counts are invalid.
    """
    lib = lib or load()
    pt = np.ascontiguousarray(permute_tokens, dtype=np.uint8)
    if pt.ndim != 2:
        raise ValueError("permute_tokens must be [A, row_bytes] bytes")
    A, rb = pt.shape
    c = np.ascontiguousarray(counts)
    if c.dtype not in (np.int32, np.int64) or c.ndim != 2:
        raise ValueError("counts must be a 2-D int32/int64 array")
    N, E = c.shape
    out_tok = np.empty_like(pt)
    ps = None if permute_scales is None else np.ascontiguousarray(permute_scales, dtype=np.uint8)
    sb = 0 if ps is None else ps.shape[1]
    out_sc = None if ps is None else np.empty_like(ps)
    pw = None if permute_topk is None else np.ascontiguousarray(permute_topk, dtype=np.float32).reshape(-1)
    out_w = None if pw is None else np.empty_like(pw)
    rc = lib.mrr_oracle_unroute(_ptr(pt), A, rb, _ptr(c), int(c.dtype == np.int64), N, E, _ptr(ps), sb,
                                _ptr(pw), _ptr(out_tok), _ptr(out_sc), _ptr(out_w))
    if rc != ORC_OK:
        raise OracleError(rc)
    return {"tokens": out_tok, "scales": out_sc, "topk_weight": out_w}
