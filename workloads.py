"""Seeded synthetic inputs for the MoE re-routing step (rank-major -> expert-major).

This module only draws random inputs: count matrices, token rows, per-token scales and
top-k weights, with the shapes and value distributions of the workloads the
MoeReRoutingV2 pages use. It holds none of the re-routing arithmetic (no offsets, no
permutation), so both the CUDA path and the CPU oracle can consume its output without
sharing any of the method's code.

Every tensor payload is returned as raw bytes (``uint8`` arrays) because the op moves
bytes; typed views are built by the caller.

Sources for the shapes:
  * "CANN ops-transformer MoeReRoutingV2" article (m.nlpx.cn/news/59074), section
    参数说明: tokens [A,H] in FLOAT16/BF16/INT8/FP8/HIFLOAT8/FP4, counts [N,E] int32/int64
    with every entry > 0, per_token_scales [A] / [A,S] fp32 or [A,K/64,2] e8m0,
    expert_topk_weight [A,1] fp32.
  * "torch_npu.npu_moe_re_routing" page (hiascend.com ptaoplist_002370), section 调用示例:
    A=16384, H=7168 int8 tokens from randint(-10, 20), a 16x16 count matrix of ones
    whose last cell takes the remainder A-255.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# bits per element of each token dtype the pages list (section 参数说明).
TOKEN_BITS = {
    "float16": 16,
    "bfloat16": 16,
    "int8": 8,
    "float8_e5m2": 8,
    "float8_e4m3fn": 8,
    "hifloat8": 8,
    "float4_e2m1": 4,
    "float4_e1m2": 4,
}

# scale layouts: bytes per element (fp32 = 4, float8_e8m0 = 1)
SCALE_ELEM_BYTES = {"none": 0, "f32_a": 4, "f32_as": 4, "e8m0": 1}


@dataclasses.dataclass
class Problem:
    """One re-routing problem instance: all payloads as raw little-endian bytes."""

    name: str
    A: int
    H: int
    N: int
    E: int
    token_dtype: str
    counts: np.ndarray            # [N, E] int32 or int64
    tokens: np.ndarray            # [A, row_bytes] uint8
    scale_layout: str             # "none" | "f32_a" | "f32_as" | "e8m0"
    scale_cols: int               # elements per scale row: 1, S or (K/64)*2
    scales: Optional[np.ndarray]  # [A, scale_row_bytes] uint8, or None
    topk: Optional[np.ndarray]    # [A] float32, or None
    idx_type: int = 0
    expert_token_num_type: int = 1

    @property
    def row_bytes(self) -> int:
        return self.H * TOKEN_BITS[self.token_dtype] // 8

    @property
    def scale_row_bytes(self) -> int:
        return self.scale_cols * SCALE_ELEM_BYTES[self.scale_layout]

    @property
    def count_is_i64(self) -> bool:
        return self.counts.dtype == np.int64

    def algorithmic_bytes(self) -> int:
        """Bytes the step must read plus write, each item once.

        tokens, scales and top-k weights are read once and written once; the count matrix is
        read; permute_token_idx (int32) and expert_token_num (count int type) are written.
        """
        cb = self.counts.dtype.itemsize
        b = 2 * self.A * self.row_bytes
        if self.scales is not None:
            b += 2 * self.A * self.scale_row_bytes
        if self.topk is not None:
            b += 2 * 4 * self.A
        b += 4 * self.A + self.N * self.E * cb + self.E * cb
        return b


# ----------------------------------------------------------------------------- counts

def counts_uniform(rng: np.random.Generator, N: int, E: int, A: int, dtype=np.int32) -> np.ndarray:
    """Every cell >= 1, the remaining A - N*E tokens spread by a uniform multinomial."""
    if A < N * E:
        raise ValueError("A must be >= N*E for positive counts")
    extra = rng.multinomial(A - N * E, np.full(N * E, 1.0 / (N * E)))
    return (1 + extra).reshape(N, E).astype(dtype)


def counts_dirichlet(rng: np.random.Generator, N: int, E: int, A: int, alpha=1.0, dtype=np.int64) -> np.ndarray:
    p = rng.dirichlet(np.full(N * E, alpha))
    extra = rng.multinomial(A - N * E, p)
    return (1 + extra).reshape(N, E).astype(dtype)


def counts_zipf_experts(rng: np.random.Generator, N: int, E: int, A: int, s=1.2, dtype=np.int32) -> np.ndarray:
    """Experts skewed by z_j ~ (j+1)^-s, ranks uniform; every cell >= 1."""
    z = (np.arange(E, dtype=np.float64) + 1.0) ** (-s)
    p = np.tile(z / N, N)
    p = p / p.sum()
    extra = rng.multinomial(A - N * E, p)
    return (1 + extra).reshape(N, E).astype(dtype)


def counts_v1_example(N: int, E: int, A: int, dtype=np.int32) -> np.ndarray:
    """The count matrix of the npu_moe_re_routing usage example: ones, last cell = rest."""
    c = np.ones((N, E), dtype=dtype)
    c[N - 1, E - 1] = A - (N * E - 1)
    return c


# ----------------------------------------------------------------------------- payloads

def _to_bf16_bytes(x: np.ndarray) -> np.ndarray:
    import torch  # CPU rounding to bf16 (round-to-nearest-even) only

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.uint8).numpy().copy()


def token_bytes(rng: np.random.Generator, A: int, H: int, token_dtype: str) -> np.ndarray:
    """[A, row_bytes] uint8 payload drawn per the dtype's workload distribution."""
    bits = TOKEN_BITS[token_dtype]
    rb = H * bits // 8
    if token_dtype == "int8":
        v = rng.integers(-10, 20, size=(A, H), dtype=np.int8)
        return v.view(np.uint8).reshape(A, rb)
    if token_dtype == "float16":
        v = rng.standard_normal(size=(A, H), dtype=np.float32).astype(np.float16)
        return v.view(np.uint8).reshape(A, rb)
    if token_dtype == "bfloat16":
        v = rng.standard_normal(size=(A, H), dtype=np.float32)
        return _to_bf16_bytes(v).reshape(A, rb)
    if token_dtype == "float8_e4m3fn":
        # uniform over the 254 non-NaN e4m3fn encodings (0x7F and 0xFF are NaN)
        v = rng.integers(0, 254, size=(A, rb), dtype=np.uint16)
        v = v + (v >= 0x7F)
        return v.astype(np.uint8)
    # e5m2, hifloat8 and packed fp4: arbitrary bytes (the op never interprets them)
    return rng.integers(0, 256, size=(A, rb), dtype=np.uint16).astype(np.uint8)


def scale_bytes(rng: np.random.Generator, A: int, layout: str, cols: int) -> Optional[np.ndarray]:
    if layout == "none":
        return None
    if layout in ("f32_a", "f32_as"):
        v = rng.standard_normal(size=(A, cols), dtype=np.float32)
        return v.view(np.uint8).reshape(A, 4 * cols)
    if layout == "e8m0":
        return rng.integers(120, 135, size=(A, cols), dtype=np.uint16).astype(np.uint8)
    raise ValueError(layout)


def topk_weights(rng: np.random.Generator, A: int) -> np.ndarray:
    return rng.random(A, dtype=np.float32)


def make_problem(rng: np.random.Generator, *, A: int, H: int, N: int, E: int,
                 token_dtype="bfloat16", count_dtype=np.int32, counts: Optional[np.ndarray] = None,
                 scale_layout="f32_a", scale_cols=1, has_topk=True, idx_type=0,
                 name="fuzz") -> Problem:
    """Draw counts -> tokens -> scales -> topk, in that order, from ``rng``."""
    if counts is None:
        counts = counts_uniform(rng, N, E, A, count_dtype)
    tok = token_bytes(rng, A, H, token_dtype)
    sc = scale_bytes(rng, A, scale_layout, scale_cols)
    tw = topk_weights(rng, A) if has_topk else None
    return Problem(name=name, A=A, H=H, N=N, E=E, token_dtype=token_dtype, counts=counts,
                   tokens=tok, scale_layout=scale_layout, scale_cols=scale_cols, scales=sc,
                   topk=tw, idx_type=idx_type)


# ----------------------------------------------------------------------------- the five workloads

CONFIG_NAMES = {
    1: "tiny A=64 H=128 bf16 N=4 E=4",
    2: "A=16384 H=7168 int8 N=16 E=16 skewed, no topk",
    3: "A=16384 H=7168 bf16 N=8 E=32 int64 counts, scales [A,4]",
    4: "A=32768 H=7168 fp8e4m3 N=32 E=8 zipf, e8m0 scales [A,112,2]",
    5: "A=262144 H=256 fp16 N=64 E=64 small rows",
}


def config(k: int, idx_type: Optional[int] = None) -> Problem:
    """Workload k (1..5), drawn with numpy default_rng(1000 + k)."""
    rng = np.random.default_rng(1000 + k)
    if k == 1:
        A, H, N, E = 64, 128, 4, 4
        c = counts_uniform(rng, N, E, A, np.int32)
        p = make_problem(rng, A=A, H=H, N=N, E=E, token_dtype="bfloat16", counts=c,
                         scale_layout="f32_a", scale_cols=1, has_topk=True, idx_type=0)
    elif k == 2:
        A, H, N, E = 16384, 7168, 16, 16
        c = counts_v1_example(N, E, A, np.int32)
        p = make_problem(rng, A=A, H=H, N=N, E=E, token_dtype="int8", counts=c,
                         scale_layout="f32_a", scale_cols=1, has_topk=False, idx_type=0)
    elif k == 3:
        A, H, N, E = 16384, 7168, 8, 32
        c = counts_dirichlet(rng, N, E, A, 1.0, np.int64)
        p = make_problem(rng, A=A, H=H, N=N, E=E, token_dtype="bfloat16", counts=c,
                         scale_layout="f32_as", scale_cols=4, has_topk=True, idx_type=1)
    elif k == 4:
        A, H, N, E = 32768, 7168, 32, 8
        c = counts_zipf_experts(rng, N, E, A, 1.2, np.int32)
        p = make_problem(rng, A=A, H=H, N=N, E=E, token_dtype="float8_e4m3fn", counts=c,
                         scale_layout="e8m0", scale_cols=(H // 64) * 2, has_topk=True, idx_type=0)
    elif k == 5:
        A, H, N, E = 262144, 256, 64, 64
        c = counts_uniform(rng, N, E, A, np.int32)
        p = make_problem(rng, A=A, H=H, N=N, E=E, token_dtype="float16", counts=c,
                         scale_layout="f32_a", scale_cols=1, has_topk=True, idx_type=0)
    else:
        raise ValueError(f"no workload {k}")
    p.name = f"C{k}: {CONFIG_NAMES[k]}"
    if idx_type is not None:
        p.idx_type = idx_type
    return p


# ----------------------------------------------------------------------------- gating top-k inputs
# Source for the shapes: "CANN 自定义算子详解：npu_moe_gating_top_k" (m.qwbw.cn/news/316089),
# section 调用示例: x ~ randn(batch, 384) float16, top-6, sigmoid; bias / additional_bias ~ rand(e).

GATING_NAMES = {
    1: "gating: T=16384 tokens x 384 experts fp16, top-6, sigmoid, no groups",
    2: "gating: T=16384 tokens x 256 experts bf16, 8 groups keep 4, top-8, sigmoid + bias, top-2 group scores",
    3: "gating: T=16384 tokens x 384 experts fp32, top-6, sigmoid, no groups",
}


def gating_config(k: int) -> dict:
    """Gating workload k (1, 2, 3), drawn with numpy default_rng(2000 + k).  x and bias are float32
    arrays holding values already rounded to the workload's dtype."""
    import torch

    rng = np.random.default_rng(2000 + k)

    def rounded(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dt).to(torch.float32).numpy()

    if k == 1:
        T, e = 16384, 384
        x = rounded(rng.standard_normal((T, e)), torch.float16)
        return dict(name=GATING_NAMES[1], dtype="float16", x=x, k=6, bias=None, k_group=1, group_count=1,
                    group_select_mode=0, norm_type=1, routed_scaling_factor=1.0, eps=1e-6)
    if k == 2:
        T, e = 16384, 256
        x = rounded(rng.standard_normal((T, e)), torch.bfloat16)
        bias = rounded(rng.random(e) * 0.1, torch.bfloat16)
        return dict(name=GATING_NAMES[2], dtype="bfloat16", x=x, k=8, bias=bias, k_group=4, group_count=8,
                    group_select_mode=1, norm_type=1, routed_scaling_factor=2.5, eps=1e-20)
    if k == 3:
        T, e = 16384, 384
        x = rng.standard_normal((T, e)).astype(np.float32)
        return dict(name=GATING_NAMES[3], dtype="float32", x=x, k=6, bias=None, k_group=1, group_count=1,
                    group_select_mode=0, norm_type=1, routed_scaling_factor=1.0, eps=1e-6)
    raise ValueError(f"no gating workload {k}")
