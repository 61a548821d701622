"""CPU oracle for MoE gating top-k (npu_moe_gating_top_k) -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may import this
module; the CUDA library never uses it and it uses nothing from the library.

Source: the article "CANN 自定义算子详解：npu_moe_gating_top_k 实现 MoE 路由与 TopK 专家选择"
(m.qwbw.cn/news/316089), sections 归一化公式 (normalisation), 分组排序公式 (group ranking),
专家选择公式 (expert selection), 路由权重缩放公式 (weight scaling), 参数说明 (parameters) and
约束说明 (constraints).  Steps, in the page's order, for every row t of x [T, e]:

  1. normOut = Softmax(x) (norm_type 0), Sigmoid(x) (1) or Softplus(x) (2), kept in float32;
  2. normOut += bias, where rows with additional_token_mask[t] true use additional_bias instead;
  3. hash routing (input_ids and tid2eid given): expert_idx = tid2eid[input_ids[t]];
     otherwise split normOut into group_count groups, score each by its maximum
     (group_select_mode 0) or the sum of its two largest values (1), keep the k_group best
     groups, and take the k largest normOut values inside them;
  4. y = normOut at the chosen experts; yOut = y / (sum(y) + eps) * routed_scaling_factor.

Readings where the page is silent:
  * the top-k decisions are taken on the float32 normOut the page stores (both the oracle and the
    GPU decide in float32); equal scores go to the lower group / expert index;
  * y and the optional normOut output include the bias (the page assigns normOut += bias before
    the selection formula reads normOut);
  * experts come out in descending score order;
  * e must be a multiple of group_count; group_select_mode 1 needs groups of at least 2 experts.
The arithmetic of step 4 is done in float64 here.
"""
from __future__ import annotations

from typing import Optional

import numpy as np


class GatingArgError(ValueError):
    pass


def normalize(x: np.ndarray, norm_type: int) -> np.ndarray:
    """Step 1 in float64: Softmax over each row, Sigmoid or Softplus elementwise."""
    x = np.asarray(x, dtype=np.float64)
    if norm_type == 0:
        z = np.exp(x - x.max(axis=-1, keepdims=True))
        return z / z.sum(axis=-1, keepdims=True)
    if norm_type == 1:
        return 1.0 / (1.0 + np.exp(-x))
    if norm_type == 2:
        return np.logaddexp(0.0, x)   # log(1 + exp(x))
    raise GatingArgError("norm_type must be 0, 1 or 2")


def check_args(T, e, k, k_group, group_count, group_select_mode, renorm, norm_type, hashing):
    """The constraints of the page's 约束说明 section and its Torch-side checks."""
    if not (1 <= k <= 64 and k <= e):
        raise GatingArgError("k must be in 1..min(e, 64)")
    if renorm != 0:
        raise GatingArgError("renorm supports 0 only")
    if group_select_mode not in (0, 1) or norm_type not in (0, 1, 2):
        raise GatingArgError("bad mode")
    if group_count < 1 or k_group < 1 or k_group > group_count or e % group_count:
        raise GatingArgError("bad grouping")
    if not hashing and k > (e // group_count) * k_group:
        raise GatingArgError("k exceeds the experts in the kept groups")
    if group_select_mode == 1 and e // group_count < 2:
        raise GatingArgError("top-2 group scores need groups of at least 2 experts")


def gating_topk(x: np.ndarray, k: int, *, bias: Optional[np.ndarray] = None,
                input_ids: Optional[np.ndarray] = None, tid2eid: Optional[np.ndarray] = None,
                additional_bias: Optional[np.ndarray] = None,
                additional_token_mask: Optional[np.ndarray] = None, k_group: int = 1,
                group_count: int = 1, routed_scaling_factor: float = 1.0, eps: float = 1e-20,
                group_select_mode: int = 0, renorm: int = 0, norm_type: int = 0) -> dict:
    """Returns y_out [T, k] float64, expert_idx [T, k] int32 and norm_out [T, e] (float32
    scores with bias, as the selection sees them)."""
    x = np.asarray(x)
    T, e = x.shape
    hashing = input_ids is not None
    if hashing != (tid2eid is not None):
        raise GatingArgError("input_ids and tid2eid come together")
    check_args(T, e, k, k_group, group_count, group_select_mode, renorm, norm_type, hashing)

    # steps 1-2: normalised scores, stored in float32, plus the row's bias
    norm32 = normalize(x.astype(np.float64), norm_type).astype(np.float32)
    score = norm32.copy()
    for t in range(T):
        use_extra = (additional_bias is not None and additional_token_mask is not None
                     and bool(additional_token_mask[t]))
        if use_extra:
            score[t] = (score[t] + np.asarray(additional_bias, np.float32)).astype(np.float32)
        elif bias is not None:
            score[t] = (score[t] + np.asarray(bias, np.float32)).astype(np.float32)

    y_out = np.zeros((T, k), np.float64)
    idx = np.zeros((T, k), np.int32)
    gsize = e // group_count
    for t in range(T):
        row = score[t]
        if hashing:
            chosen = [int(v) for v in tid2eid[int(input_ids[t])][:k]]
        else:
            # step 3: rank the groups, keep the best k_group (ties: lower group index)
            gscores = []
            for g in range(group_count):
                vals = sorted(row[g * gsize:(g + 1) * gsize].tolist(), reverse=True)
                gscores.append(vals[0] if group_select_mode == 0
                               else float(np.float32(vals[0]) + np.float32(vals[1])))
            keep = sorted(range(group_count), key=lambda g: (-gscores[g], g))[:k_group]
            cand = [j for g in sorted(keep) for j in range(g * gsize, (g + 1) * gsize)]
            # then the k largest scores among the kept experts (ties: lower expert index)
            chosen = sorted(cand, key=lambda j: (-float(row[j]), j))[:k]
        y = np.array([float(row[j]) for j in chosen], np.float64)
        # step 4: scale the weights
        y_out[t] = y / (y.sum() + eps) * routed_scaling_factor
        idx[t] = chosen
    return {"y_out": y_out, "expert_idx": idx, "norm_out": score}
