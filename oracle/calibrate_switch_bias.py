"""Derive the router bias of the Switch-style skewed workload.

The workload asks for a router bias on four experts large enough that about
70% of the tokens have their largest logit there (it mirrors the 70% share of
the collapsed split drawn in "MoE 混合专家模型稀疏激活的架构原理与负载均衡挑战",
§2.2 figure 坍缩路由). This script bisects that bias on the seed-0 inputs of
the workload using only the float64 oracle's router, rounds it to a multiple
of 1/64 (exact in fp32) and prints it with the share it gives.

Run:  python -m oracle.calibrate_switch_bias
The printed value is stored as SWITCH_SKEW_BIAS in moe_inputs.py.
"""
import numpy as np

import moe_inputs
from oracle import moe_oracle as O


def share_on_skewed(l0: np.ndarray, beta: float, n_skew: int) -> float:
    l = l0.copy()
    l[:, :n_skew] += beta
    return float(np.mean(O.topk_experts(l, 1)[:, 0] < n_skew))


def main(target=0.70):
    w = moe_inputs.workload("switch_skewed", router_bias="none")
    x = moe_inputs.make_x(w)
    w_r, _ = moe_inputs.make_router(w)
    l0 = O.router_logits(x, w_r)
    n = moe_inputs.SWITCH_SKEW_EXPERTS
    lo, hi = 0.0, 10.0
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if share_on_skewed(l0, mid, n) < target:
            lo = mid
        else:
            hi = mid
    beta = round(hi * 64) / 64
    share = share_on_skewed(l0, beta, n)
    print(f"beta={beta!r} share={share:.4f} (bisection point {hi:.6f})")
    return beta, share


if __name__ == "__main__":
    main()
