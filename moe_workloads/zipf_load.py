"""Expert-load statistics of the Zipf-skewed routing workload for several bias scales.

``python -m moe_workloads.zipf_load`` draws the 535B-shaped layer's x and W_r
at seed 0 and T=16384, routes them with the fp64 oracle's logits for each
bias scale beta, and prints the hottest expert's load over the mean load and
the number of experts that receive no token.
"""
import torch

from moe_workloads import SHAPES, _normal, tensor_seed, zipf_bias
from oracle import moe_oracle


def load_stats(beta, x, wr, shape):
    b = zipf_bias(shape, beta)
    logits, _ = moe_oracle.router_logits(x, wr, b)
    idx = torch.topk(logits, shape.top_k, dim=1).indices   # statistics only: ties do not matter
    counts = torch.bincount(idx.flatten(), minlength=shape.n_experts).double()
    mean = shape.T * shape.top_k / shape.n_experts
    return float(counts.max() / mean), int((counts == 0).sum())


def main():
    s = SHAPES["l535b_zipf_t16384"]
    x = _normal((s.T, s.d_model), 1.0, torch.bfloat16, "cpu", tensor_seed(s.seed, "x"))
    wr = _normal((s.d_model, s.n_experts), s.d_model ** -0.5, torch.bfloat16, "cpu",
                 tensor_seed(s.seed, "w_router"))
    for beta in (0.2, 0.3, 0.37, 0.45, 0.6, 0.8, 1.0, 1.5, 2.0):
        ratio, zeros = load_stats(beta, x, wr, s)
        print(f"beta={beta:.2f}  hottest/mean={ratio:6.2f}  experts with no token={zeros}")


if __name__ == "__main__":
    main()
