"""Run one workload of the path a few times, for a profiler to attach to.

    python -m nvfp4_block_scaled_quant_gb300.profile_case moe --experts 64 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case decode --T 1 --experts 384 --iters 8
    python -m nvfp4_block_scaled_quant_gb300.profile_case gemm --M 4096 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case linear --M 32 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case grouped --M 1 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case dispatch --T 128 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case norm --M 128 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case router --T 128 --iters 3
    python -m nvfp4_block_scaled_quant_gb300.profile_case quant --M 4096 --iters 3

``moe`` runs 128-token prefill chunks (hidden 7168, intermediate 2048, top-8
Zipf(1.1) routing, shared expert; ``--T`` above 1 sets the batch instead, e.g.
4096 for the whole prefill's 128-row tiles) over ``--experts`` experts, so the weights
held on the device stay a few GB while the per-tile work of every kernel is
the same as in the 384-expert layer.  The kernels launch in the same order and
configuration as in the benchmark.  ``dispatch`` runs routing + amax + the
quantise/permute of x for a 384-expert layer (the prefill chunks' routing at
T = 128, the decode routing below, the 32 chunks at once for T = 4096; no expert
weights are needed); ``norm`` the fused RMSNorm -> NVFP4 quantiser over hidden
7168; ``router`` the router gate (384 experts, hidden 7168, top-8); ``quant``
the activation quantiser over K = 7168 (M = 1024 .. 16384 are the large-GEMM
sweep's activations); ``linear`` the dense 1536 -> 16384 linear and ``grouped`` the
fixed-group 8 x (4096 -> 1024) linear at ``--M`` tokens.
"""

from __future__ import annotations

import argparse
import sys

import torch

from . import build as B


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("case", choices=["moe", "decode", "gemm", "linear", "grouped", "dispatch", "norm", "router", "quant"])
    p.add_argument("--T", type=int, default=1)
    p.add_argument("--experts", type=int, default=64)
    p.add_argument("--M", type=int, default=4096)
    p.add_argument("--iters", type=int, default=3)
    a = p.parse_args(argv)
    B.build()
    from . import model, ops, workloads

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if a.case == "moe":
        cfg = workloads.PREFILL
        E = a.experts
        T = a.T if a.T > 1 else cfg.T
        W = model.make_moe_weights(E, cfg.H, cfg.I, workloads.BENCH_WEIGHT_SEED, dev, shared=True)
        sub = workloads.MoEConfig("profile", T, cfg.H, cfg.I, E, cfg.topk, True, "zipf", True)
        a2 = torch.full((E + 1,), 0.02, dtype=torch.float32, device=dev)
        ws = ops.moe_workspace(T, cfg.H, cfg.I, E, cfg.topk, True, dev)
        y = torch.empty(T, cfg.H, dtype=torch.bfloat16, device=dev)
        for i in range(a.iters):
            x = workloads.activations(T, cfg.H, seed=700_000 + i, device=dev, outliers=True)
            ids, w = workloads.routing(sub, seed=800_000 + i, device=dev)
            ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
    elif a.case == "decode":
        cfg = workloads.DECODE[a.T]
        E = a.experts
        W = model.make_moe_weights(E, cfg.H, cfg.I, workloads.BENCH_WEIGHT_SEED, dev, shared=True)
        sub = workloads.MoEConfig("profile", a.T, cfg.H, cfg.I, E, cfg.topk, True, "uniform", False)
        a2 = torch.full((E + 1,), 0.02, dtype=torch.float32, device=dev)
        ws = ops.moe_workspace(a.T, cfg.H, cfg.I, E, cfg.topk, True, dev)
        y = torch.empty(a.T, cfg.H, dtype=torch.bfloat16, device=dev)
        for i in range(a.iters):
            x = workloads.activations(a.T, cfg.H, seed=900_000 + i, device=dev)
            ids, w = workloads.routing(sub, seed=950_000 + i, device=dev)
            ops.moe_forward(x, ids, w, W, a2, workspace=ws, out=y)
    elif a.case == "gemm":
        K = N = 7168
        dw = model.make_dense_weight(N, K, seed=70, device=dev)
        x = workloads.activations(a.M, K, seed=80, device=dev)
        q, sf, gs = ops.quantize_act(x)
        y = torch.empty(a.M, N, dtype=torch.bfloat16, device=dev)
        for _ in range(a.iters):
            ops.gemm(q, sf, gs, K, dw.w, dw.sf, dw.ws2, N, out=y)
    elif a.case == "dispatch":
        T = a.T
        cfg = workloads.PREFILL if T == 128 else (workloads.PREFILL_WHOLE if T == 4096 else workloads.DECODE[T])
        W = ops.MoEWeights(cfg.E, cfg.H, cfg.I, *([torch.empty(0, device=dev)] * 6))  # shapes only
        W.sh_w13 = torch.empty(0, device=dev)
        ws = ops.moe_workspace(T, cfg.H, cfg.I, cfg.E, cfg.topk, True, dev)
        g = torch.empty(1, dtype=torch.float32, device=dev)
        if T == 4096:
            x, ids, _ = workloads.prefill_whole(device="cpu")
            ins = [(x.to(dev), ids.to(dev))] * a.iters
        elif T == 128:
            ins = [workloads.prefill_chunk(i, device=dev)[:2] for i in range(a.iters)]
        else:
            ins = [workloads.decode_step(T, step=i, device=dev)[:2] for i in range(a.iters)]
        for x, ids in ins:
            ops.moe_dispatch(x, ids, W, g, True, ws)
    elif a.case == "norm":
        K = 7168
        gamma = workloads.norm_weight(K, seed=5, device=dev)
        for i in range(a.iters):
            x = workloads.activations(a.M, K, seed=500 + i, device=dev, outliers=True)
            ops.rmsnorm_quantize(x, gamma, workloads.RMSNORM_EPS)
    elif a.case == "router":
        _, H, E, k = workloads.ROUTER[a.T]
        q, sfw, ws2 = model.quantize_weight(workloads.weight(E, H, workloads.ROUTER_WEIGHT_SEED, dev))
        wg = ops.router_prepare(q, sfw, ws2, E, H)
        for i in range(a.iters):
            x = workloads.activations(a.T, H, seed=40 + i, device=dev)
            ops.router(x, wg, k)
    elif a.case == "quant":
        for i in range(a.iters):
            x = workloads.activations(a.M, 7168, seed=80 + i, device=dev)
            ops.quantize_act(x)
    elif a.case == "grouped":
        _, G, K, N = workloads.GROUPED_LINEAR.get(a.M, (a.M, 8, 4096, 1024))
        gw = model.make_grouped_weight(G, N, K, seed=90, device=dev)
        x = workloads.activations(a.M, G * K, seed=95, device=dev, outliers=True)
        for _ in range(a.iters):
            ops.grouped_linear(x, gw.w, gw.sf, gw.ws2, G, N)
    else:
        K, N = 1536, 16384
        dw = model.make_dense_weight(N, K, seed=50, device=dev)
        x = workloads.activations(a.M, K, seed=60, device=dev, outliers=True)
        for _ in range(a.iters):
            ops.linear(x, dw.w, dw.sf, dw.ws2, N)
    torch.cuda.synchronize()
    st, flags = ops.device_error()
    if st != 0:
        print(f"device fault flags {flags:#x}", file=sys.stderr)
        return 1
    print(f"{a.case}: {a.iters} iterations done")
    return 0


if __name__ == "__main__":
    sys.exit(main())
