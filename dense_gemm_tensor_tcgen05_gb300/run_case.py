"""Run one GEMM configuration a few times (for profilers and quick timing).

    python -m dense_gemm_tensor_tcgen05_gb300.run_case --dtype bf16 --M 8192 --N 8192 \
        --K 8192 [--dist normal --sigma 0.011] [--iters 5] [--tile-n 256 --split-k 1 ...]

Inputs are the seeded synthetic matrices of ``inputs.make``; the product runs
through the C ABI (gemm_f16f32 / gemm_bf16f32 / sgemm_f32 / the _bt entry
points for tf32, e4m3 and e5m2, or gemm_ex when plan options are given).  For
tf32, e4m3 and e5m2, B is stored as its N x K transpose.  Prints the plan and
the mean time per call.
"""
from __future__ import annotations

import argparse
import math


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--dtype", choices=["f16", "bf16", "f32", "tf32", "e4m3", "e5m2"], default="bf16")
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--N", type=int, default=8192)
    ap.add_argument("--K", type=int, default=8192)
    ap.add_argument("--dist", default="normal")
    ap.add_argument("--sigma", type=float, default=0.0, help="0: 1/sqrt(K) for normal")
    ap.add_argument("--iters", type=int, default=5)
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--swap-ab", type=int, default=-1)
    ap.add_argument("--group-m", type=int, default=0)
    ap.add_argument("--cta-pair", type=int, default=0)
    a = ap.parse_args()

    import numpy as np
    import torch

    import dense_gemm_tensor_tcgen05_gb300 as g
    from dense_gemm_tensor_tcgen05_gb300 import build, inputs

    build.build()
    sigma = a.sigma or (1 / math.sqrt(a.K) if a.dist == "normal" else 1.0)
    A = inputs.make(a.dist, a.dtype, a.M, a.K, 1, 0, sigma)
    B = inputs.make(a.dist, a.dtype, a.K, a.N, 1, 1, sigma)
    code = {"f16": 0, "bf16": 1, "f32": 2, "tf32": 3, "e4m3": 4, "e5m2": 5}[a.dtype]
    bt = code >= 3
    if bt:
        B = np.ascontiguousarray(B.T)
    if a.dtype in ("f32", "tf32"):
        Ad, Bd = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    elif bt:
        Ad, Bd = torch.from_numpy(A.view(np.uint8)).cuda(), torch.from_numpy(B.view(np.uint8)).cuda()
    else:
        Ad, Bd = torch.from_numpy(A.view(np.int16)).cuda(), torch.from_numpy(B.view(np.int16)).cuda()
    Cd = torch.empty((a.M, a.N), dtype=torch.float32, device="cuda")
    opts = {k: v for k, v in dict(tile_n=a.tile_n, split_k=a.split_k, swap_ab=a.swap_ab,
                                  group_m=a.group_m, cta_pair=a.cta_pair).items()
            if v not in (0, -1)}
    if bt and opts:
        opts["trans_b"] = 1
    args = (Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), a.M, a.N, a.K, a.K,
            a.K if bt else a.N, a.N)
    s = torch.cuda.current_stream().cuda_stream
    if opts:
        opts.setdefault("swap_ab", -1)
        call = lambda: g.gemm_ex(*args, dtype=code, stream=s, **opts)
        plan = g.gemm_plan_describe(code, *args, **opts)
    else:
        fn = {0: g.gemm_f16f32, 1: g.gemm_bf16f32, 2: g.sgemm_f32, 3: g.gemm_tf32f32_bt,
              4: g.gemm_e4m3f32_bt, 5: g.gemm_e5m2f32_bt}[code]
        call = lambda: fn(*args, stream=s)
        plan = g.gemm_plan_describe(code, *args, **({"trans_b": 1} if bt else {}))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    call()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(a.iters):
        call()
    e1.record()
    torch.cuda.synchronize()
    g.gemm_device_error(s)
    ms = e0.elapsed_time(e1) / a.iters
    tf = 2.0 * a.M * a.N * a.K / ms / 1e9
    print(f"{a.dtype} {a.M}x{a.N}x{a.K} plan=[{plan}] {ms:.4f} ms/call {tf:.1f} TFLOP/s")


if __name__ == "__main__":
    main()
