"""Single-kernel timing driver (CUDA events) for the library's hot kernels.

Runs one kernel of the calibration path on synthetic inputs at a chosen shape
through the C ABI's test hooks and prints the average launch time with the
algorithmic bytes/flops.  It is also the small, self-contained case used for
Nsight Compute captures of one kernel, e.g.

  python -m drift_aware_kv_gb300.kbench gemm --M 136 --N 24576 --K 4096
  python -m drift_aware_kv_gb300.kbench attn --R 136 --N 768 --H 32 --Hkv 32
  python -m drift_aware_kv_gb300.kbench kmeans --P 32 --nw 96 --d 4096
"""
from __future__ import annotations

import argparse
import json

import torch


def _time(fn, iters, warmup=3):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(iters):
        fn()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def bench_gemm(a):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(a.M, a.K, device="cuda", generator=g).to(torch.bfloat16)
    W = (0.02 * torch.randn(a.N, a.K, device="cuda", generator=g)).to(torch.bfloat16)
    C = torch.empty(a.M, a.N, device="cuda")
    if a.path == 2:  # library comparison point (cuBLAS through torch), not a path of the product
        ms = _time(lambda: torch.matmul(A, W.t()), a.iters)
    else:
        ms = _time(lambda: P.debug_gemm(A, W, C, a.path), a.iters)
    byts = (a.N * a.K + a.M * a.K) * 2 + a.M * a.N * 4
    return dict(kernel="gemm", M=a.M, N=a.N, K=a.K, path=a.path, us=ms * 1e3, GBps=byts / ms / 1e6,
                TFLOPs=2 * a.M * a.N * a.K / ms / 1e9)


def bench_attn(a):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    dh = a.dh
    q = (1.6 * torch.randn(a.R, a.H * dh, device="cuda", generator=g)).to(torch.bfloat16)
    kv = (1.6 * torch.randn(a.N, 2, a.Hkv * dh, device="cuda", generator=g)).to(torch.bfloat16)
    tracked = torch.tensor([r >= a.R - a.tracked for r in range(a.R)], dtype=torch.uint8, device="cuda")
    prev = torch.zeros(a.R, a.H, a.N, device="cuda")
    plse = torch.zeros(a.R, a.H, device="cuda")
    out = torch.empty(a.R, a.H * dh, dtype=torch.bfloat16, device="cuda")
    kl = torch.empty(a.R, a.H, device="cuda")
    P.attention_noalloc(q, kv, a.H, a.Hkv, tracked, prev, plse, 0, 1, out, kl)
    ms = _time(lambda: P.attention_noalloc(q, kv, a.H, a.Hkv, tracked, prev, plse, 1, 1, out, kl), a.iters)
    byts = a.N * 2 * a.Hkv * dh * 2 + a.R * a.H * dh * 4 + a.tracked * a.H * a.N * 8
    return dict(kernel="attention", R=a.R, N=a.N, H=a.H, Hkv=a.Hkv, us=ms * 1e3, GBps=byts / ms / 1e6,
                TFLOPs=4 * a.R * a.N * a.H * dh / ms / 1e9)


def bench_kmeans(a):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    Hw = torch.randn(a.P, a.nw, a.d, device="cuda", generator=g)
    ms = _time(lambda: P.debug_kmeans(Hw, 8, 10, 0, 0), a.iters)
    byts = a.P * a.nw * a.d * 4 + a.P * 3 * 8 * a.d * 4 + a.P * a.nw * a.d * 9 // 16
    return dict(kernel="kmeans_nvfp4", P=a.P, nw=a.nw, d=a.d, us=ms * 1e3, GBps=byts / ms / 1e6)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["gemm", "attn", "kmeans"])
    ap.add_argument("--M", type=int, default=136)
    ap.add_argument("--N", type=int, default=None, help="gemm N (default 4096) / attention keys (default 768)")
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--path", type=int, default=1, help="0 CUDA cores, 1 tcgen05, 2 cuBLAS (reference point)")
    ap.add_argument("--R", type=int, default=136)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=32)
    ap.add_argument("--dh", type=int, default=128)
    ap.add_argument("--tracked", type=int, default=8)
    ap.add_argument("--P", type=int, default=32)
    ap.add_argument("--nw", type=int, default=96)
    ap.add_argument("--d", type=int, default=4096)
    ap.add_argument("--iters", type=int, default=20)
    a = ap.parse_args()
    if a.N is None:
        a.N = 4096 if a.kernel == "gemm" else 768
    from drift_aware_kv_gb300.build import build
    build()
    fn = {"gemm": bench_gemm, "attn": bench_attn, "kmeans": bench_kmeans}[a.kernel]
    print(json.dumps(fn(a)))


if __name__ == "__main__":
    main()
