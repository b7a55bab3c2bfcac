"""Single-kernel timing driver (CUDA events) for the library's hot kernels.

Runs one kernel of the calibration path on synthetic inputs at a chosen shape
through the C ABI's test hooks and prints the average launch time with the
algorithmic bytes/flops.  It is also the small, self-contained case used for
Nsight Compute captures of one kernel, e.g.

  python -m drift_aware_kv_gb300.kbench gemm --M 136 --N 24576 --K 4096
  python -m drift_aware_kv_gb300.kbench attn --R 136 --N 768 --H 32 --Hkv 32
  python -m drift_aware_kv_gb300.kbench kmeans --P 32 --nw 96 --d 4096
  python -m drift_aware_kv_gb300.kbench stale --rows 24576 --Hkv 32 --dh 128
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


L2_BYTES = 129 * 2**20


def bench_gemm(a):
    """Average launch time over a rotation of weight copies that together exceed
    L2 (as in the layer loop, where every projection reads weights it has not
    read since the previous step)."""
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    A = torch.randn(a.M, a.K, device="cuda", generator=g).to(torch.bfloat16)
    wbytes = a.N * a.K * 2
    ncopy = max(2, -(-3 * L2_BYTES // wbytes))
    Ws = [(0.02 * torch.randn(a.N, a.K, device="cuda", generator=g)).to(torch.bfloat16) for _ in range(ncopy)]
    C = torch.empty(a.M, a.N, device="cuda")
    it = [0]

    def nxt():
        it[0] = (it[0] + 1) % ncopy
        return Ws[it[0]]

    if getattr(a, "swiglu", False):
        # gate and up halves of each weight copy, SwiGLU fused into the epilogue
        F = a.N // 2
        act = torch.empty(a.M, F, dtype=torch.bfloat16, device="cuda")
        ms = _time(lambda: (lambda W: P.debug_gemm_swiglu(A, W[:F], W[F:], act, 1))(nxt()), a.iters)
    elif a.cublas:  # library comparison point (cuBLAS through torch), not a path of the product
        ms = _time(lambda: torch.matmul(A, nxt().t()), a.iters)
    else:
        path = P.gemm_path(a.path, a.stages, a.splits, getattr(a, "bn", 0))
        ms = _time(lambda: P.debug_gemm(A, nxt(), C, path, N=a.N), a.iters)
    byts = (a.N * a.K + a.M * a.K) * 2 + a.M * a.N * 4
    return dict(kernel="gemm", M=a.M, N=a.N, K=a.K, path=-1 if a.cublas else a.path, stages=a.stages, splits=a.splits,
                bn=getattr(a, "bn", 0), us=ms * 1e3, GBps=byts / ms / 1e6,
                TFLOPs=2 * a.M * a.N * a.K / ms / 1e9)


def bench_attn(a):
    if a.batch > 1:
        return bench_attn_batch(a)
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
    P.attention_impl(getattr(a, "impl", 0))
    P.attention_noalloc(q, kv, a.H, a.Hkv, tracked, prev, plse, 0, 1, out, kl)
    ms = _time(lambda: P.attention_noalloc(q, kv, a.H, a.Hkv, tracked, prev, plse, 1, 1, out, kl), a.iters)
    byts = a.N * 2 * a.Hkv * dh * 2 + a.R * a.H * dh * 4 + a.tracked * a.H * a.N * 8
    return dict(kernel="attention", impl=getattr(a, "impl", 0), R=a.R, N=a.N, H=a.H, Hkv=a.Hkv, us=ms * 1e3, GBps=byts / ms / 1e6,
                TFLOPs=4 * a.R * a.N * a.H * dh / ms / 1e9)


def bench_attn_batch(a):
    """The layer loop's launch shape: `batch` sequences of R rows (the last
    `tracked` of each with KL drift) over N keys each, one launch."""
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    dh, S = a.dh, a.batch
    q = (1.6 * torch.randn(S * a.R, a.H * dh, device="cuda", generator=g)).to(torch.bfloat16)
    kv = (1.6 * torch.randn(S, a.N, 2, a.Hkv * dh, device="cuda", generator=g)).to(torch.bfloat16)
    tracked = [r >= a.R - a.tracked for r in range(a.R)]
    prev = torch.zeros(S * a.R, a.H, a.N, device="cuda")
    plse = torch.zeros(S * a.R, a.H, device="cuda")
    out = torch.empty(S * a.R, a.H * dh, dtype=torch.bfloat16, device="cuda")
    kl = torch.empty(S * a.R, a.H, device="cuda")
    P.attention_impl(getattr(a, "impl", 0))
    P.debug_attention_batch(q, kv, a.H, a.Hkv, tracked, prev, plse, 0, 1, out, kl)
    ms = _time(lambda: P.debug_attention_batch(q, kv, a.H, a.Hkv, tracked, prev, plse, 1, 1, out, kl), a.iters)
    byts = S * (a.N * 2 * a.Hkv * dh * 2 + a.R * a.H * dh * 4 + a.tracked * a.H * a.N * 8)
    return dict(kernel="attention", impl=getattr(a, "impl", 0), batch=S, R=a.R, N=a.N, H=a.H, Hkv=a.Hkv,
                us=ms * 1e3, GBps=byts / ms / 1e6, TFLOPs=4 * S * a.R * a.N * a.H * dh / ms / 1e9,
                note="includes the hook's host-side table build and a stream synchronise per call")


def bench_kmeans(a):
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    Hw = torch.randn(a.P, a.nw, a.d, device="cuda", generator=g)
    ms = _time(lambda: P.debug_kmeans(Hw, 8, 10, 0, 0), a.iters)
    byts = a.P * a.nw * a.d * 4 + a.P * 3 * 8 * a.d * 4 + a.P * a.nw * a.d * 9 // 16
    return dict(kernel="kmeans_nvfp4", P=a.P, nw=a.nw, d=a.d, us=ms * 1e3, GBps=byts / ms / 1e6)


def bench_stale(a):
    """KV-cache staleness kernel over a cache pair of `rows` rows [2, Hkv*dh] bf16
    (LLaDA-8B, batch 1: 32 layers x 768 positions = 24576 rows, 805 MB)."""
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    kv = torch.randn(a.rows, 2, a.Hkv * a.dh, device="cuda", generator=g).to(torch.bfloat16)
    ref = (kv.float() + 0.1 * torch.randn(kv.shape, device="cuda", generator=g)).to(torch.bfloat16)
    E = torch.empty(a.rows, device="cuda")
    ms = _time(lambda: P.kv_staleness(kv, ref, a.Hkv, E), a.iters)
    byts = a.rows * (4 * a.Hkv * a.dh * 2 + 4)
    return dict(kernel="kv_staleness", rows=a.rows, Hkv=a.Hkv, dh=a.dh, us=ms * 1e3, GBps=byts / ms / 1e6)


def bench_codec(a):
    """Encode + decode of one storage format over `rows` window rows of width d
    (residual against 8 anchors), bytes moved = the fp32 states read and written
    plus the codes and scales written and read back."""
    from drift_aware_kv_gb300 import polestar as P
    g = torch.Generator(device="cuda").manual_seed(0)
    h = torch.randn(a.rows, a.d, device="cuda", generator=g)
    anchors = torch.randn(8, a.d, device="cuda", generator=g)
    labels = torch.randint(0, 8, (a.rows,), device="cuda", generator=g).to(torch.uint8)
    out = torch.empty_like(h)
    codes, scales = P.codec_encode(a.fmt, h, anchors, labels)

    def run():
        P.codec_encode(a.fmt, h, anchors, labels)
        P.codec_decode(a.fmt, codes, scales, a.rows, a.d, anchors, labels, out=out)

    ms = _time(run, a.iters)
    nc, ns = P.codec_bytes(a.fmt, a.rows, a.d)
    byts = 2 * a.rows * a.d * 4 + 2 * (nc + ns)
    return dict(kernel="codec", fmt=a.fmt, rows=a.rows, d=a.d, us=ms * 1e3, GBps=byts / ms / 1e6)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["gemm", "attn", "kmeans", "stale", "codec"])
    ap.add_argument("--fmt", default="nvfp4", help="codec: fp16, fp8, int8, mxfp4, int2, nvfp4")
    ap.add_argument("--rows", type=int, default=24576, help="staleness: cache rows (layers x positions)")
    ap.add_argument("--M", type=int, default=136)
    ap.add_argument("--N", type=int, default=None, help="gemm N (default 4096) / attention keys (default 768)")
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--path", type=int, default=1,
                    help="0 CUDA cores, 1 tcgen05 (library's choice), 2 row-tiled tcgen05, "
                         "3 weight-stationary tcgen05, 7 two-SM pair tiles")
    ap.add_argument("--cublas", action="store_true", help="time cuBLAS (through torch) instead: comparison point")
    ap.add_argument("--swiglu", action="store_true",
                    help="gate/up projection with the SwiGLU activation fused (N = 2F: gate and up halves)")
    ap.add_argument("--stages", type=int, default=0, help="tcgen05 ring depth (0 = library's choice)")
    ap.add_argument("--bn", type=int, default=0, help="row-tiled columns per tile (0 = library's choice)")
    ap.add_argument("--splits", type=int, default=0,
                    help="tcgen05 cluster K split, or k-blocks per stage for path 7 (0 = library's choice)")
    ap.add_argument("--impl", type=int, default=0,
                    help="attention kernel: 0 library's choice, 1 pipelined mma.sync, 2 tcgen05")
    ap.add_argument("--R", type=int, default=136)
    ap.add_argument("--batch", type=int, default=1, help="attention: sequences in one launch")
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
    fn = {"gemm": bench_gemm, "attn": bench_attn, "kmeans": bench_kmeans, "stale": bench_stale,
          "codec": bench_codec}[a.kernel]
    print(json.dumps(fn(a)))


if __name__ == "__main__":
    main()
