"""ctypes binding of the Polestar C ABI (``include/polestar.h``).

Argument marshalling only: every step of the calibration + commit path runs in
the CUDA library.  The functions keep the C names; ``Polestar`` is a small
convenience wrapper that owns a context for torch-allocated weights/streams.
If the library is missing the binding raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libpolestar.so")

OK, ERR_INVALID_ARG, ERR_CUDA, ERR_OOM, ERR_STATE, ERR_TIMEOUT, ERR_UNSUPPORTED = range(7)
FP32, BF16 = 0, 1
(BUF_KV, BUF_CENTROID, BUF_CSUM, BUF_ANCHOR, BUF_LABELS, BUF_CODES, BUF_SCALES, BUF_ACT_OUT,
 BUF_UPDATE, BUF_CONF, BUF_DREL, BUF_TAUD, BUF_PROXY, BUF_WINDOW_H, BUF_DRIFT, BUF_TOPK,
 BUF_SELECTED, BUF_DELTA, BUF_PROXY_LSE, BUF_ACTIVE_PREV, BUF_ACTIVE_LSE, BUF_THETA,
 BUF_THETA_N) = range(23)

EXPORTED = ("polestar_init", "polestar_calibrate_step", "polestar_commit", "polestar_step_host",
            "polestar_release", "polestar_last_error", "polestar_launch_count", "polestar_debug_read",
            "polestar_profile_begin", "polestar_profile_end", "polestar_debug_gemm",
            "polestar_debug_attention", "polestar_debug_kmeans", "polestar_attention_noalloc",
            "polestar_debug_gemm_choice",
            "polestar_debug_attention_impl", "polestar_debug_gemm_swiglu", "polestar_full_forward",
            "polestar_kv_staleness", "polestar_cache_staleness", "polestar_debug_attention_items",
            "polestar_debug_window", "polestar_debug_trigger", "polestar_debug_stalled_wait",
            "polestar_codec_bytes", "polestar_codec_encode", "polestar_codec_decode",
            "polestar_debug_write", "polestar_debug_enter_block", "polestar_decode_logits",
            "polestar_decode_tokens", "polestar_embed", "polestar_debug_attention_batch",
            "polestar_debug_qkv_fusion")
CODECS = {"fp16": 0, "fp8": 1, "int8": 2, "mxfp4": 3, "int2": 4, "nvfp4": 5}
KERNEL_CLASSES = ("gemm_step", "gemm_entry", "attention", "cluster", "select", "commit", "rows",
                  "attention_entry", "cluster_entry", "rows_entry")


class polestar_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("rope_base", C.c_float), ("rms_eps", C.c_float), ("dtype", C.c_int32),
                ("batch", C.c_int32), ("prompt_len", C.c_int32), ("gen_len", C.c_int32),
                ("block", C.c_int32), ("prefix_win", C.c_int32), ("suffix_win", C.c_int32),
                ("K", C.c_int32), ("topk", C.c_int32), ("tau_upd", C.c_int32), ("hist", C.c_int32),
                ("kmeans_iters", C.c_int32), ("tau_s", C.c_float), ("tau_suf", C.c_float),
                ("alpha", C.c_float), ("seed", C.c_uint64), ("host_offload", C.c_int32)]


class polestar_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
                                          "attn_norm", "ffn_norm")]


class polestar_step_out(C.Structure):
    _fields_ = [("drift", C.c_void_p), ("topk", C.c_void_p), ("selected", C.c_void_p),
                ("labels", C.c_void_p), ("delta", C.c_void_p), ("fire", C.POINTER(C.c_uint8)),
                ("win_len", C.c_int32), ("win_max", C.c_int32)]


class polestar_kernel_stats(C.Structure):
    _fields_ = [("launches", C.c_uint64), ("ms", C.c_double), ("bytes", C.c_double),
                ("flops", C.c_double), ("dropped", C.c_uint64)]


_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libpolestar.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run drift_aware_kv_gb300.build.build() first")
    lib = C.CDLL(path)
    P = C.c_void_p
    lib.polestar_init.argtypes = [C.POINTER(polestar_config), C.POINTER(polestar_layer_weights), P, P,
                                  C.POINTER(P)]
    lib.polestar_calibrate_step.argtypes = [P, P, C.POINTER(C.c_int32), C.c_int32, C.c_int32,
                                            C.POINTER(polestar_step_out)]
    lib.polestar_commit.argtypes = [P, P, C.c_int32, P, P, P]
    lib.polestar_step_host.argtypes = [P, P, C.POINTER(C.c_int32), C.c_int32, C.c_int32, P, C.c_int32, P, P]
    lib.polestar_decode_logits.argtypes = [P, P, P, C.c_int32, P]
    lib.polestar_decode_tokens.argtypes = [P, P, C.c_int32, P, P, P, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
    lib.polestar_embed.argtypes = [P, P, C.c_int32, P, P, P, P]
    lib.polestar_release.argtypes = [P]
    lib.polestar_release.restype = None
    lib.polestar_last_error.argtypes = [P]
    lib.polestar_last_error.restype = C.c_char_p
    lib.polestar_launch_count.argtypes = [P]
    lib.polestar_launch_count.restype = C.c_uint64
    lib.polestar_debug_read.argtypes = [P, C.c_int32, C.c_int32, P, C.c_size_t]
    lib.polestar_debug_write.argtypes = [P, C.c_int32, C.c_int32, P, C.c_size_t]
    lib.polestar_debug_enter_block.argtypes = [P, C.c_int32, C.POINTER(C.c_int32)]
    lib.polestar_debug_gemm.argtypes = [P, C.c_int32, P, C.c_int32, P, C.c_int32, C.c_int32, P, C.c_int32,
                                        C.c_int32, C.c_int32, C.c_int32, P]
    lib.polestar_debug_gemm.restype = C.c_int
    lib.polestar_debug_attention.argtypes = [P, P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, P, P,
                                             P, C.c_int32, C.c_int32, P, P, C.c_int32, P]
    lib.polestar_debug_attention.restype = C.c_int
    lib.polestar_attention_noalloc.argtypes = [P, P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, P, P,
                                               P, C.c_int32, C.c_int32, P, P, P]
    lib.polestar_attention_noalloc.restype = C.c_int
    lib.polestar_debug_kmeans.argtypes = [P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_uint64,
                                          C.c_int32, P, P, P, P, P, P, P]
    lib.polestar_debug_kmeans.restype = C.c_int
    lib.polestar_debug_gemm_choice.argtypes = [C.c_int32, C.c_int32, C.POINTER(C.c_int32), C.c_int32,
                                               C.POINTER(C.c_int32)]
    lib.polestar_debug_gemm_choice.restype = C.c_int
    lib.polestar_codec_bytes.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.POINTER(C.c_int64),
                                         C.POINTER(C.c_int64)]
    lib.polestar_codec_bytes.restype = C.c_int64
    lib.polestar_codec_encode.argtypes = [C.c_int32, P, C.c_int32, C.c_int32, P, P, P, P, P]
    lib.polestar_codec_encode.restype = C.c_int
    lib.polestar_codec_decode.argtypes = [C.c_int32, P, P, C.c_int32, C.c_int32, P, P, P, P]
    lib.polestar_codec_decode.restype = C.c_int
    lib.polestar_debug_stalled_wait.argtypes = [P, C.c_int64]
    lib.polestar_debug_stalled_wait.restype = C.c_int
    lib.polestar_full_forward.argtypes = [P, P]
    lib.polestar_kv_staleness.argtypes = [P, P, C.c_int64, C.c_int32, C.c_int32, C.c_int32, P, P]
    lib.polestar_cache_staleness.argtypes = [P, P, P]
    lib.polestar_profile_begin.argtypes = [P, C.c_int32]
    lib.polestar_profile_end.argtypes = [P, C.POINTER(polestar_kernel_stats), C.c_int32]
    for f in ("polestar_init", "polestar_calibrate_step", "polestar_commit", "polestar_step_host",
              "polestar_debug_read", "polestar_debug_write", "polestar_debug_enter_block",
              "polestar_profile_begin", "polestar_profile_end",
              "polestar_full_forward", "polestar_kv_staleness", "polestar_cache_staleness"):
        getattr(lib, f).restype = C.c_int
    _lib = lib
    return lib


class PolestarError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"polestar status {status}: {msg}")
        self.status = status


def _check(st: int, ctx=None):
    if st != OK:
        msg = load().polestar_last_error(ctx).decode()
        raise PolestarError(st, msg)


def make_config(w, host_offload: bool = False) -> polestar_config:
    """polestar_config from a workload description (attributes as in synth.Workload)."""
    return polestar_config(
        n_layers=w.n_layers, d_model=w.d_model, n_heads=w.n_heads, n_kv_heads=w.n_kv_heads,
        head_dim=w.head_dim, ffn_dim=w.ffn_dim, rope_base=w.rope_base, rms_eps=w.rms_eps,
        dtype=BF16 if w.dtype == "bf16" else FP32, batch=w.batch, prompt_len=w.prompt_len,
        gen_len=w.gen_len, block=w.block, prefix_win=w.prefix_win, suffix_win=w.suffix_win, K=w.K,
        topk=w.topk, tau_upd=w.tau_upd, hist=w.hist, kmeans_iters=w.kmeans_iters, tau_s=w.tau_s,
        tau_suf=w.tau_suf, alpha=w.alpha, seed=w.seed, host_offload=int(host_offload))


class Polestar:
    """Owns one library context.  Weights are torch CUDA tensors (kept alive here)."""

    def __init__(self, workload, layer_weights: List[Dict], stream=None, side_stream=None,
                 host_offload: bool = False):
        import torch
        self.lib = load()
        self.w = workload
        self.weights = layer_weights
        self.cfg = make_config(workload, host_offload)
        arr = (polestar_layer_weights * workload.n_layers)()
        for i, lw in enumerate(layer_weights):
            for name in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down", "attn_norm", "ffn_norm"):
                t = lw[name]
                assert t.is_cuda and t.is_contiguous()
                setattr(arr[i], name, t.data_ptr())
        self._arr = arr
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.side = side_stream if side_stream is not None else self.stream
        ctx = C.c_void_p()
        st = self.lib.polestar_init(C.byref(self.cfg), arr, C.c_void_p(self.stream.cuda_stream),
                                    C.c_void_p(self.side.cuda_stream), C.byref(ctx))
        if st != OK:
            raise PolestarError(st, self.lib.polestar_last_error(None).decode())
        self.ctx = ctx
        self.last_out = polestar_step_out()

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.polestar_release(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def calibrate_step(self, x0, n_unmasked: Sequence[int], block_index: int, block_entry: bool):
        arr = (C.c_int32 * self.w.batch)(*[int(v) for v in n_unmasked])
        _check(self.lib.polestar_calibrate_step(self.ctx, C.c_void_p(x0.data_ptr()), arr, int(block_index),
                                                int(bool(block_entry)), C.byref(self.last_out)), self.ctx)
        return self.last_out

    def commit(self, logits, masked_u8, commit_mask_u8, conf=None):
        _check(self.lib.polestar_commit(self.ctx, C.c_void_p(logits.data_ptr()), int(logits.shape[-1]),
                                        C.c_void_p(masked_u8.data_ptr()),
                                        C.c_void_p(commit_mask_u8.data_ptr()),
                                        C.c_void_p(conf.data_ptr()) if conf is not None else None),
               self.ctx)

    def decode_logits(self, lm_head, final_norm, logits):
        """LM-head logits [batch, 2B, vocab] (fp32, written) of the rows the commit
        gate scores for the step just calibrated (polestar_decode_logits)."""
        _check(self.lib.polestar_decode_logits(self.ctx, C.c_void_p(lm_head.data_ptr()),
                                               C.c_void_p(final_norm.data_ptr()), int(lm_head.shape[0]),
                                               C.c_void_p(logits.data_ptr())), self.ctx)

    def decode_tokens(self, logits, commit_mask_u8, tokens_i32, masked_u8):
        """Greedy tokens into the committed positions after the progress rule
        (polestar_decode_tokens); returns (tokens committed this step, active-block
        positions still masked), one list entry per sequence."""
        b = self.w.batch
        cnt = (C.c_int32 * b)()
        left = (C.c_int32 * b)()
        _check(self.lib.polestar_decode_tokens(self.ctx, C.c_void_p(logits.data_ptr()), int(logits.shape[-1]),
                                               C.c_void_p(commit_mask_u8.data_ptr()),
                                               C.c_void_p(tokens_i32.data_ptr()),
                                               C.c_void_p(masked_u8.data_ptr()), cnt, left), self.ctx)
        return [int(v) for v in cnt], [int(v) for v in left]

    def embed(self, embedding, mask_emb, tokens_i32, masked_u8, x0):
        """Layer-0 inputs x0 [batch, N, d] from the tokens and the mask
        (polestar_embed)."""
        _check(self.lib.polestar_embed(self.ctx, C.c_void_p(embedding.data_ptr()), int(embedding.shape[0]),
                                       C.c_void_p(mask_emb.data_ptr()), C.c_void_p(tokens_i32.data_ptr()),
                                       C.c_void_p(masked_u8.data_ptr()), C.c_void_p(x0.data_ptr())), self.ctx)

    def step_host(self, x0_host, n_unmasked, block_index, block_entry, logits_host, masked_host,
                  commit_host):
        arr = (C.c_int32 * self.w.batch)(*[int(v) for v in n_unmasked])
        _check(self.lib.polestar_step_host(self.ctx, C.c_void_p(x0_host.data_ptr()), arr, int(block_index),
                                           int(bool(block_entry)), C.c_void_p(logits_host.data_ptr()),
                                           int(logits_host.shape[-1]), C.c_void_p(masked_host.data_ptr()),
                                           C.c_void_p(commit_host.data_ptr())), self.ctx)

    def full_forward(self, x0):
        """Recompute the whole K/V cache from x0 by a full-sequence forward
        (polestar_full_forward); nothing else of the context changes."""
        _check(self.lib.polestar_full_forward(self.ctx, C.c_void_p(x0.data_ptr())), self.ctx)

    def staleness(self, ref: "Polestar", out=None):
        """KV-cache staleness E [n_layers, batch, N] (CUDA fp32 tensor) of this
        context's cache against `ref`'s (polestar_cache_staleness)."""
        import torch
        w = self.w
        if out is None:
            out = torch.empty(w.n_layers, w.batch, w.seq_len, dtype=torch.float32, device="cuda")
        _check(self.lib.polestar_cache_staleness(self.ctx, ref.ctx, C.c_void_p(out.data_ptr())), self.ctx)
        return out

    def launch_count(self) -> int:
        return int(self.lib.polestar_launch_count(self.ctx))

    def read(self, which: int, layer: int, shape, dtype):
        """Copy an internal buffer to a new CPU torch tensor of the given shape/dtype."""
        import torch
        out = torch.empty(shape, dtype=dtype)
        _check(self.lib.polestar_debug_read(self.ctx, which, layer, C.c_void_p(out.data_ptr()),
                                            out.numel() * out.element_size()), self.ctx)
        return out

    def write(self, which: int, layer: int, src):
        """Copy a CPU torch tensor into an internal state buffer (polestar_debug_write)."""
        src = src.contiguous()
        _check(self.lib.polestar_debug_write(self.ctx, which, layer, C.c_void_p(src.data_ptr()),
                                             src.numel() * src.element_size()), self.ctx)

    def enter_block(self, block_index: int, cum=None):
        """Host bookkeeping as after block_index's entry step (polestar_debug_enter_block)."""
        arr = (C.c_int32 * self.w.batch)(*(cum or [0] * self.w.batch))
        _check(self.lib.polestar_debug_enter_block(self.ctx, int(block_index), arr), self.ctx)

    def profile_begin(self, capacity: int):
        _check(self.lib.polestar_profile_begin(self.ctx, int(capacity)), self.ctx)

    def profile_end(self) -> Dict[str, dict]:
        arr = (polestar_kernel_stats * len(KERNEL_CLASSES))()
        _check(self.lib.polestar_profile_end(self.ctx, arr, len(KERNEL_CLASSES)), self.ctx)
        return {name: dict(launches=int(a.launches), ms=float(a.ms), bytes=float(a.bytes),
                           flops=float(a.flops), dropped=int(a.dropped))
                for name, a in zip(KERNEL_CLASSES, arr)}


def gemm_path(kernel: int, stages: int = 0, splits: int = 0, bn: int = 0, kpack: int = 0) -> int:
    """`path` of polestar_debug_gemm: kernel 0 CUDA cores, 1 tcgen05 (library's
    choice), 2 row-tiled tcgen05, 3 weight-stationary tcgen05, 7 persistent
    two-SM pair tiles (cta_group::2); stages / splits override the ring depth
    and the cluster K split (kernels 2, 3) or the k-blocks per stage (kernel 7);
    bn the columns per tile of kernels 2 and 7 (a multiple of 16); kpack the
    64-column k-blocks per stage of kernel 2 (1 or 2); 0 = automatic."""
    return kernel | (kpack << 4) | (stages << 8) | (splits << 16) | ((bn // 16) << 24)


def debug_gemm_swiglu(A, Wg, Wu, act, path: int = 1, m_dev=None, stream=None):
    """act = bf16(silu(A Wg^T) * (A Wu^T)) through polestar_debug_gemm_swiglu;
    torch CUDA tensors (A [M, K], Wg/Wu [F, K], act [M, >= F] bf16, unit inner
    stride); path as gemm_path with kernel 1 (library), 2 (row-tiled) or 7
    (two-SM pair tiles)."""
    lib = load()
    lib.polestar_debug_gemm_swiglu.argtypes = [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p,
                                               C.c_int32, C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                               C.c_void_p]
    lib.polestar_debug_gemm_swiglu.restype = C.c_int
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    M, K = A.shape
    F = Wg.shape[0]
    _check(lib.polestar_debug_gemm_swiglu(_ptr(A), A.stride(0), _ptr(Wg), _ptr(Wu), Wg.stride(0), _ptr(act),
                                          act.stride(0), M, _ptr(m_dev) if m_dev is not None else None, F, K,
                                          int(path), C.c_void_p(st.cuda_stream)))


def qkv_fusion(on: int) -> int:
    """Q/K/V projection with the rotary embedding in the pair kernel's epilogue
    (polestar_debug_qkv_fusion): 1 on (default), 0 projection + row kernel;
    returns the previous setting."""
    lib = load()
    lib.polestar_debug_qkv_fusion.argtypes = [C.c_int32]
    lib.polestar_debug_qkv_fusion.restype = C.c_int32
    return int(lib.polestar_debug_qkv_fusion(int(on)))


def attention_impl(impl: int) -> int:
    """Select the attention kernel (polestar_debug_attention_impl): 0 library's
    choice, 1 pipelined mma.sync only, 2 tcgen05 wherever it applies; returns
    the previous setting."""
    lib = load()
    lib.polestar_debug_attention_impl.argtypes = [C.c_int32]
    lib.polestar_debug_attention_impl.restype = C.c_int32
    old = lib.polestar_debug_attention_impl(int(impl))
    if old < 0:
        raise ValueError(f"invalid attention kernel selection {impl}")
    return old


def gemm_choice(M: int, Ns, K: int) -> dict:
    """The projection launch the library picks (polestar_debug_gemm_choice)."""
    lib = load()
    arr = (C.c_int32 * len(Ns))(*[int(n) for n in Ns])
    out = (C.c_int32 * 4)()
    _check(lib.polestar_debug_gemm_choice(int(M), len(Ns), arr, int(K), out))
    return dict(kernel=int(out[0]), bn=int(out[1]), splits=int(out[2]), stages=int(out[3]))


def debug_gemm(A, W, out, path: int, m_dev=None, stream=None, N=None):
    """out = A @ W^T through the library's projection kernel (``path`` as built
    by gemm_path).  torch CUDA tensors, row-major with unit inner stride."""
    import torch
    lib = load()
    M, K = A.shape
    if N is None:
        N = W.shape[0]
    st = stream if stream is not None else torch.cuda.current_stream()
    dt = BF16 if A.dtype == torch.bfloat16 else FP32
    ldw = W.stride(0) if W.dim() == 2 else K
    _check(lib.polestar_debug_gemm(C.c_void_p(A.data_ptr()), A.stride(0), C.c_void_p(W.data_ptr()), ldw,
                                   C.c_void_p(out.data_ptr()), out.stride(0), M,
                                   C.c_void_p(m_dev.data_ptr()) if m_dev is not None else None, N, K, dt,
                                   path, C.c_void_p(st.cuda_stream)))


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def debug_attention(q, kv, H, Hkv, tracked, prev, prev_lse, measure, store, out, kl, stream=None):
    """Row attention + KL on caller tensors (one sequence); see polestar_debug_attention."""
    import torch
    lib = load()
    R = q.shape[0]
    N = kv.shape[0]
    dh = q.shape[1] // H
    st = stream if stream is not None else torch.cuda.current_stream()
    tr = (C.c_uint8 * R)(*[int(bool(v)) for v in tracked])
    dt = BF16 if q.dtype == torch.bfloat16 else FP32
    _check(lib.polestar_debug_attention(_ptr(q), _ptr(kv), N, H, Hkv, dh, R, tr, _ptr(prev), _ptr(prev_lse),
                                        int(measure), int(store), _ptr(out), _ptr(kl), dt,
                                        C.c_void_p(st.cuda_stream)))


def debug_attention_batch(q, kv, H, Hkv, tracked, prev, prev_lse, measure, store, out, kl, stream=None):
    """The same over kv [batch, N, 2, Hkv*dh] and q [batch * R, H*dh] in one
    launch; tracked has R entries (the same rows of every sequence); see
    polestar_debug_attention_batch."""
    import torch
    lib = load()
    batch, N = kv.shape[0], kv.shape[1]
    R = q.shape[0] // batch
    dh = q.shape[1] // H
    st = stream if stream is not None else torch.cuda.current_stream()
    tr = (C.c_uint8 * R)(*[int(bool(v)) for v in tracked])
    dt = BF16 if q.dtype == torch.bfloat16 else FP32
    _check(lib.polestar_debug_attention_batch(_ptr(q), _ptr(kv), batch, N, H, Hkv, dh, R, tr, _ptr(prev),
                                              _ptr(prev_lse), int(measure), int(store), _ptr(out), _ptr(kl), dt,
                                              C.c_void_p(st.cuda_stream)))


def debug_kmeans(Hw, K, iters, seed, block, stream=None):
    """Spherical K-means + residual NVFP4 of P problems Hw [P, nw, d] (fp32, CUDA).
    Returns dict of CUDA tensors labels, z, csum, anchor, codes, scales."""
    import torch
    lib = load()
    P_, nw, d = Hw.shape
    dev = Hw.device
    out = dict(labels=torch.empty(P_, nw, dtype=torch.uint8, device=dev),
               z=torch.empty(P_, K, d, device=dev), csum=torch.empty(P_, K, d, device=dev),
               anchor=torch.empty(P_, K, d, device=dev),
               codes=torch.empty(P_, nw, d // 2, dtype=torch.uint8, device=dev),
               scales=torch.empty(P_, nw, d // 16, dtype=torch.uint8, device=dev))
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.polestar_debug_kmeans(_ptr(Hw), P_, nw, d, K, iters, int(seed), int(block), _ptr(out["labels"]),
                                     _ptr(out["z"]), _ptr(out["csum"]), _ptr(out["anchor"]),
                                     _ptr(out["codes"]), _ptr(out["scales"]), C.c_void_p(st.cuda_stream)))
    return out


def attention_noalloc(q, kv, H, Hkv, tracked_dev, prev, prev_lse, measure, store, out, kl, stream=None):
    """Row attention + KL drift using only the library's fixed device scratch
    (no allocation); `tracked_dev` is a CUDA uint8 tensor [R] or None."""
    import torch
    lib = load()
    R = q.shape[0]
    N = kv.shape[0]
    dh = q.shape[1] // H
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.polestar_attention_noalloc(_ptr(q), _ptr(kv), N, H, Hkv, dh, R, _ptr(tracked_dev), _ptr(prev),
                                          _ptr(prev_lse), int(measure), int(store), _ptr(out), _ptr(kl),
                                          C.c_void_p(st.cuda_stream)))


def kv_staleness(kv, kv_ref, n_kv_heads: int, E=None, stream=None):
    """App. C.2 staleness of the rows of two caches laid out [rows, 2, Hkv*dh]
    (CUDA tensors, fp32 or bf16, any leading shape) through polestar_kv_staleness;
    returns E [rows] fp32 (CUDA)."""
    import torch
    lib = load()
    assert kv.shape == kv_ref.shape and kv.dtype == kv_ref.dtype
    assert kv.is_contiguous() and kv_ref.is_contiguous()
    kvdim = kv.shape[-1]
    rows = kv.numel() // (2 * kvdim)
    dh = kvdim // n_kv_heads
    if E is None:
        E = torch.empty(rows, dtype=torch.float32, device=kv.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    dt = BF16 if kv.dtype == torch.bfloat16 else FP32
    _check(lib.polestar_kv_staleness(_ptr(kv), _ptr(kv_ref), rows, int(n_kv_heads), int(dh), dt, _ptr(E),
                                     C.c_void_p(st.cuda_stream)))
    return E


def codec_bytes(fmt: str, rows: int, d: int):
    """(code bytes, scale bytes) of `rows` rows of width d (polestar_codec_bytes)."""
    lib = load()
    cb, sb = C.c_int64(), C.c_int64()
    if lib.polestar_codec_bytes(CODECS[fmt], int(rows), int(d), C.byref(cb), C.byref(sb)) < 0:
        raise PolestarError(ERR_INVALID_ARG, f"codec {fmt}: unsupported size {rows} x {d}")
    return int(cb.value), int(sb.value)


def codec_encode(fmt: str, h, anchors=None, labels=None, stream=None):
    """Encode h [rows, d] fp32 (CUDA) in a storage format, as the residual
    against anchors[labels] when given; returns (codes, scales) uint8 tensors."""
    import torch
    lib = load()
    rows, d = h.shape
    nc, ns = codec_bytes(fmt, rows, d)
    codes = torch.empty(max(nc, 16), dtype=torch.uint8, device=h.device)
    scales = torch.empty(max(ns, 16), dtype=torch.uint8, device=h.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.polestar_codec_encode(CODECS[fmt], _ptr(h), rows, d, _ptr(anchors) if anchors is not None else None,
                                     _ptr(labels) if labels is not None else None, _ptr(codes), _ptr(scales),
                                     C.c_void_p(st.cuda_stream)))
    return codes[:nc], scales[:ns]


def codec_decode(fmt: str, codes, scales, rows: int, d: int, anchors=None, labels=None, out=None, stream=None):
    """Decode (codes, scales) of codec_encode back to fp32 [rows, d] (CUDA)."""
    import torch
    lib = load()
    if out is None:
        out = torch.empty(rows, d, dtype=torch.float32, device=codes.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib.polestar_codec_decode(CODECS[fmt], _ptr(codes), _ptr(scales), rows, d,
                                     _ptr(anchors) if anchors is not None else None,
                                     _ptr(labels) if labels is not None else None, _ptr(out),
                                     C.c_void_p(st.cuda_stream)))
    return out
