"""Seeded synthetic workloads for the Polestar calibration + commit path.

This module only *draws inputs*: random-init weights, the per-step layer-0 hidden
states of a masked-diffusion trajectory, the mask state and per-token logits.  It
holds none of the method's arithmetic (no normalisation, attention, clustering,
quantisation, drift or gating).  Both the CUDA library's tests/benchmark and the
CPU oracle receive the very same tensors from here.

Workload shapes follow the model families the Polestar paper evaluates
("Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs", §5.1 Experimental Setup: LLaDA-8B-Instruct and
Dream-7B-Instruct, generation lengths 256/512, block size B = 32, Table 5 default
hyper-parameters).  Weights are random N(0, 0.02); no trained checkpoint and no
dataset item is used.

Trajectory recipe (one denoising step = one call of ``Trajectory.next_step``):
  * prompt rows of the layer-0 hidden states are N(0, 1); generated rows start at
    one fixed N(0, 1) "mask embedding";
  * between steps every row of the active block's local window
    (2B prefix + B suffix) gets N(0, 0.05) noise, and a random fraction of those
    rows (10 %, or a per-sequence fraction for the batched workloads) gets an extra
    N(0, 0.3) kick -- the perturbations accumulate;
  * between steps 3-6 (4-6 where every step must refresh) still-masked tokens of
    the active block flip to the embedding of a random vocabulary id;
  * a block ends when every sequence of the batch has unmasked all of its tokens;
    the next step is then the entry of the next block;
  * logits for the 2B rows (active block + suffix block) are N(0, 1) with the
    row maximum raised so that its softmax probability equals a target
    c ~ U(0.5, 0.99).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

MASK64 = (1 << 64) - 1


def _mix64(x: int) -> int:
    """splitmix64 finaliser (Steele, Lea & Flood 2014); used only to derive seeds."""
    x = (x + 0x9E3779B97F4A7C15) & MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & MASK64
    return x ^ (x >> 31)


def derive_seed(*parts: int) -> int:
    """Fold integers into one 63-bit torch seed."""
    h = 0x243F6A8885A308D3
    for p in parts:
        h = _mix64(h ^ (int(p) & MASK64))
    return h & ((1 << 63) - 1)


@dataclasses.dataclass
class Workload:
    """Model shape + Polestar hyper-parameters of one synthetic workload."""

    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    rope_base: float
    rms_eps: float
    dtype: str  # "fp32" or "bf16": storage type of weights, inputs, K/V cache
    batch: int
    prompt_len: int
    gen_len: int
    vocab: int
    embed_vocab: int  # ids a flipped token can take
    block: int = 32
    prefix_win: int = 64
    suffix_win: int = 32
    K: int = 8
    topk: int = 4
    tau_upd: int = 3
    hist: int = 5
    kmeans_iters: int = 10
    tau_s: float = 0.9
    tau_suf: float = 0.9
    alpha: float = 10.0
    seed: int = 0
    flips: tuple = (3, 6)
    extra_frac: tuple = (0.1, 0.1)  # U(lo, hi) per sequence; (0.1, 0.1) = fixed 10 %
    n_steps: Optional[int] = None  # None: run until every block is decoded
    norm_gain_std: float = 0.0  # RMSNorm gains 1 + N(0, std) (0: gains 1, as in the benchmark shapes)
    qk_std: float = 0.02  # std of the query/key projections
    vo_std: float = 0.02  # std of the value/output projections
    lm_std: Optional[float] = None  # LM head std for closed-loop decoding (None: 4 / sqrt(d))

    @property
    def seq_len(self) -> int:
        return self.prompt_len + self.gen_len

    @property
    def n_blocks(self) -> int:
        return self.gen_len // self.block

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _llada(name, **kw):
    base = dict(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128,
                ffn_dim=12288, rope_base=500000.0, rms_eps=1e-5, dtype="bf16",
                vocab=126464, embed_vocab=126464)
    base.update(kw)
    return Workload(name=name, **base)


WORKLOADS: Dict[str, Workload] = {
    # single decoder layer in fp32: 64 prompt + 128 generated tokens, 16 steps
    "tiny_l1_d256_fp32": Workload(
        name="tiny_l1_d256_fp32", n_layers=1, d_model=256, n_heads=4, n_kv_heads=4,
        head_dim=64, ffn_dim=688, rope_base=10000.0, rms_eps=1e-6, dtype="fp32",
        batch=1, prompt_len=64, gen_len=128, vocab=512, embed_vocab=512, n_steps=16),
    # LLaDA-8B shape, batch 1, prompt 512, generation 256
    "llada8b_p512_g256_b1": _llada("llada8b_p512_g256_b1", batch=1, prompt_len=512,
                                   gen_len=256),
    # LLaDA-8B shape, batch 8, generation 512, per-sequence kick fraction U(0.05,0.2)
    "llada8b_p512_g512_b8": _llada("llada8b_p512_g512_b8", batch=8, prompt_len=512,
                                   gen_len=512, extra_frac=(0.05, 0.2)),
    # Dream-7B shape (GQA 28/4), batch 4
    "dream7b_p512_g256_b4": Workload(
        name="dream7b_p512_g256_b4", n_layers=28, d_model=3584, n_heads=28, n_kv_heads=4,
        head_dim=128, ffn_dim=18944, rope_base=1000000.0, rms_eps=1e-6, dtype="bf16",
        batch=4, prompt_len=512, gen_len=256, vocab=152064, embed_vocab=152064),
    # LLaDA-8B stress: batch 32, prompt 1024, generation 1024, refresh every step
    "llada8b_p1024_g1024_b32": _llada("llada8b_p1024_g1024_b32", batch=32,
                                      prompt_len=1024, gen_len=1024, flips=(4, 6),
                                      extra_frac=(0.05, 0.3)),
    # small bf16 stacks that the CPU oracle finishes in seconds (parity cases)
    "mini_l2_d512_bf16": Workload(
        name="mini_l2_d512_bf16", n_layers=2, d_model=512, n_heads=4, n_kv_heads=4,
        head_dim=128, ffn_dim=1376, rope_base=500000.0, rms_eps=1e-5, dtype="bf16",
        batch=2, prompt_len=64, gen_len=128, vocab=2048, embed_vocab=2048, n_steps=14,
        extra_frac=(0.05, 0.2)),
    # closed-loop decoding (embedding -> layer stack -> LM head -> gate -> tokens):
    # attention weights raised so that positions differ, LM head scaled so that
    # confidences spread over the gate's branches
    "loop_l1_d256_fp32": Workload(
        name="loop_l1_d256_fp32", n_layers=1, d_model=256, n_heads=4, n_kv_heads=4,
        head_dim=64, ffn_dim=688, rope_base=10000.0, rms_eps=1e-6, dtype="fp32",
        batch=2, prompt_len=64, gen_len=128, vocab=512, embed_vocab=512,
        qk_std=0.16, vo_std=0.12, lm_std=0.5),
    "loop_l2_d512_bf16": Workload(
        name="loop_l2_d512_bf16", n_layers=2, d_model=512, n_heads=4, n_kv_heads=4,
        head_dim=128, ffn_dim=1376, rope_base=500000.0, rms_eps=1e-5, dtype="bf16",
        batch=2, prompt_len=64, gen_len=128, vocab=2048, embed_vocab=2048,
        qk_std=0.1, vo_std=0.08, lm_std=0.35),
    "mini_gqa_l2_d448_bf16": Workload(
        name="mini_gqa_l2_d448_bf16", n_layers=2, d_model=448, n_heads=7, n_kv_heads=1,
        head_dim=64, ffn_dim=1184, rope_base=1000000.0, rms_eps=1e-6, dtype="bf16",
        batch=1, prompt_len=96, gen_len=96, vocab=1000, embed_vocab=1000, n_steps=12),
}


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


def _randn(shape, seed: int, device, std: float = 1.0) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        out.mul_(std)
    return out


WEIGHT_NAMES = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def weight_shapes(w: Workload) -> Dict[str, tuple]:
    d, hq, hk, F = w.d_model, w.n_heads * w.head_dim, w.n_kv_heads * w.head_dim, w.ffn_dim
    return {"wq": (hq, d), "wk": (hk, d), "wv": (hk, d), "wo": (d, hq),
            "w_gate": (F, d), "w_up": (F, d), "w_down": (d, F)}


def make_layer_weights(w: Workload, layer: int, device="cpu") -> Dict[str, torch.Tensor]:
    """Random-init weights of one decoder layer: matrices N(0, 0.02) (query/key
    and value/output projections N(0, qk_std) / N(0, vo_std): the closed-loop
    decoding variants raise them so that attention, not the residual stream
    alone, shapes each position's output), norm gains 1 (or 1 + N(0,
    norm_gain_std), distinct per norm and layer, in test variants).

    Matrices are row-major [out_features, in_features] (y = x @ W^T)."""
    dt = torch_dtype(w)
    out = {}
    stds = {"wq": w.qk_std, "wk": w.qk_std, "wv": w.vo_std, "wo": w.vo_std}
    for i, (name, shape) in enumerate(weight_shapes(w).items()):
        out[name] = _randn(shape, derive_seed(w.seed, 0x57, layer, i), device, stds.get(name, 0.02)).to(dt)
    if w.norm_gain_std > 0:
        # distinct, non-unit gains for the two norms of every layer (test variant)
        out["attn_norm"] = (1.0 + _randn((w.d_model,), derive_seed(w.seed, 0x6A1, layer), device,
                                          w.norm_gain_std)).to(dt)
        out["ffn_norm"] = (1.0 + _randn((w.d_model,), derive_seed(w.seed, 0x6A2, layer), device,
                                         w.norm_gain_std)).to(dt)
    else:
        out["attn_norm"] = torch.ones(w.d_model, dtype=dt, device=device)
        out["ffn_norm"] = torch.ones(w.d_model, dtype=dt, device=device)
    return out


def make_weights(w: Workload, device="cpu") -> List[Dict[str, torch.Tensor]]:
    return [make_layer_weights(w, l, device) for l in range(w.n_layers)]


def make_decode_weights(w: Workload, device="cpu", lm_std: Optional[float] = None) -> Dict[str, torch.Tensor]:
    """Random-init tensors around the layer stack for closed-loop decoding, in the
    storage dtype: token embedding [V, d] N(0, 1) (the scale of the trajectory's
    prompt rows), the [MASK] embedding [d] (the trajectory's mask embedding), the
    LM head [V, d] N(0, lm_std) and the final norm gain [d] (1, or
    1 + N(0, norm_gain_std)).  lm_std defaults to 4 / sqrt(d): a unit-RMS row then
    gives logits of standard deviation 4, whose max-softmax confidences spread
    over (0, 1) at the parity vocabularies, so the gate's branches all occur."""
    dt = torch_dtype(w)
    V, d = w.vocab, w.d_model
    if lm_std is None:
        lm_std = w.lm_std if w.lm_std is not None else 4.0 / math.sqrt(d)
    out = {
        "embed": _randn((V, d), derive_seed(w.seed, 0xE3B), device).to(dt),
        "mask_emb": _randn((d,), derive_seed(w.seed, 0x3A5), "cpu").to(device).to(dt),
        "lm_head": _randn((V, d), derive_seed(w.seed, 0x1A4), device, lm_std).to(dt),
    }
    if w.norm_gain_std > 0:
        out["final_norm"] = (1.0 + _randn((d,), derive_seed(w.seed, 0x6A3), device, w.norm_gain_std)).to(dt)
    else:
        out["final_norm"] = torch.ones(d, dtype=dt, device=device)
    return out


def make_prompt(w: Workload, device="cpu"):
    """Prompt tokens U[0, V) per sequence, generated positions masked: returns
    (tokens [batch, N] int32 with 0 at masked positions, masked [batch, N] bool)."""
    N = w.seq_len
    g = torch.Generator(device="cpu").manual_seed(derive_seed(w.seed, 0x9A0))
    tokens = torch.zeros(w.batch, N, dtype=torch.int32)
    tokens[:, : w.prompt_len] = torch.randint(0, w.vocab, (w.batch, w.prompt_len), generator=g, dtype=torch.int32)
    masked = torch.zeros(w.batch, N, dtype=torch.bool)
    masked[:, w.prompt_len:] = True
    return tokens.to(device), masked.to(device)


def block_span(w: Workload, b: int):
    start = w.prompt_len + b * w.block
    return start, start + w.block


def window_positions(w: Workload, b: int) -> List[int]:
    """Positions of the 2B-prefix + B-suffix local window of block b, clipped to the
    sequence (prefix [start-2B, start), suffix [end, end+B))."""
    start, end = block_span(w, b)
    pre = [p for p in range(start - w.prefix_win, start) if p >= 0]
    suf = [p for p in range(end, end + w.suffix_win) if p < w.seq_len]
    return pre + suf


class Trajectory:
    """Seeded synthetic masked-diffusion trajectory (inputs of every step).

    device "cpu" (the default) draws every value from per-sequence CPU generators:
    the inputs the CPU oracle and the parity tests share.  Another device draws
    the same recipe from per-sequence generators of that device (other values,
    same distributions), which keeps the large workloads' inputs -- a gigabyte
    of logits per step at batch 32 -- off the host in the throughput benchmark."""

    def __init__(self, w: Workload, device="cpu"):
        self.w = w
        self.dev = torch.device(device)
        N, d = w.seq_len, w.d_model
        self.gens = []
        for s in range(w.batch):
            g = torch.Generator(device=self.dev)
            g.manual_seed(derive_seed(w.seed, 0x5E0, s))
            self.gens.append(g)
        self.mask_emb = _randn((d,), derive_seed(w.seed, 0x3A5), "cpu").to(self.dev)
        self.X = torch.empty(w.batch, N, d, dtype=torch.float32, device=self.dev)
        self.masked = torch.zeros(w.batch, N, dtype=torch.bool, device=self.dev)
        self.frac = []
        for s in range(w.batch):
            g = self.gens[s]
            self.X[s, : w.prompt_len] = torch.randn(w.prompt_len, d, generator=g, device=self.dev)
            self.X[s, w.prompt_len:] = self.mask_emb
            self.masked[s, w.prompt_len:] = True
            lo, hi = w.extra_frac
            self.frac.append(lo + (hi - lo) * float(torch.rand((), generator=g, device=self.dev)))
        self.block = 0
        self.block_entry = True
        self.n_unmasked = [0] * w.batch
        self.t = 0
        self.done = False

    def _vocab_row(self, vid: int) -> torch.Tensor:
        return _randn((self.w.d_model,), derive_seed(self.w.seed, 0xE3B, vid), "cpu").to(self.dev)

    def _logits(self, s: int):
        """[2B, V] fp32 logits with row max-prob c ~ U(0.5, 0.99); returns (logits, c)."""
        w, g = self.w, self.gens[s]
        rows = 2 * w.block
        dev = self.dev
        lg = torch.randn(rows, w.vocab, generator=g, dtype=torch.float32, device=dev)
        c = 0.5 + 0.49 * torch.rand(rows, generator=g, dtype=torch.float64, device=dev)
        a = lg.argmax(dim=1)
        l64 = lg.double()
        ar = torch.arange(rows, device=dev)
        l64[ar, a] = -math.inf
        rest = torch.logsumexp(l64, dim=1)
        lg[ar, a] = (torch.log(c / (1 - c)) + rest).float()
        return lg, c

    def next_step(self) -> Optional[dict]:
        """Inputs of the next denoising step, then advance the synthetic state."""
        w = self.w
        if self.done or (w.n_steps is not None and self.t >= w.n_steps):
            return None
        logits, targets = [], []
        for s in range(w.batch):
            lg, c = self._logits(s)
            logits.append(lg)
            targets.append(c)
        step = dict(
            t=self.t,
            block_index=self.block,
            block_entry=self.block_entry,
            n_unmasked=list(self.n_unmasked),
            x0=self.X.clone(),
            masked=self.masked.clone(),
            logits=torch.stack(logits),
            conf_target=torch.stack(targets),
        )
        self._advance()
        return step

    def _advance(self):
        w = self.w
        start, end = block_span(w, self.block)
        dev = self.dev
        win = torch.tensor(window_positions(w, self.block), dtype=torch.long, device=dev)
        lo, hi = w.flips
        for s in range(w.batch):
            g = self.gens[s]
            nw = len(win)
            self.X[s, win] += 0.05 * torch.randn(nw, w.d_model, generator=g, device=dev)
            kick = torch.rand(nw, generator=g, device=dev) < self.frac[s]
            if bool(kick.any()):
                rows = win[kick]
                self.X[s, rows] += 0.3 * torch.randn(len(rows), w.d_model, generator=g, device=dev)
            still = torch.nonzero(self.masked[s, start:end]).flatten() + start
            m = int(torch.randint(lo, hi + 1, (), generator=g, device=dev))
            m = min(m, len(still))
            if m > 0:
                pick = still[torch.randperm(len(still), generator=g, device=dev)[:m]]
                ids = torch.randint(0, w.embed_vocab, (m,), generator=g, device=dev)
                for p, vid in zip(pick.tolist(), ids.tolist()):
                    self.X[s, p] = self._vocab_row(vid)
                    self.masked[s, p] = False
            self.n_unmasked[s] = m
        self.t += 1
        if not bool(self.masked[:, start:end].any()):
            if self.block + 1 < w.n_blocks:
                self.block += 1
                self.block_entry = True
            else:
                self.done = True
        else:
            self.block_entry = False
