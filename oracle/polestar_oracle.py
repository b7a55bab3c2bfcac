"""CPU oracle of the Polestar calibration + commit path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` may import this module.  It shares no code with the
CUDA library (``drift_aware_kv_gb300/csrc``) and never imports it.

Plain, slow, obviously-correct numpy in float64 (the pages fix no precision; float64
is at least as strict as the single-precision oracle the build plan names, and
numpy's BLAS may use several threads -- the timed legs report the thread count).
Citations name the paper
"Polestar: Drift-Aware Cache Calibration and Token Commitment for Efficient
Inference of Diffusion LLMs" (arXiv 2607.14107) by section / equation / Algorithm 1.

Storage precision.  Where the library stores a tensor in bf16 (workload dtype
"bf16": weights, layer-0 inputs, GEMM A-operands, Q/K/V) the oracle rounds the
same value to bf16 at the same point (``_store``); all other arithmetic is
float64.  Decisions that the method takes on a fp32 quantity (the NVFP4 scale and
code choice, Appendix C.3) are taken here in IEEE fp32 as well.

Parity status per function (what pins it, see tests/test_oracle_*.py):
  number formats   pinned (torch float8_e4m3fn table / RNE, E2M1 grid of the format)
  rmsnorm / rope   pinned (torch rms_norm, complex-rotation form)
  decoder layer    pinned (qkv -> attention -> O + residual -> RMSNorm -> SwiGLU -> down +
                   residual equals per-element loops, distinct non-unit norm gains; silu vs torch)
  attention / KL   pinned (torch sdpa, scipy rel_entr, KL(a||a)=0, Pinsker bound)
  spherical kmeans pinned (brute force on tiny inputs, unit norms, objective monotone)
  top-k            pinned (full sort)
  NVFP4 residual   pinned (grid membership, round trip, error bound, Table 11 ordering)
  commit gate      pinned (worked value c=0.8 -> tau_d=0.1, limits; closed-form cases of the
                   current-block, history, suffix and block-entry rules)
  centroid update  pinned (exact cache: layer-0 member sums equal the closed form)
  proxy query      pinned (no rotary: equals the position-0 token's query)
  trigger          pinned (closed-form refresh sequences of the tau_upd rule on the engine itself,
                   restart at block entry)
  confidence       pinned (generator's target max-probability)
  sparse refresh   pinned (k = K, exact cache: equals the block-entry forward)
  KV staleness     pinned (closed forms: 0 on itself, 2 on the negation, per-head rotation)
  full forward     pinned (equals the even block-entry forward; zero staleness after it)
  whole step       parity unpinned beyond the pins above (no worked example exists)
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

MASK64 = (1 << 64) - 1

# --------------------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------------------


def to_f32(x):
    """Round float64 values to IEEE binary32 (round-to-nearest-even), back to float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def to_bf16(x):
    """Round to bfloat16, nearest-even, through the binary32 bit pattern."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


# E2M1 (1 sign, 2 exponent, 1 mantissa bit; App. C.3): magnitudes by 3-bit code
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_value(byte):
    """Decode an FP8 E4M3 byte (bias 7, no infinities, 0x7F/0xFF = NaN)."""
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = sign * (1.0 + m / 8.0) * np.power(2.0, e - 7.0)
    sub = sign * (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, v)


def e4m3_round(v):
    """Round non-negative values to E4M3, nearest-even, saturating at 448.

    Returns (value, byte, margin) where margin is the distance (in units of the
    local quantum) between v and the nearest rounding midpoint."""
    v = np.asarray(v, dtype=np.float64)
    assert np.all(v >= 0)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    e = np.maximum(e, -6.0)  # below 2^-6 the quantum is fixed (subnormals)
    quantum = np.power(2.0, e - 3.0)
    q = v / quantum
    n = np.floor(q)
    frac = q - n
    up = (frac > 0.5) | ((frac == 0.5) & (np.mod(n, 2) == 1))
    n = n + up
    val = np.minimum(n * quantum, 448.0)
    margin = np.abs(frac - 0.5)
    margin = np.where(v >= 448.0, np.inf, margin)
    # encode the byte
    with np.errstate(divide="ignore"):
        ee = np.floor(np.log2(np.where(val > 0, val, 1.0)))
    is_norm = val >= 2.0 ** -6
    exp_field = np.where(is_norm, ee + 7, 0)
    mant = np.where(is_norm, val / np.power(2.0, ee) * 8 - 8, val / 2.0 ** -9)
    byte = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    byte = np.where(val == 0, 0, byte)
    return val, byte.astype(np.uint8), margin


def e2m1_round(x):
    """Round fp32 values to E2M1 codes (bit 3 = sign, bits 0-2 = magnitude index),
    nearest with ties to the even index, saturating at 6.

    Returns (codes, margin) with margin = |x| distance to the nearest rounding
    midpoint (inf above the saturation threshold)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    mids = (E2M1_VALUES[:-1] + E2M1_VALUES[1:]) / 2.0  # 0.25 .. 5
    idx = np.zeros(a.shape, dtype=np.int64)
    for i, m in enumerate(mids):
        lower, upper = i, i + 1
        # strictly above the midpoint -> upper; exactly on it -> the even index
        go_up = (a > m) | ((a == m) & (upper % 2 == 0))
        idx = np.where(go_up, upper, idx)
    margin = np.min(np.abs(a[..., None] - mids), axis=-1)
    margin = np.where(a > 6.0, np.inf, margin)
    sign = np.signbit(x).astype(np.int64)
    return (sign << 3 | idx).astype(np.uint8), margin


def e2m1_value(code):
    c = np.asarray(code, dtype=np.int64)
    return np.where(c & 8, -1.0, 1.0) * E2M1_VALUES[c & 7]


def nvfp4_encode(r):
    """NVFP4 encoding of residual rows (App. C.3): groups of 16 channels, one E4M3
    scale s = RNE_e4m3(amax/6) per group, elements q = RNE_e2m1(r/s); all-zero
    groups (s == 0) give +0 codes.  Divisions are IEEE fp32, as in the library.

    r: [rows, d] fp32-valued.  Returns (codes [rows, d] u8, scale bytes [rows, d/16],
    margin [rows, d])."""
    r32 = np.asarray(r, dtype=np.float64).astype(np.float32)
    rows, d = r32.shape
    g = r32.reshape(rows, d // 16, 16)
    amax = np.max(np.abs(g), axis=-1)
    sval, sbyte, smargin = e4m3_round((amax / np.float32(6.0)).astype(np.float64))
    s32 = sval.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        xs = (g / s32[..., None]).astype(np.float64)
    xs = np.where(s32[..., None] == 0, 0.0, xs)
    codes, emargin = e2m1_round(xs)
    codes = np.where(s32[..., None] == 0, 0, codes).astype(np.uint8)
    emargin = np.where(s32[..., None] == 0, np.inf, emargin)
    margin = np.minimum(emargin, smargin[..., None])
    return codes.reshape(rows, d), sbyte.reshape(rows, d // 16), margin.reshape(rows, d)


def nvfp4_decode(codes, sbytes):
    """Decoded residual values (fp32-valued): e2m1(q) * e4m3(s)."""
    rows, d = codes.shape
    s = e4m3_value(sbytes).reshape(rows, d // 16, 1)
    v = e2m1_value(codes).reshape(rows, d // 16, 16) * s
    return to_f32(v.reshape(rows, d))


# --------------------------------------------------------------------------------------
# seeded K-means initialisation (splitmix64 + Fisher-Yates)
# --------------------------------------------------------------------------------------


def splitmix64_stream(state: int):
    """splitmix64 (Steele, Lea & Flood 2014, Vigna's reference form) as a generator."""
    x = state & MASK64
    while True:
        x = (x + 0x9E3779B97F4A7C15) & MASK64
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def kmeans_init(seed: int, seq: int, block: int, layer: int, n: int, K: int) -> List[int]:
    """First K entries of a Fisher-Yates (Durstenfeld) permutation of range(n), drawn
    from splitmix64 started at seed ^ seq<<40 ^ block<<20 ^ layer."""
    gen = splitmix64_stream(seed ^ (seq << 40) ^ (block << 20) ^ layer)
    perm = list(range(n))
    for i in range(n - 1, 0, -1):
        j = next(gen) % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    return perm[:K]


# --------------------------------------------------------------------------------------
# model pieces (LLaDA / Dream decoder layer: RMSNorm, QKV, RoPE, attention, SwiGLU)
# --------------------------------------------------------------------------------------


def rmsnorm(x, gain, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * gain


def rope(x, pos, base):
    """Rotate-half rotary embedding; x: [rows, heads, dh], pos: [rows]."""
    dh = x.shape[-1]
    half = dh // 2
    inv = base ** (-np.arange(half, dtype=np.float64) * 2.0 / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def logsumexp(s, axis=-1):
    m = np.max(s, axis=axis, keepdims=True)
    return (m + np.log(np.sum(np.exp(s - m), axis=axis, keepdims=True))).squeeze(axis)


def kl_div(s, lse, s_prev, lse_prev):
    """KL(P || Q) per row of scores, with P = softmax(s), Q = softmax(s_prev)
    (Eq. 4): sum_j p_j (log p_j - log q_j)."""
    logp = s - lse[..., None]
    logq = s_prev - lse_prev[..., None]
    return np.sum(np.exp(logp) * (logp - logq), axis=-1)


def topk_clusters(D, k):
    """The k largest drifts, ties to the lower cluster id (§4.1, Algorithm 1 TopK).

    Returns (ids in rank order, relative gap between the k-th and (k+1)-th)."""
    order = sorted(range(len(D)), key=lambda c: (-D[c], c))
    ids = order[:k]
    if k < len(D):
        a, b = D[order[k - 1]], D[order[k]]
        margin = (a - b) / max(abs(a), 1e-300)
    else:
        margin = math.inf
    return ids, margin


def spherical_kmeans(H, K, iters, init_idx):
    """Spherical K-means (§4.1 "Cluster and Quantize Hidden States").

    Rows are projected to the unit sphere; each iteration assigns every row to the
    centroid of largest cosine (ties to the lower id) and resets each centroid to
    the normalised sum of its members; an empty cluster keeps its centroid.
    Returns labels (last assignment), z (last update), s (member sums; z for an
    empty cluster), A (raw member means, the residual anchors) and the smallest
    best-vs-second cosine gap seen over all assignments."""
    H = np.asarray(H, dtype=np.float64)
    X = H / np.linalg.norm(H, axis=1, keepdims=True)
    z = X[list(init_idx)].copy()
    s = z.copy()
    labels = np.zeros(len(X), dtype=np.int64)
    min_gap = math.inf
    for _ in range(iters):
        cos = X @ z.T
        labels = np.argmax(cos, axis=1)
        srt = np.sort(cos, axis=1)
        if K > 1:
            min_gap = min(min_gap, float(np.min(srt[:, -1] - srt[:, -2])))
        for c in range(K):
            mem = labels == c
            if np.any(mem):
                s[c] = X[mem].sum(axis=0)
                z[c] = s[c] / np.linalg.norm(s[c])
            else:
                s[c] = z[c]
    A = np.zeros_like(z)
    for c in range(K):
        mem = labels == c
        if np.any(mem):
            A[c] = H[mem].mean(axis=0)
    return labels, z, s, to_f32(A), min_gap


def confidence(logits):
    """Max softmax probability of each row (§2 confidence score; the synthetic
    vocabulary has no [MASK] id to exclude)."""
    l = np.asarray(logits, dtype=np.float64)
    m = np.max(l, axis=-1, keepdims=True)
    return 1.0 / np.sum(np.exp(l - m), axis=-1)


def drift_threshold(c, tau_s, alpha):
    """Confidence-conditioned dynamic threshold tau_d = alpha (tau_s - c)^2 (§4.2)."""
    return alpha * (tau_s - c) ** 2


def kv_staleness(kv, kv_ref, n_kv_heads, head_dim):
    """KV-cache staleness of App. C.2 for every row of two caches.

    kv, kv_ref: rows of K then V, [rows, 2, n_kv_heads * head_dim] or any shape
    with the same element order (e.g. [L, batch, N, 2, Hkv, dh]).  For each row,
    the cosine similarity of the cached and the recomputed vector is taken per KV
    head and averaged over heads, separately for K and for V; the staleness is one
    minus the mean of those two averages.  A zero vector has no direction: two zero
    vectors count as identical (cos 1), a zero against a non-zero vector as
    orthogonal (cos 0).  Returns E [rows]."""
    a = np.asarray(kv, dtype=np.float64).reshape(-1, 2, n_kv_heads, head_dim)
    b = np.asarray(kv_ref, dtype=np.float64).reshape(-1, 2, n_kv_heads, head_dim)
    dot = np.sum(a * b, axis=-1)
    na = np.sum(a * a, axis=-1)
    nb = np.sum(b * b, axis=-1)
    both = (na > 0) & (nb > 0)
    cos = np.where(both, dot / np.sqrt(np.where(both, na * nb, 1.0)),
                   np.where((na == 0) & (nb == 0), 1.0, 0.0))
    per_kv = cos.mean(axis=-1)  # [..., 2]: head-averaged cosine of K and of V
    return 1.0 - 0.5 * (per_kv[..., 0] + per_kv[..., 1])


# --------------------------------------------------------------------------------------
# the engine: block entry, within-block calibration step, commit gate
# --------------------------------------------------------------------------------------


@dataclass
class SeqState:
    kv: List[np.ndarray]  # per layer [N, 2, Hkv, dh]
    labels: List[np.ndarray] = field(default_factory=list)
    z: List[np.ndarray] = field(default_factory=list)
    s: List[np.ndarray] = field(default_factory=list)
    A: List[np.ndarray] = field(default_factory=list)
    codes: List[np.ndarray] = field(default_factory=list)
    sbytes: List[np.ndarray] = field(default_factory=list)
    code_margin: List[np.ndarray] = field(default_factory=list)
    P_prev: List[tuple] = field(default_factory=list)  # per layer (scores [K,H,N], lse [K,H])
    A_prev: Optional[tuple] = None  # last layer, active rows (scores [B,H,N], lse [B,H])
    theta: List[List[float]] = field(default_factory=list)
    cum: int = 0
    fire: bool = False
    sel_last: Optional[np.ndarray] = None
    delta: Optional[np.ndarray] = None


class PolestarOracle:
    """Reference engine with the library's call structure.

    cfg: any object with the workload fields (see drift_aware_kv_gb300.synth.Workload).
    weights: per layer dict of float64 arrays (values already in the storage dtype).
    """

    def __init__(self, cfg, weights, exact_cache: bool = False, store_noise: float = 0.0, noise_seed: int = 0):
        self.cfg = cfg
        self.W = weights
        self.bf16 = cfg.dtype == "bf16"
        # exact_cache=True keeps window hidden states unquantised (test switch)
        self.exact_cache = exact_cache
        # store_noise > 0 (test switch, bf16 workloads only): every value is
        # multiplied by (1 + u * store_noise), u ~ U(-1, 1) drawn from a seeded
        # generator, just before it is rounded to bf16.  This models an fp32
        # computation of the same value, whose last-bit differences decide the
        # bf16 rounding of values that lie close to a rounding midpoint; running
        # perturbed copies beside an unperturbed one measures how far each output
        # of the method moves under such differences.  0 = exact float64 values.
        self.store_noise = float(store_noise)
        self._noise_rng = np.random.default_rng(noise_seed) if store_noise > 0 else None
        # follow (test switch): another oracle on the same inputs, stepped first,
        # whose decisions -- the K-means labels and the top-k clusters -- this one
        # adopts instead of its own (which it still reports: "own_labels",
        # "own_topk"), so that a perturbed copy keeps the leader's decision path
        # and differs from it by rounding alone.
        self.follow: Optional["PolestarOracle"] = None
        self.last_recs = None
        c = cfg
        self.N = c.prompt_len + c.gen_len
        self.seqs: List[SeqState] = []
        for _ in range(c.batch):
            kv = [np.zeros((self.N, 2, c.n_kv_heads, c.head_dim)) for _ in range(c.n_layers)]
            self.seqs.append(SeqState(kv=kv))
        self.block = None
        self.block_entry = None
        self.exact_H: List[List[np.ndarray]] = [[] for _ in range(c.batch)]

    # ---- helpers --------------------------------------------------------------------
    def _store(self, x):
        if not self.bf16:
            return np.asarray(x, dtype=np.float64)
        if self._noise_rng is not None:
            x = np.asarray(x, dtype=np.float64)
            x = x * (1.0 + self.store_noise * self._noise_rng.uniform(-1.0, 1.0, x.shape))
        return to_bf16(x)

    def _span(self, b):
        start = self.cfg.prompt_len + b * self.cfg.block
        return start, start + self.cfg.block

    def window(self, b):
        """Local window of block b: [start-2B, start) and [end, end+B), clipped (§4.1)."""
        start, end = self._span(b)
        pre = [p for p in range(start - self.cfg.prefix_win, start) if p >= 0]
        suf = [p for p in range(end, end + self.cfg.suffix_win) if p < self.N]
        return pre + suf

    def qkv(self, l, h, pos):
        c, w = self.cfg, self.W[l]
        x = self._store(rmsnorm(h, w["attn_norm"], c.rms_eps))
        q = (x @ w["wq"].T).reshape(len(h), c.n_heads, c.head_dim)
        k = (x @ w["wk"].T).reshape(len(h), c.n_kv_heads, c.head_dim)
        v = (x @ w["wv"].T).reshape(len(h), c.n_kv_heads, c.head_dim)
        q = self._store(rope(q, pos, c.rope_base))
        k = self._store(rope(k, pos, c.rope_base))
        v = self._store(v)
        return q, k, v

    def scores(self, q, kv):
        """Scaled dot-product scores of queries [R, H, dh] against all N cached keys
        (grouped-query: head h reads kv head h // (H / Hkv)). Returns [R, H, N]."""
        c = self.cfg
        grp = c.n_heads // c.n_kv_heads
        s = np.empty((len(q), c.n_heads, len(kv)))
        for h in range(c.n_heads):  # s[r, h, n] = sum_d q[r, h, d] K[n, h // grp, d]
            s[:, h, :] = q[:, h, :] @ kv[:, 0, h // grp, :].T
        return s / math.sqrt(c.head_dim)

    def attend(self, q, kv):
        """Bidirectional attention over all N positions (Eq. 3). Returns the output
        [R, H*dh] (stored dtype) plus (scores, lse)."""
        c = self.cfg
        grp = c.n_heads // c.n_kv_heads
        s = self.scores(q, kv)
        lse = np.empty((len(q), c.n_heads))
        o = np.empty((len(q), c.n_heads, c.head_dim))
        for h in range(c.n_heads):  # o[r, h, :] = sum_n softmax(s[r, h, :])_n V[n, h // grp, :]
            lse[:, h] = logsumexp(s[:, h, :])
            p = np.exp(s[:, h, :] - lse[:, h, None])
            o[:, h, :] = p @ kv[:, 1, h // grp, :]
        return self._store(o.reshape(len(q), c.n_heads * c.head_dim)), s, lse

    def post(self, l, h, attn):
        """Output projection + residual, then the SwiGLU FFN + residual."""
        c, w = self.cfg, self.W[l]
        h1 = h + attn @ w["wo"].T
        y = self._store(rmsnorm(h1, w["ffn_norm"], c.rms_eps))
        a = self._store(silu(y @ w["w_gate"].T) * (y @ w["w_up"].T))
        return h1 + a @ w["w_down"].T

    def proxy_scores(self, l, z, kv):
        """Proxy queries q_c = W_q RMSNorm(z_c) (no rotary: a centroid has no position)
        and their scores against every cached key (§4.1 Measuring Drift)."""
        c, w = self.cfg, self.W[l]
        x = self._store(rmsnorm(z, w["attn_norm"], c.rms_eps))
        q = self._store((x @ w["wq"].T).reshape(len(z), c.n_heads, c.head_dim))
        s = self.scores(q, kv)
        return s, logsumexp(s)

    def _encode(self, st, l, rows_idx, H_rows):
        """Residual NVFP4 of rows against their cluster anchors (Algorithm 1,
        ResidualQuantization)."""
        lab = st.labels[l][rows_idx]
        r = to_f32(to_f32(H_rows) - st.A[l][lab])
        codes, sb, mg = nvfp4_encode(r)
        st.codes[l][rows_idx] = codes
        st.sbytes[l][rows_idx] = sb
        st.code_margin[l][rows_idx] = mg

    def _cached_H(self, st, l, seq_i):
        """Dequantize(H', Z) of Algorithm 1: anchor of the row's cluster + decoded
        residual (fp32 arithmetic)."""
        if self.exact_cache:
            return self.exact_H[seq_i][l].copy()
        dec = nvfp4_decode(st.codes[l], st.sbytes[l])
        return to_f32(dec + st.A[l][st.labels[l]])

    # ---- full-sequence forward (no cache reuse; the reference of App. C.2) -------------
    def full_forward_kv(self, x0_seq):
        """Keys and values of every position at every layer from a forward pass over
        the whole sequence x0_seq [N, d], recomputing everything (the no-cache
        decoding of §3 against which App. C.2 measures staleness).  Returns a list
        of [N, 2, Hkv, dh] arrays in the storage dtype; no state changes."""
        pos = np.arange(self.N)
        h = np.asarray(x0_seq, dtype=np.float64)
        out = []
        for l in range(self.cfg.n_layers):
            q, k, v = self.qkv(l, h, pos)
            kv = np.stack([k, v], axis=1)
            out.append(kv)
            o, _, _ = self.attend(q, kv)
            h = self.post(l, h, o)
        return out

    def full_forward(self, x0):
        """Replace every sequence's K/V cache by the full-sequence recompute from
        x0 [batch, N, d]; window state, centroids, NVFP4 store and histories are
        kept (a full refresh of the cache alone)."""
        x0 = np.asarray(x0, dtype=np.float64)
        for si, st in enumerate(self.seqs):
            st.kv = self.full_forward_kv(x0[si])

    # ---- block entry (Algorithm 1, block-entry phase; §4.1 Block entry) ---------------
    def _block_entry(self, si, st, x0, b):
        c = self.cfg
        start, end = self._span(b)
        win = self.window(b)
        if b % 2 == 0:
            rows = list(range(self.N))  # full-sequence refresh at alternate entries
        else:
            rows = sorted(set(win) | set(range(start, end)))
        pos = np.array(rows)
        widx = np.array([rows.index(p) for p in win])
        aidx = np.array([rows.index(p) for p in range(start, end)])
        h = np.asarray(x0[rows], dtype=np.float64)
        Hw = []
        for l in range(c.n_layers):
            Hw.append(h[widx].copy())
            q, k, v = self.qkv(l, h, pos)
            st.kv[l][pos, 0] = k
            st.kv[l][pos, 1] = v
            o, s, lse = self.attend(q, st.kv[l])
            if l == c.n_layers - 1:
                st.A_prev = (s[aidx], lse[aidx])
            h = self.post(l, h, o)
        nw = len(win)
        st.labels, st.z, st.s, st.A = [], [], [], []
        st.codes, st.sbytes, st.code_margin, st.P_prev = [], [], [], []
        out = dict(kmeans_margin=[], labels=[], z=[], A=[], own_labels=[], act_out=h[aidx].copy())
        self.exact_H[si] = [x.copy() for x in Hw]
        for l in range(c.n_layers):
            init = kmeans_init(c.seed, si, b, l, nw, c.K)
            lab, z, s, A, gap = spherical_kmeans(Hw[l], c.K, c.kmeans_iters, init)
            out["own_labels"].append(lab)
            if self.follow is not None:
                lab, z, s, A = self._adopt_labels(Hw[l], self.follow.seqs[si].labels[l], z)
            st.labels.append(lab)
            st.z.append(z)
            st.s.append(s)
            st.A.append(A)
            st.codes.append(np.zeros((nw, c.d_model), dtype=np.uint8))
            st.sbytes.append(np.zeros((nw, c.d_model // 16), dtype=np.uint8))
            st.code_margin.append(np.zeros((nw, c.d_model)))
            self._encode(st, l, np.arange(nw), Hw[l])
            st.P_prev.append(self.proxy_scores(l, z, st.kv[l]))
            out["kmeans_margin"].append(gap)
        st.cum = 0
        st.fire = False
        st.sel_last = None
        st.delta = None
        st.theta = [[] for _ in range(c.block)]
        return out

    @staticmethod
    def _adopt_labels(H, labels, z_own):
        """The last update of spherical K-means for given final labels: member
        sums of the unit rows, their normalisation, and the raw member means
        (an empty cluster keeps this oracle's own centroid)."""
        H = np.asarray(H, dtype=np.float64)
        X = H / np.linalg.norm(H, axis=1, keepdims=True)
        K = len(z_own)
        z, s, A = z_own.copy(), z_own.copy(), np.zeros_like(z_own)
        for c in range(K):
            mem = labels == c
            if np.any(mem):
                s[c] = X[mem].sum(axis=0)
                z[c] = s[c] / np.linalg.norm(s[c])
                A[c] = H[mem].mean(axis=0)
        return np.asarray(labels).copy(), z, s, to_f32(A)

    # ---- within-block step (Algorithm 1, layer loop; §4.1 Update Schedule) -------------
    def _step(self, si, st, x0, b, n_unmasked):
        c = self.cfg
        start, end = self._span(b)
        win = self.window(b)
        nw = len(win)
        wpos = np.array(win)
        apos = np.arange(start, end)
        st.cum += int(n_unmasked)
        fire = st.cum > c.tau_upd
        if fire:
            st.cum = 0
        st.fire = fire
        act = np.asarray(x0[start:end], dtype=np.float64)
        U = np.asarray(x0[win], dtype=np.float64)  # layer-0 packet: current inputs
        sel = np.ones(nw, dtype=bool)
        rec = dict(fire=fire, D=[], topk=[], topk_margin=[], sel=[], own_topk=[])
        for l in range(c.n_layers):
            kv = st.kv[l]
            if fire:
                Hc = self._cached_H(st, l, si)
                idx = np.nonzero(sel)[0]
                lab = st.labels[l][idx]
                old_hat = Hc[idx] / np.linalg.norm(Hc[idx], axis=1, keepdims=True)
                new = U[idx]
                new_hat = new / np.linalg.norm(new, axis=1, keepdims=True)
                for r, cl in enumerate(lab):
                    st.s[l][cl] += new_hat[r] - old_hat[r]
                st.z[l] = st.s[l] / np.linalg.norm(st.s[l], axis=1, keepdims=True)
                Hc[idx] = new
                if self.exact_cache:
                    self.exact_H[si][l][idx] = new
                self._encode(st, l, idx, new)
                _, k, v = self.qkv(l, new, wpos[idx])
                kv[wpos[idx], 0] = k
                kv[wpos[idx], 1] = v
            q, k, v = self.qkv(l, act, apos)
            kv[apos, 0] = k
            kv[apos, 1] = v
            if fire:
                s, lse = self.proxy_scores(l, st.z[l], kv)
                ps, plse = st.P_prev[l]
                D = np.mean(kl_div(s, lse, ps, plse), axis=1)
                st.P_prev[l] = (s, lse)
                ids, margin = topk_clusters(D, c.topk)
                rec["own_topk"].append(ids)
                if self.follow is not None:
                    ids = list(self.follow.last_recs[si]["topk"][l])
                sel = np.isin(st.labels[l], ids)
                rec["D"].append(D)
                rec["topk"].append(ids)
                rec["topk_margin"].append(margin)
                rec["sel"].append(sel.copy())
            o, s_a, lse_a = self.attend(q, kv)
            if l == c.n_layers - 1:
                ps, plse = st.A_prev
                st.delta = np.mean(kl_div(s_a, lse_a, ps, plse), axis=1)
                st.A_prev = (s_a, lse_a)
            act_next = self.post(l, act, o)
            if fire:
                idx = np.nonzero(sel)[0]
                qw, _, _ = self.qkv(l, Hc[idx], wpos[idx])
                ow, _, _ = self.attend(qw, kv)
                U = np.zeros((nw, c.d_model))
                U[idx] = self.post(l, Hc[idx], ow)
            act = act_next
        st.sel_last = sel if fire else None
        rec["act_out"] = act
        rec["U_last"] = U if fire else None
        rec["delta"] = st.delta
        return rec

    def calibrate_step(self, x0, n_unmasked, block_index, block_entry):
        """One denoising step of Polestar-Cache over every layer for every sequence.

        x0: [batch, N, d] layer-0 hidden states (values in the storage dtype)."""
        x0 = np.asarray(x0, dtype=np.float64)
        self.block, self.block_entry = block_index, bool(block_entry)
        recs = []
        for si, st in enumerate(self.seqs):
            if block_entry:
                recs.append(self._block_entry(si, st, x0[si], block_index))
            else:
                recs.append(self._step(si, st, x0[si], block_index, n_unmasked[si]))
        self.last_recs = recs
        return recs

    def decode_rows(self, recs):
        """Last-layer hidden states of the 2B rows the commit gate scores, per
        sequence [2B, d]: the active block's outputs, and for the suffix block the
        update packets U(t, L) of the rows the last layer refreshed (Algorithm 1,
        suffix commit); rows without a fresh state are zero (they cannot commit)."""
        c = self.cfg
        B = c.block
        start, end = self._span(self.block)
        win = self.window(self.block)
        out = []
        for si, st in enumerate(self.seqs):
            rows = np.zeros((2 * B, c.d_model))
            rec = recs[si]
            if "act_out" in rec:
                rows[:B] = rec["act_out"]
                if rec.get("U_last") is not None and st.sel_last is not None:
                    for wi, p in enumerate(win):
                        if end <= p < start + 2 * B and st.sel_last[wi]:
                            rows[p - start] = rec["U_last"][wi]
            out.append(rows)
        return out

    # ---- Polestar-Commit (§4.2; Algorithm 1, commit phases) ------------------------------
    def commit(self, logits, masked):
        """Commit mask for the 2B rows (active block, then suffix block) of every
        sequence; also returns c, Delta and tau_d per row."""
        c = self.cfg
        B = c.block
        b = self.block
        start, end = self._span(b)
        out = []
        for si, st in enumerate(self.seqs):
            conf = confidence(logits[si])
            m = np.zeros(2 * B, dtype=bool)
            delta_rel = np.zeros(2 * B)
            tau_d = np.zeros(2 * B)
            margin = np.full(2 * B, math.inf)
            margin_drift = np.full(2 * B, math.inf)
            pos = np.arange(start, start + 2 * B)
            valid = pos < self.N
            msk = np.zeros(2 * B, dtype=bool)
            msk[valid] = np.asarray(masked[si])[pos[valid]]
            cur = np.arange(B)
            if self.block_entry:
                m[cur] = msk[cur] & (conf[cur] >= c.tau_s)
                margin[cur] = np.abs(conf[cur] - c.tau_s)
            else:
                for j in range(B):
                    hist = st.theta[j][-c.hist:] if c.hist > 0 else []
                    mean = float(np.mean(hist)) if hist else 0.0
                    delta_rel[j] = st.delta[j] - mean
                    st.theta[j].append(float(st.delta[j]))
                    if c.hist > 0:
                        st.theta[j] = st.theta[j][-c.hist:]
                    else:
                        st.theta[j] = []
                tau_d[cur] = drift_threshold(conf[cur], c.tau_s, c.alpha)
                m[cur] = msk[cur] & ((conf[cur] >= c.tau_s) | (delta_rel[cur] >= tau_d[cur]))
                margin[cur] = np.abs(conf[cur] - c.tau_s)
                margin_drift[cur] = np.abs(delta_rel[cur] - tau_d[cur])
                if st.fire and st.sel_last is not None:
                    win = self.window(b)
                    for wi, p in enumerate(win):
                        if p >= end and st.sel_last[wi]:
                            j = p - start
                            m[j] = msk[j] and conf[j] >= c.tau_suf
                            margin[j] = abs(conf[j] - c.tau_suf)
            out.append(dict(commit=m, conf=conf, delta_rel=delta_rel, tau_d=tau_d,
                            margin=margin, margin_drift=margin_drift))
        return out


# --------------------------------------------------------------------------------------
# closed-loop decoding: LM head, greedy tokens, the progress rule (Algorithm 1 in full)
# --------------------------------------------------------------------------------------


def lm_logits(h, w_lm, gain, eps, bf16):
    """Logits m_theta(v | y, i) of the LM head (Eq. 1) for hidden states h [R, d]:
    RMSNorm with the final gain, rounded to the storage dtype like every
    projection input, then W_lm [V, d]."""
    x = rmsnorm(h, gain, eps)
    if bf16:
        x = to_bf16(x)
    return x @ np.asarray(w_lm, dtype=np.float64).T


def greedy_tokens(logits):
    """y^_i = argmax_v logits (Eq. 1; the synthetic vocabulary has no [MASK] id),
    ties to the lower id; also the gap between the two largest logits relative
    to the largest magnitude (the decision's margin)."""
    l = np.asarray(logits, dtype=np.float64)
    ids = np.argmax(l, axis=-1)  # first maximum: the lower id on ties
    top2 = np.sort(l, axis=-1)[..., -2:]
    margin = (top2[..., 1] - top2[..., 0]) / np.maximum(np.abs(top2[..., 1]), 1e-300)
    return ids, margin


def progress_rule(commit, conf, masked_cur):
    """Every step makes progress.  The paper builds its decoder on the
    Fast-dLLM-style block decoder (App. D.1) without spelling out the case in
    which the gate commits nothing; read here as that decoder's fallback: a step
    that commits no token of the current block while some are still masked
    commits the masked one of highest confidence (ties to the lower position).
    commit / masked_cur: [B] bool of the current block; returns the new
    current-block commit flags."""
    out = np.array(commit, dtype=bool).copy()
    m = np.asarray(masked_cur, dtype=bool)
    if m.any() and not (out & m).any():
        c = np.where(m, np.asarray(conf, dtype=np.float64), -np.inf)
        out[int(np.argmax(c))] = True
    return out


def embed_inputs(tokens, masked, embed, mask_emb):
    """Layer-0 hidden states of one step (§2: the model reads the partially
    unmasked sequence): the embedding row of every decoded token, the [MASK]
    embedding at masked positions.  tokens [N] int, masked [N] bool,
    embed [V, d], mask_emb [d]; returns [N, d]."""
    E = np.asarray(embed, dtype=np.float64)
    out = E[np.asarray(tokens)].copy()
    out[np.asarray(masked, dtype=bool)] = np.asarray(mask_emb, dtype=np.float64)
    return out


def apply_commits(tokens, masked, commit, ids, start):
    """Committed positions take their greedy tokens and leave the mask
    (Algorithm 1: y_i <- y^_i for committed i).  commit / ids: the 2B rows from
    `start` (active block, then suffix block); rows past the sequence end are
    ignored.  Updates tokens [N] / masked [N] in place; returns the number of
    tokens committed."""
    n = 0
    N = len(tokens)
    for j in range(len(commit)):
        p = start + j
        if p < N and commit[j] and masked[p]:
            tokens[p] = int(ids[j])
            masked[p] = False
            n += 1
    return n


def weights_to_numpy(layer_weights):
    """torch tensors (any dtype) -> float64 numpy, per layer dict."""
    out = []
    for lw in layer_weights:
        out.append({k: v.detach().to("cpu").double().numpy() for k, v in lw.items()})
    return out
