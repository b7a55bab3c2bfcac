"""Lockstep parity harness: runs the CUDA library (through the C ABI) and the CPU
oracle on the same seeded trajectory and compares every step.

Exactness bar: cluster ids, top-k sets, selected rows, NVFP4 codes/scales and
commit masks are compared exactly; a mismatch is accepted only when the
oracle's decision margin is below NEAR_TIE (a near tie), and is then counted.
After a near-tie divergence the two states legitimately differ.  The library
then takes over the oracle's state through the state import (labels,
centroids, NVFP4 store, K/V caches, score and drift histories, trigger counts:
oracle -> GPU only, nothing flows back) and lockstep comparison goes on from the
next step (resync=False: both engines keep running and comparison resumes at
the next block entry with an even block index, which recomputes every state
from x0 alone).
Floating-point outputs use the tolerances below (K/V, hidden states and update
packets by relative L2 error).

Drift tolerance.  KL drift must agree to KL_ABS + KL_REL |D| (1e-5 + 1e-3 rel).
In a bf16 stack the queries and keys feeding the drift are bf16 roundings of
values the GPU computes in fp32 and the oracle in float64; a value within the
fp32 error of a bf16 rounding midpoint can round either way, and each such
element moves a score by ~2^-8 of its size.  The oracle measures that
sensitivity itself: beside the unperturbed oracle, N_PERTURBED copies run the
same trajectory with every bf16 store perturbed at the fp32 level
(``PolestarOracle(store_noise=...)``) and adopt the unperturbed oracle's
decisions (K-means labels, top-k sets) so that they differ from it by rounding
alone.  The largest deviation of their D, delta and Delta from the unperturbed
values (over the clusters of a layer, the rows of a block), times BAND_FACTOR,
is that step's sensitivity band.  KL is held to 1e-5 + 1e-3 rel plus that
band, and a decision (K-means labels, top-k set, the Delta >= tau_d branch of
the gate) may differ only where its margin lies inside the band or where a
perturbed copy's own decision already differs; those are counted as
sensitivity ties, apart from the near ties.
Nothing in the band comes from the GPU side.  fp32 workloads store no bf16
value and run no perturbed copy: their band is zero."""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

from drift_aware_kv_gb300 import polestar as P
from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O

NEAR_TIE = 1e-4
KL_ABS, KL_REL = 1e-5, 1e-3
N_PERTURBED = 2
BAND_FACTOR = 3.0


def store_noise_for(w) -> float:
    """Relative size of the fp32-level perturbation of a bf16 store: about the
    error of an fp32 dot product over d_model terms (sqrt(d) units of 2^-23)."""
    return math.sqrt(w.d_model) * 2.0 ** -23


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / max(den, 1e-30))


def unpack_codes(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


@dataclasses.dataclass
class Report:
    steps: int = 0
    compared: int = 0
    near_ties: int = 0
    diverged_at: int = -1
    max_kv_err: float = 0.0
    max_act_err: float = 0.0
    max_u_err: float = 0.0
    max_kl_err: float = 0.0
    code_mismatch: int = 0
    max_dec_err: float = 0.0
    fires: int = 0
    commits: int = 0
    sensitivity_ties: int = 0
    max_band_rel: float = 0.0
    max_centroid_err: float = 0.0
    resyncs: int = 0
    max_u_band: float = 0.0
    notes: list = dataclasses.field(default_factory=list)


class Lockstep:
    """start_block > 0: the trajectory's inputs are drawn from its start, but the
    engines join at that block's entry, with every layer's K/V cache first set
    (on both sides: the oracle's arrays and the library's buffers through
    polestar_debug_write) to the same seeded N(0, 1) values in the storage
    dtype.  An odd start block's entry forwards only window + block rows, so the
    rest of the cache stays the seeded one: the within-block path runs at full
    width without a full-sequence forward on the CPU."""

    def __init__(self, w: synth.Workload, kv_tol: float, act_tol: float, n_perturbed=None, start_block=0,
                 resync=True):
        self.w = w
        self.start_block = start_block
        self.resync = resync
        self.kv_tol, self.act_tol = kv_tol, act_tol
        # block-entry centroids/anchors: fp32 path ~1e-6; bf16 path inherits the
        # bf16 rounding of the A operands of the preceding layers
        self.state_tol = 1e-5 if w.dtype == "fp32" else 1e-3
        # member sums after incremental updates accumulate every refresh of the
        # block in fp32 (up to Wmax unit rows per update, a few updates): about
        # 1000 roundings of 2^-24 -> 1e-4 relative
        self.update_tol = 1e-4 if w.dtype == "fp32" else 1e-3
        W_cpu = synth.make_weights(w, "cpu")
        Wn = O.weights_to_numpy(W_cpu)
        self.orc = O.PolestarOracle(w, Wn)
        if n_perturbed is None:
            n_perturbed = N_PERTURBED if w.dtype == "bf16" else 0
        self.pert = [O.PolestarOracle(w, Wn, store_noise=store_noise_for(w), noise_seed=i + 1)
                     for i in range(n_perturbed)]
        for o in self.pert:
            o.follow = self.orc
        self.Wg = [{k: v.cuda() for k, v in lw.items()} for lw in W_cpu]
        self.lib = P.Polestar(w, self.Wg)
        self.tr = synth.Trajectory(w)
        self.rep = Report()
        self.conf_tol = None
        self.diverged = False
        self.N = w.seq_len
        self.Wmax = w.prefix_win + w.suffix_win

    def read_layer(self, which, layer, shape, dtype):
        return self.lib.read(which, layer, shape, dtype)

    def _seed_caches(self):
        """The same seeded K/V cache on both sides (see the class docstring)."""
        w = self.w
        dt = synth.torch_dtype(w)
        g = torch.Generator(device="cpu").manual_seed(synth.derive_seed(w.seed, 0xCAC4E))
        for l in range(w.n_layers):
            kv = torch.randn(w.batch, self.N, 2, w.n_kv_heads * w.head_dim, generator=g).to(dt)
            self.lib.write(P.BUF_KV, l, kv)
            kvn = kv.double().numpy().reshape(w.batch, self.N, 2, w.n_kv_heads, w.head_dim)
            for o in [self.orc] + self.pert:
                for s in range(w.batch):
                    o.seqs[s].kv[l] = kvn[s].copy()

    def run(self, max_steps=None):
        w, rep = self.w, self.rep
        dt = synth.torch_dtype(w)
        if self.start_block > 0:
            while True:  # inputs of the earlier blocks are drawn but not run
                st = self.tr.next_step()
                if st["block_entry"] and st["block_index"] == self.start_block:
                    break
            self._seed_caches()
            pending = st
        else:
            pending = None
        while True:
            st = pending if pending is not None else self.tr.next_step()
            pending = None
            if st is None or (max_steps is not None and rep.steps >= max_steps):
                break
            x0 = st["x0"].to(dt)
            if st["block_entry"] and st["block_index"] % 2 == 0:
                # full refresh: every state is a function of x0 again
                self.diverged = False
            x0n = x0.double().numpy()
            recs = self.orc.calibrate_step(x0n, st["n_unmasked"], st["block_index"], st["block_entry"])
            self.recs_p = [o.calibrate_step(x0n, st["n_unmasked"], st["block_index"], st["block_entry"])
                           for o in self.pert]
            xg = x0.cuda()
            out = self.lib.calibrate_step(xg, st["n_unmasked"], st["block_index"], st["block_entry"])
            torch.cuda.synchronize()
            ok = True
            if not self.diverged:
                ok = self._compare_step(st, recs, out)
            # drift histories before this step's commit (the bound on Delta uses them)
            self.theta_before = [[list(t) for t in s.theta] for s in self.orc.seqs]
            coms = self.orc.commit(st["logits"].numpy(), st["masked"].numpy())
            self.coms_p = [o.commit(st["logits"].numpy(), st["masked"].numpy()) for o in self.pert]
            lg = st["logits"].cuda()
            mk = st["masked"].to(torch.uint8).cuda()
            cm = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
            self.lib.commit(lg, mk, cm)
            torch.cuda.synchronize()
            if not self.diverged:
                ok = ok and self._compare_commit(st, coms, cm.cpu().numpy())
                if ok:
                    ok = self._after_commit(st, coms, lg, mk, cm)
                if ok:
                    rep.compared += 1
            rep.steps += 1
            if not ok:
                if rep.diverged_at < 0:
                    rep.diverged_at = st["t"]
                if self.resync:
                    # the library takes over the oracle's state (labels, centroids,
                    # store, caches, histories: oracle -> GPU only) and lockstep
                    # comparison goes on from the next step
                    self._import_oracle_state(st)
                    rep.resyncs += 1
                else:
                    self.diverged = True
        return rep

    def _after_commit(self, st, coms, lg, mk, cm):
        """Hook after a commit that matched the oracle's (True: keep going)."""
        return True

    def _import_oracle_state(self, st):
        """The oracle's calibration state after this step, written into the
        library's context through the state import (polestar_debug_write +
        polestar_debug_enter_block)."""
        w, o = self.w, self.orc
        b, L, N, K, H, B, d, Wm = w.batch, w.n_layers, self.N, w.K, w.n_heads, w.block, w.d_model, self.Wmax
        dt = synth.torch_dtype(w)
        nw = len(o.window(st["block_index"]))
        f32 = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), dtype=torch.float64).to(torch.float32)
        for l in range(L):
            self.lib.write(P.BUF_KV, l, torch.tensor(
                np.stack([o.seqs[s].kv[l].reshape(N, 2, -1) for s in range(b)])).to(dt))
            lab = np.zeros((b, Wm), dtype=np.uint8)
            codes = np.zeros((b, Wm, d // 2), dtype=np.uint8)
            scales = np.zeros((b, Wm, d // 16), dtype=np.uint8)
            for s in range(b):
                q = o.seqs[s]
                lab[s, :nw] = q.labels[l]
                codes[s, :nw] = q.codes[l][:, 0::2] | (q.codes[l][:, 1::2] << 4)
                scales[s, :nw] = q.sbytes[l]
            self.lib.write(P.BUF_LABELS, l, torch.tensor(lab))
            self.lib.write(P.BUF_CODES, l, torch.tensor(codes))
            self.lib.write(P.BUF_SCALES, l, torch.tensor(scales))
            for which, attr in ((P.BUF_CENTROID, "z"), (P.BUF_CSUM, "s"), (P.BUF_ANCHOR, "A")):
                self.lib.write(which, l, f32(np.stack([getattr(o.seqs[s], attr)[l] for s in range(b)])))
            self.lib.write(P.BUF_PROXY, l, f32(np.stack([o.seqs[s].P_prev[l][0] for s in range(b)])))
            self.lib.write(P.BUF_PROXY_LSE, l, f32(np.stack([o.seqs[s].P_prev[l][1] for s in range(b)])))
        self.lib.write(P.BUF_ACTIVE_PREV, 0, f32(np.stack([o.seqs[s].A_prev[0] for s in range(b)])))
        self.lib.write(P.BUF_ACTIVE_LSE, 0, f32(np.stack([o.seqs[s].A_prev[1] for s in range(b)])))
        hist = max(1, w.hist)
        th = np.zeros((b, B, hist))
        thn = np.zeros((b, B), dtype=np.int32)
        for s in range(b):
            for j in range(B):
                t = o.seqs[s].theta[j][-hist:] if w.hist > 0 else []
                th[s, j, :len(t)] = t
                thn[s, j] = len(t)
        self.lib.write(P.BUF_THETA, 0, f32(th))
        self.lib.write(P.BUF_THETA_N, 0, torch.tensor(thn))
        self.lib.enter_block(st["block_index"], [o.seqs[s].cum for s in range(b)])

    # ---- the oracle's own sensitivity (perturbed copies) --------------------------
    def _live(self):
        return list(range(len(self.pert)))

    def _band(self, values_nom, values_pert):
        """BAND_FACTOR x the largest deviation of the perturbed copies from
        the unperturbed value, over the whole array (one band for the clusters of
        a layer or the rows of a block); 0 without perturbed copies."""
        if not values_pert:
            return 0.0
        dev = max(float(np.max(np.abs(np.asarray(v) - np.asarray(values_nom)))) for v in values_pert)
        return BAND_FACTOR * dev

    # ------------------------------------------------------------------
    def _decision(self, name, equal, margin, tie=NEAR_TIE):
        """Exact decision check; returns False (stop) on an accepted near tie."""
        if equal:
            return True
        if margin < tie:
            self.rep.near_ties += 1
            self.rep.notes.append(f"near tie in {name} (margin {margin:.2e})")
            return False
        raise AssertionError(f"{name}: mismatch with oracle margin {margin:.3e}")

    def _compare_step(self, st, recs, out):
        w, rep = self.w, self.rep
        L, b, K, d = w.n_layers, w.batch, w.K, w.d_model
        nw = out.win_len
        if st["block_entry"]:
            for l in range(L):
                lab = self.read_layer(P.BUF_LABELS, l, (b, self.Wmax), torch.uint8).numpy()
                for s in range(b):
                    o = self.orc.seqs[s]
                    same = np.array_equal(lab[s, :nw], o.labels[l])
                    if not same and recs[s]["kmeans_margin"][l] >= NEAR_TIE and any(
                            not np.array_equal(self.recs_p[i][s]["own_labels"][l], o.labels[l]) for i in self._live()):
                        self._sensitivity_tie(f"kmeans labels (l={l}, s={s})", recs[s]["kmeans_margin"][l], 0.0)
                        return False
                    if not self._decision(f"kmeans labels (l={l}, s={s})", same, recs[s]["kmeans_margin"][l]):
                        return False
                codes = unpack_codes(self.read_layer(P.BUF_CODES, l, (b, self.Wmax, d // 2),
                                                     torch.uint8).numpy())
                scales = self.read_layer(P.BUF_SCALES, l, (b, self.Wmax, d // 16), torch.uint8).numpy()
                anchor = self.read_layer(P.BUF_ANCHOR, l, (b, K, d), torch.float32).numpy()
                z = self.read_layer(P.BUF_CENTROID, l, (b, K, d), torch.float32).numpy()
                for s in range(b):
                    o = self.orc.seqs[s]
                    ea, ez = rel_l2(anchor[s], o.A[l]), rel_l2(z[s], o.z[l])
                    # the oracle's own spread of these states under fp32-level
                    # rounding noise (perturbed copies), times BAND_FACTOR
                    band_a = BAND_FACTOR * max([rel_l2(q.seqs[s].A[l], o.A[l]) for q in self.pert] or [0.0])
                    band_z = BAND_FACTOR * max([rel_l2(q.seqs[s].z[l], o.z[l]) for q in self.pert] or [0.0])
                    rep.max_centroid_err = max(rep.max_centroid_err, ea, ez)
                    assert ea < max(self.state_tol, band_a), f"anchors rel err {ea} (layer {l}, seq {s}, band {band_a})"
                    assert ez < max(self.state_tol, band_z), f"centroids rel err {ez} (layer {l}, seq {s}, band {band_z})"
                    self._check_codes(codes[s, :nw], scales[s, :nw], o, l, s=s, nw=nw)
        else:
            fire = [bool(out.fire[s]) for s in range(b)]
            assert fire == [bool(r["fire"]) for r in recs], "trigger"
            rep.fires += sum(fire)
            drift = np.stack([self.read_layer(P.BUF_DRIFT, l, (b, K), torch.float32).numpy()
                              for l in range(L)])
            topk = np.stack([self.read_layer(P.BUF_TOPK, l, (b, w.topk), torch.int32).numpy()
                             for l in range(L)])
            sel = np.stack([self.read_layer(P.BUF_SELECTED, l, (b, self.Wmax), torch.uint8).numpy()
                            for l in range(L)])
            live = self._live()
            for s in range(b):
                if not fire[s]:
                    continue
                for l in range(L):
                    D_o = recs[s]["D"][l]
                    pert = [self.recs_p[i][s]["D"][l] for i in live]
                    band = self._band(D_o, pert)
                    rep.max_band_rel = max(rep.max_band_rel, band / max(float(np.max(np.abs(D_o))), 1e-30))
                    err = np.abs(drift[l, s] - D_o)
                    tol = KL_ABS + KL_REL * np.abs(D_o) + band
                    rep.max_kl_err = max(rep.max_kl_err, float(np.max(err / (KL_ABS + KL_REL * np.abs(D_o)))))
                    assert np.all(err <= tol), f"drift D (l={l}, s={s}): err {err}, tol {tol}"
                    # the selected set is the decision; the order inside it is not
                    same = sorted(topk[l, s]) == sorted(recs[s]["topk"][l])
                    if not same:
                        order = sorted(range(K), key=lambda c: (-D_o[c], c))
                        gap = D_o[order[w.topk - 1]] - D_o[order[w.topk]] if w.topk < K else math.inf
                        unstable = any(sorted(self.recs_p[i][s]["own_topk"][l]) != sorted(recs[s]["topk"][l])
                                       for i in live)
                        if recs[s]["topk_margin"][l] >= NEAR_TIE and (gap <= 2 * band or unstable):
                            self._sensitivity_tie(f"top-k (l={l}, s={s})", gap, band)
                            return False
                    if not self._decision(f"top-k (l={l}, s={s})", same, recs[s]["topk_margin"][l]):
                        return False
                    assert np.array_equal(sel[l, s, :nw].astype(bool), recs[s]["sel"][l]), "selection"
            delta = self.read_layer(P.BUF_DELTA, 0, (b, w.block), torch.float32).numpy()
            self.delta_band = []
            for s in range(b):
                d_o = recs[s]["delta"]
                band = self._band(d_o, [self.recs_p[i][s]["delta"] for i in live])
                self.delta_band.append(band)
                err = np.abs(delta[s] - d_o)
                tol = KL_ABS + KL_REL * np.abs(d_o) + band
                assert np.all(err <= tol), \
                    f"token drift delta (s={s}, step {st['t']}): worst {int(np.argmax(err - tol))}, err {err.max():.3e}, " \
                    f"oracle {d_o[np.argmax(err - tol)]:.6e}, library {delta[s][np.argmax(err - tol)]:.6e}"
            act = self.read_layer(P.BUF_ACT_OUT, 0, (b, w.block, d), torch.float32).numpy()
            for s in range(b):
                e = rel_l2(act[s], recs[s]["act_out"])
                rep.max_act_err = max(rep.max_act_err, e)
                assert e < self.act_tol, f"active-row output rel err {e}"
            if any(fire):
                # unit centroids and member sums after this step's incremental update
                for l in range(L):
                    zg = self.read_layer(P.BUF_CENTROID, l, (b, K, d), torch.float32).numpy()
                    sg = self.read_layer(P.BUF_CSUM, l, (b, K, d), torch.float32).numpy()
                    for s in range(b):
                        if not fire[s]:
                            continue
                        o = self.orc.seqs[s]
                        for name, got, ref, pert in (("z", zg[s], o.z[l], [q.seqs[s].z[l] for q in self.pert]),
                                                     ("s", sg[s], o.s[l], [q.seqs[s].s[l] for q in self.pert])):
                            band = BAND_FACTOR * max([rel_l2(x, ref) for x in pert] or [0.0])
                            e = rel_l2(got, ref)
                            rep.max_centroid_err = max(rep.max_centroid_err, e)
                            assert e < max(self.update_tol, band), \
                                f"centroid {name} after the update rel err {e} (layer {l}, seq {s}, band {band})"
                U = self.read_layer(P.BUF_UPDATE, 0, (b, self.Wmax, d), torch.float32).numpy()
                for s in range(b):
                    if not fire[s]:
                        continue
                    selm = recs[s]["sel"][-1]
                    ref = recs[s]["U_last"][selm]
                    e = rel_l2(U[s, :nw][selm], ref)
                    rep.max_u_err = max(rep.max_u_err, e)
                    # the packets are computed from NVFP4-decoded window states, whose
                    # code choices amplify upstream bf16 differences: the oracle's
                    # perturbed copies give the spread that this alone causes
                    band = BAND_FACTOR * max([rel_l2(self.recs_p[i][s]["U_last"][selm], ref)
                                              for i in self._live()] or [0.0])
                    rep.max_u_band = max(rep.max_u_band, band)
                    assert e < max(self.act_tol, band), f"update packet rel err {e} (band {band})"
                    for l in range(L):
                        self._check_codes(None, None, self.orc.seqs[s], l, s=s, nw=nw)
        # K/V cache of every layer
        dt = synth.torch_dtype(w)
        for l in range(L):
            kv = self.read_layer(P.BUF_KV, l, (b, self.N, 2, w.n_kv_heads, w.head_dim), dt).double().numpy()
            for s in range(b):
                e = rel_l2(kv[s], self.orc.seqs[s].kv[l])
                rep.max_kv_err = max(rep.max_kv_err, e)
                assert e < self.kv_tol, f"K/V cache rel err {e} (layer {l}, seq {s})"
        return True

    def _sensitivity_tie(self, name, margin, band):
        self.rep.sensitivity_ties += 1
        self.rep.notes.append(f"sensitivity tie in {name} (margin {margin:.2e}, oracle band {band:.2e})")

    def _check_codes(self, codes, scales, o, l, s=None, nw=None):
        """NVFP4 store of layer l.  Where the encoder's inputs are exact on both
        sides (fp32 workloads; layer 0, whose rows are the caller's x0) the codes
        and scales must match bit for bit up to near ties.  Deeper layers of a
        bf16 stack carry the upstream bf16 rounding differences into the residual
        r = h - A, so there the decoded hidden states are compared instead."""
        w = self.w
        d = w.d_model
        if codes is None:
            codes = unpack_codes(self.read_layer(P.BUF_CODES, l, (w.batch, self.Wmax, d // 2),
                                                 torch.uint8).numpy())[s, :nw]
            scales = self.read_layer(P.BUF_SCALES, l, (w.batch, self.Wmax, d // 16), torch.uint8).numpy()[s, :nw]
        oc, osb, om = o.codes[l], o.sbytes[l], o.code_margin[l]
        exact = w.dtype == "fp32" or l == 0
        if not exact:
            lab = o.labels[l]
            dec_g = O.nvfp4_decode(codes, scales) + o.A[l][lab]
            dec_o = O.nvfp4_decode(oc, osb) + o.A[l][lab]
            e = rel_l2(dec_g, dec_o)
            self.rep.max_dec_err = max(self.rep.max_dec_err, e)
            # NVFP4 rounding amplifies the upstream bf16 differences of the rows
            # it encodes; the oracle's perturbed copies measure that amplification
            si = s
            band = BAND_FACTOR * max([rel_l2(O.nvfp4_decode(q.seqs[si].codes[l], q.seqs[si].sbytes[l]) + o.A[l][lab],
                                             dec_o) for q in self.pert] or [0.0])
            assert e < max(self.act_tol, band), f"decoded window states rel err {e} (layer {l}, band {band})"
            return
        bad = codes != oc
        sbad = np.repeat(scales != osb, 16, axis=1)
        bad = bad | sbad
        if np.any(bad):
            worst = float(np.max(om[bad]))
            self.rep.code_mismatch += int(bad.sum())
            if worst >= NEAR_TIE:
                raise AssertionError(f"NVFP4 codes differ with oracle margin {worst:.3e} "
                                     f"({int(bad.sum())} elements, layer {l})")

    def _compare_commit(self, st, coms, cm):
        w = self.w
        conf = self.read_layer(P.BUF_CONF, 0, (w.batch, 2 * w.block), torch.float32).numpy()
        drel = self.read_layer(P.BUF_DREL, 0, (w.batch, 2 * w.block), torch.float32).numpy()
        taud = self.read_layer(P.BUF_TAUD, 0, (w.batch, 2 * w.block), torch.float32).numpy()
        live = self._live()
        for s in range(w.batch):
            co = coms[s]
            valid = np.arange(2 * w.block) + w.prompt_len + st["block_index"] * w.block < self.N
            # both sides score the same logits unless a closed loop sets conf_tol
            # (each side's own logits: the tolerance their difference allows)
            ctol = self.conf_tol[s] if self.conf_tol is not None else 1e-6 + 1e-5 * np.abs(co["conf"])
            assert np.all(np.abs(conf[s][valid] - co["conf"][valid]) <= ctol[valid]), "confidence"
            # Delta = delta - mean(history): each term carries the delta tolerance
            band = self._band(co["delta_rel"], [self.coms_p[i][s]["delta_rel"] for i in live])
            d_now = self.orc.seqs[s].delta
            hist_abs = np.array([np.mean(np.abs(t[-w.hist:])) if (t and w.hist > 0) else 0.0
                                 for t in self.theta_before[s]])
            tol_d = 2 * KL_ABS + KL_REL * (np.abs(d_now) + hist_abs) if d_now is not None else np.full(w.block, KL_ABS)
            tol = np.zeros(2 * w.block)
            tol[:w.block] = tol_d
            assert np.all(np.abs(drel[s] - co["delta_rel"]) <= tol + band), "Delta"
            # tau_d = alpha (tau_s - c)^2 moves with c: over the confidence
            # tolerance, the oracle's own threshold function bounds the change
            tt = 1e-6 + 1e-4 * np.abs(co["tau_d"])
            if self.conf_tol is not None:
                lo = O.drift_threshold(co["conf"] - ctol, w.tau_s, w.alpha)
                hi = O.drift_threshold(co["conf"] + ctol, w.tau_s, w.alpha)
                tt = tt + np.maximum(np.abs(lo - co["tau_d"]), np.abs(hi - co["tau_d"]))
                tt[w.block:] = 1e-6  # the suffix block has no drift threshold
            assert np.all(np.abs(taud[s] - co["tau_d"]) <= tt), "tau_d"
            tol = tol + np.where(np.arange(2 * w.block) < w.block, tt, 0.0)
            eq = np.array_equal(cm[s].astype(bool), co["commit"])
            if not eq:
                diff = cm[s].astype(bool) != co["commit"]
                conf_tie = co["margin"][diff] < NEAR_TIE
                drift_tie = co["margin_drift"][diff] < NEAR_TIE
                if np.all(conf_tie | drift_tie):
                    if not self._decision(f"commit mask (s={s})", False, 0.0):
                        return False
                unstable = any(not np.array_equal(self.coms_p[i][s]["commit"], co["commit"]) for i in live)
                in_band = co["margin_drift"][diff] <= tol[diff] + band
                conf_band = co["margin"][diff] <= ctol[diff]
                if np.all(conf_tie | in_band | conf_band) or unstable:
                    self._sensitivity_tie(f"commit mask (s={s})", float(np.min(co["margin_drift"][diff])), band)
                    return False
                raise AssertionError(f"commit mask (s={s}): mismatch with oracle margins "
                                     f"{co['margin'][diff]} / {co['margin_drift'][diff]}")
            self.commits_add(co)
        return True

    def commits_add(self, co):
        self.rep.commits += int(co["commit"].sum())


class DecodeTokensLockstep(Lockstep):
    """Lockstep whose every matched commit is followed by polestar_decode_tokens
    on copies of the step's mask (and a zero token array), against the oracle's
    progress_rule + greedy_tokens + apply_commits on the same logits: the
    progress rule's choice, the greedy ids, the token / mask update and the
    counts must agree exactly (the choice up to confidences within the
    confidence tolerance of each other)."""

    def __init__(self, *a, **kw):
        super().__init__(*a, **kw)
        self.progress_steps = 0
        self.tokens_checked = 0

    def _after_commit(self, st, coms, lg, mk, cm):
        w = self.w
        b, B, N = w.batch, w.block, self.N
        start = w.prompt_len + st["block_index"] * B
        tok_g = torch.zeros(b, N, dtype=torch.int32, device="cuda")
        msk_g = mk.clone()
        cm_g = cm.clone()
        counts, left = self.lib.decode_tokens(lg, cm_g, tok_g, msk_g)
        tok_o = np.zeros((b, N), dtype=np.int64)
        msk_o = st["masked"].numpy().copy()
        lgn = st["logits"].numpy()
        cmg = cm_g.cpu().numpy().astype(bool)
        for s in range(b):
            co = coms[s]
            c = co["commit"].copy()
            c[:B] = O.progress_rule(c[:B], co["conf"][:B], msk_o[s, start:start + B])
            if c[:B].sum() > co["commit"][:B].sum():
                self.progress_steps += 1
            if not np.array_equal(cmg[s], c):
                jo = int(np.argmax(c & ~co["commit"]))
                jg = int(np.argmax(cmg[s] & ~co["commit"]))
                gap = abs(co["conf"][jo] - co["conf"][jg])
                if not self._decision(f"progress rule (s={s})", False, gap, tie=1e-6 + 1e-5 * co["conf"][jo]):
                    return False
            ids, _ = O.greedy_tokens(lgn[s])
            O.apply_commits(tok_o[s], msk_o[s], c, ids, start)
            assert counts[s] == int(c[(np.arange(2 * B) + start) < N].sum()), "committed count"
            assert left[s] == int(msk_o[s, start:start + B].sum()), "still masked"
        assert np.array_equal(tok_g.cpu().numpy(), tok_o), "tokens"
        assert np.array_equal(msk_g.cpu().numpy().astype(bool), msk_o), "mask"
        self.tokens_checked += int(sum(counts))
        return True


class ClosedLoop(Lockstep):
    """Closed-loop generation in lockstep (Algorithm 1 in full).  Each side
    decodes its own tokens: the library through polestar_embed ->
    polestar_calibrate_step -> polestar_decode_logits -> polestar_commit ->
    polestar_decode_tokens, the oracle through embed_inputs -> calibrate_step ->
    decode_rows + lm_logits -> commit -> progress_rule + greedy_tokens +
    apply_commits, both from the same prompt and the same seeded embedding,
    [MASK] embedding, LM head and final norm.

    Per step: x0 bit-exact; the calibration state as in Lockstep; the logits
    per sequence within logit_tol relative L2 (or the oracle's perturbed copies'
    band); rows without a fresh state zero on both sides; the gate's decisions,
    the progress rule's choice, the greedy tokens and the committed counts exact
    up to decisions whose oracle margin lies within what the logits' difference
    allows (a logit error e moves a confidence by at most a factor exp(2e) and
    decides an argmax only inside a top-2 gap of 2e).  After such a tie the
    library takes over the oracle's tokens, mask and calibration state and the
    loop goes on."""

    def __init__(self, w, kv_tol, act_tol, logit_tol, elem_tol, n_perturbed=None):
        super().__init__(w, kv_tol, act_tol, n_perturbed=n_perturbed)
        self.logit_tol, self.elem_tol = logit_tol, elem_tol
        dw = synth.make_decode_weights(w, "cpu")
        self.dn = {k: v.double().numpy() for k, v in dw.items()}
        self.dg = {k: v.cuda() for k, v in dw.items()}
        from drift_aware_kv_gb300.decode import Generator
        self.gen = Generator(self.lib, self.dg)
        self.max_logit_err = 0.0
        self.steps_by_kind = dict(gate=0, progress=0, suffix=0)

    def _logits_oracle(self, o, recs):
        w = self.w
        rows = o.decode_rows(recs)
        return np.stack([O.lm_logits(r, self.dn["lm_head"], self.dn["final_norm"], w.rms_eps, w.dtype == "bf16")
                         for r in rows])

    def run(self, max_steps=None):
        w, rep = self.w, self.rep
        b, B, N = w.batch, w.block, self.N
        tok, msk = synth.make_prompt(w)
        tok_o = tok.numpy().astype(np.int64)
        msk_o = msk.numpy().copy()
        tok_g = tok.to(torch.int32).cuda()
        msk_g = msk.to(torch.uint8).cuda()
        for blk in range(w.n_blocks):
            start = w.prompt_len + blk * B
            entry = True
            nun = [0] * b
            for _ in range(B):
                if max_steps is not None and rep.steps >= max_steps:
                    return rep
                st = dict(t=rep.steps, block_index=blk, block_entry=entry, n_unmasked=list(nun))
                # ---- layer-0 inputs
                x0n = np.stack([O.embed_inputs(tok_o[s], msk_o[s], self.dn["embed"], self.dn["mask_emb"])
                                for s in range(b)])
                self.lib.embed(self.dg["embed"], self.dg["mask_emb"], tok_g, msk_g, self.gen.x0)
                torch.cuda.synchronize()
                assert np.array_equal(self.gen.x0.double().cpu().numpy(), x0n), "layer-0 inputs"
                # ---- calibration
                recs = self.orc.calibrate_step(x0n, nun, blk, entry)
                self.recs_p = [o.calibrate_step(x0n, nun, blk, entry) for o in self.pert]
                out = self.lib.calibrate_step(self.gen.x0, nun, blk, entry)
                torch.cuda.synchronize()
                ok = self._compare_step(st, recs, out)
                # ---- logits of the 2B rows
                lg_o = self._logits_oracle(self.orc, recs)
                lg_p = [self._logits_oracle(o, self.recs_p[i]) for i, o in enumerate(self.pert)]
                self.lib.decode_logits(self.dg["lm_head"], self.dg["final_norm"], self.gen.logits)
                torch.cuda.synchronize()
                lg_g = self.gen.logits.double().cpu().numpy()
                eps_row = np.zeros((b, 2 * B))
                for s in range(b):
                    zero_o = ~np.any(lg_o[s] != 0, axis=1)
                    zero_g = ~np.any(lg_g[s] != 0, axis=1)
                    if ok:
                        assert np.array_equal(zero_o, zero_g), f"rows without a fresh state (s={s})"
                    live = ~zero_o
                    rms = np.sqrt(np.mean(lg_o[s] ** 2, axis=1))
                    pdev = np.max([np.max(np.abs(p[s] - lg_o[s]), axis=1) for p in lg_p], axis=0) if lg_p \
                        else np.zeros(2 * B)
                    eps_row[s] = np.maximum(self.elem_tol * rms, BAND_FACTOR * pdev)
                    if ok and live.any():
                        e = rel_l2(lg_g[s][live], lg_o[s][live])
                        band = BAND_FACTOR * max([rel_l2(p[s][live], lg_o[s][live]) for p in lg_p] or [0.0])
                        self.max_logit_err = max(self.max_logit_err, e)
                        assert e < max(self.logit_tol, band), f"logits rel err {e} (s={s}, band {band})"
                # ---- gate
                self.theta_before = [[list(t) for t in q.theta] for q in self.orc.seqs]
                coms = self.orc.commit(lg_o, msk_o)
                self.coms_p = [o.commit(lg_p[i], msk_o) for i, o in enumerate(self.pert)]
                self.conf_tol = [c["conf"] * np.expm1(2 * eps_row[s]) + 1e-6 for s, c in enumerate(coms)]
                self.lib.commit(self.gen.logits, msk_g, self.gen.commit, self.gen.conf)
                torch.cuda.synchronize()
                cm_gate = self.gen.commit.cpu().numpy().astype(bool)
                if ok:
                    ok = self._compare_commit(st, coms, cm_gate)
                # ---- progress rule, greedy tokens, token update
                counts, left = self.lib.decode_tokens(self.gen.logits, self.gen.commit, tok_g, msk_g)
                cm_g = self.gen.commit.cpu().numpy().astype(bool)
                n_o = []
                for s in range(b):
                    co = coms[s]
                    cm = co["commit"].copy()
                    cur_masked = msk_o[s, start:start + B].copy()
                    cm[:B] = O.progress_rule(cm[:B], co["conf"][:B], cur_masked)
                    if cm[:B].sum() > co["commit"][:B].sum():
                        self.steps_by_kind["progress"] += 1
                    ids_o, id_margin = O.greedy_tokens(lg_o[s])
                    ids_g = O.greedy_tokens(lg_g[s])[0]
                    if ok and not np.array_equal(cm_g[s], cm):
                        # only the progress rule's choice can differ here
                        jo = int(np.argmax(cm & ~co["commit"])) if (cm & ~co["commit"]).any() else -1
                        jg = int(np.argmax(cm_g[s] & ~cm_gate[s])) if (cm_g[s] & ~cm_gate[s]).any() else -1
                        assert jo >= 0 and jg >= 0, f"progress rule (s={s}): oracle {jo}, library {jg}"
                        gap = abs(co["conf"][jo] - co["conf"][jg])
                        if gap <= self.conf_tol[s][jo] + self.conf_tol[s][jg] or gap < NEAR_TIE:
                            self._sensitivity_tie(f"progress rule (s={s})", gap, self.conf_tol[s][jo])
                            ok = False
                        else:
                            raise AssertionError(f"progress rule (s={s}): oracle {jo}, library {jg}, gap {gap:.3e}")
                    if ok:
                        both = cm & (np.arange(2 * B) + start < N)
                        bad = both & (ids_o != ids_g)
                        if bad.any():
                            top = np.max(np.abs(lg_o[s]), axis=1)
                            gap = id_margin * top
                            if np.all((gap[bad] <= 2 * eps_row[s][bad]) | (id_margin[bad] < NEAR_TIE)):
                                self._sensitivity_tie(f"greedy token (s={s})", float(np.min(gap[bad])), 0.0)
                                ok = False
                            else:
                                raise AssertionError(f"greedy tokens (s={s}): rows {np.nonzero(bad)[0]}, "
                                                     f"gaps {gap[bad]}, tolerance {2 * eps_row[s][bad]}")
                    n_o.append(O.apply_commits(tok_o[s], msk_o[s], cm, ids_o, start))
                left_o = [int(msk_o[s, start:start + B].sum()) for s in range(b)]
                if ok:
                    assert np.array_equal(tok_g.cpu().numpy(), tok_o), "tokens"
                    assert np.array_equal(msk_g.cpu().numpy().astype(bool), msk_o), "mask"
                    assert counts == n_o and left == left_o, f"counts {counts}/{n_o}, left {left}/{left_o}"
                    rep.compared += 1
                    self.commits_add_loop(coms, cm_gate, B)
                else:
                    if rep.diverged_at < 0:
                        rep.diverged_at = st["t"]
                    tok_g.copy_(torch.tensor(tok_o, dtype=torch.int32))
                    msk_g.copy_(torch.tensor(msk_o, dtype=torch.uint8))
                    self._import_oracle_state(st)
                    rep.resyncs += 1
                self.conf_tol = None
                rep.steps += 1
                nun = n_o
                entry = False
                if max(left_o) == 0:
                    break
            else:
                raise AssertionError(f"block {blk} not decoded within {B} steps")
        assert not msk_o[:, w.prompt_len:].any() and not msk_g.any().item(), "generation left masked tokens"
        return rep

    def commits_add_loop(self, coms, cm_gate, B):
        for co in coms:
            self.rep.commits += int(co["commit"].sum())
            self.steps_by_kind["gate"] += int(co["commit"][:B].sum())
            self.steps_by_kind["suffix"] += int(co["commit"][B:].sum())
