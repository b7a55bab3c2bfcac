"""KV-cache staleness (App. C.2 "KV-Cache Staleness Metric") and the full-sequence
forward on the GPU, through the C ABI, against the oracle.

* polestar_kv_staleness on caller buffers: every row against the oracle's metric
  on the same values (fp32 and bf16; MHA, GQA and head size 64 shapes; identical,
  negated, orthogonal and zero rows; the LLaDA-8B cache of one sequence, 32
  layers x 768 positions, on sampled rows).
* polestar_full_forward: the recomputed cache against the oracle's full-sequence
  forward; a calibrating context refreshed by it has zero staleness; a call
  between polestar_calibrate_step and polestar_commit leaves that commit as it
  was.
* polestar_cache_staleness between a calibrating and a reference context equals
  the oracle's metric on the two caches read back, and over a trajectory
  Polestar's window cache stays fresher than a cache that is not refreshed.

Tolerance: E is computed in fp32 from values both sides hold exactly, so the
difference is rounding in sums of at most Hkv*dh products: 2e-5 absolute."""
import numpy as np
import pytest
import torch

from drift_aware_kv_gb300 import polestar as P
from drift_aware_kv_gb300 import synth
from oracle import polestar_oracle as O

pytestmark = pytest.mark.gpu
E_TOL = 2e-5


def _cache_pair(rows, Hkv, dh, dtype, seed, noise=0.3):
    g = torch.Generator(device="cpu").manual_seed(seed)
    a = torch.randn(rows, 2, Hkv * dh, generator=g)
    b = a + noise * torch.randn(rows, 2, Hkv * dh, generator=g)
    if rows >= 6:
        b[0] = a[0]                      # identical: E = 0
        b[1] = -a[1]                     # negated: E = 2
        a[2] = 0.0
        b[2] = 0.0                       # zero against zero: E = 0
        a[3, 0, :dh] = 0.0               # one zero head of K: cos 0 there
        b[4] = 4.0 * a[4]                # scaled by a power of two (exact in bf16): E = 0
        b[5] = torch.roll(a[5], 1, dims=-1)
    return a.to(dtype), b.to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rows,Hkv,dh", [(37, 32, 128), (19, 4, 128), (11, 4, 64), (6, 1, 8), (1, 2, 16)])
def test_kernel_matches_oracle(dtype, rows, Hkv, dh):
    a, b = _cache_pair(rows, Hkv, dh, dtype, seed=rows * 131 + dh)
    E = P.kv_staleness(a.cuda(), b.cuda(), Hkv).cpu().numpy()
    ref = O.kv_staleness(a.double().numpy(), b.double().numpy(), Hkv, dh)
    assert E.shape == (rows,)
    assert np.max(np.abs(E - ref)) <= E_TOL
    if rows >= 6:
        assert abs(E[0]) <= 1e-6 and abs(E[1] - 2) <= 1e-6 and abs(E[2]) <= 1e-6 and abs(E[4]) <= 1e-6


def test_kernel_full_llada_cache_sampled():
    """One sequence's LLaDA-8B cache (32 layers x 768 positions x 2 x 4096, bf16):
    every row computed on the device, 64 sampled rows checked against the oracle."""
    L, N, Hkv, dh = 32, 768, 32, 128
    g = torch.Generator(device="cuda").manual_seed(7)
    a = torch.randn(L * N, 2, Hkv * dh, device="cuda", generator=g).to(torch.bfloat16)
    step = 0.05 * torch.rand(L * N, 1, 1, device="cuda", generator=g)
    b = (a.float() + step * torch.randn(L * N, 2, Hkv * dh, device="cuda", generator=g)).to(torch.bfloat16)
    E = P.kv_staleness(a, b, Hkv)
    torch.cuda.synchronize()
    idx = torch.randperm(L * N, generator=torch.Generator().manual_seed(1))[:64]
    ref = O.kv_staleness(a[idx.cuda()].double().cpu().numpy(), b[idx.cuda()].double().cpu().numpy(), Hkv, dh)
    assert np.max(np.abs(E[idx.cuda()].cpu().numpy() - ref)) <= E_TOL
    assert float(E.min()) >= -1e-6 and float(E.max()) <= 2.0


def test_kernel_rejects_bad_arguments():
    lib = P.load()
    a = torch.zeros(4, 2, 64, device="cuda")
    E = torch.empty(4, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    import ctypes as C
    args = lambda dh, dt=P.FP32: (C.c_void_p(a.data_ptr()), C.c_void_p(a.data_ptr()), 4, 8, dh, dt,  # noqa: E731
                                 C.c_void_p(E.data_ptr()), C.c_void_p(s))
    assert lib.polestar_kv_staleness(*args(12)) == P.ERR_INVALID_ARG      # head size not a multiple of 8
    assert lib.polestar_kv_staleness(*args(8, 7)) == P.ERR_INVALID_ARG    # unknown dtype
    bad = (C.c_void_p(a.data_ptr() + 4),) + args(8)[1:]
    assert lib.polestar_kv_staleness(*bad) == P.ERR_INVALID_ARG           # misaligned
    assert lib.polestar_kv_staleness(*args(8)) == P.OK


def _read_kv(lib, w):
    dt = synth.torch_dtype(w)
    return np.stack([lib.read(P.BUF_KV, l, (w.batch, w.seq_len, 2, w.n_kv_heads * w.head_dim), dt)
                     .double().numpy() for l in range(w.n_layers)])


def _contexts(w, n):
    W = synth.make_weights(w, "cpu")
    Wg = [{k: v.cuda() for k, v in lw.items()} for lw in W]
    return W, Wg, [P.Polestar(w if i != 1 else w.replace(tau_upd=10 ** 6), Wg) for i in range(n)]


@pytest.mark.parametrize("name,kv_tol", [("tiny_l1_d256_fp32", 1e-5), ("mini_l2_d512_bf16", 1e-2),
                                         ("mini_gqa_l2_d448_bf16", 1e-2)])
def test_full_forward_and_cache_staleness(name, kv_tol):
    """Contexts: 0 = Polestar, 1 = no refresh within blocks, 2 = reference
    (polestar_full_forward every step), 3 = Polestar with a full forward slipped
    in between calibrate_step and commit at one step."""
    w = synth.WORKLOADS[name].replace(n_layers=2, n_steps=10)
    W, Wg, (pol, none, ref, mix) = _contexts(w, 4)
    orc = O.PolestarOracle(w, O.weights_to_numpy(W))
    tr = synth.Trajectory(w)
    dt = synth.torch_dtype(w)
    win_pol, win_none = [], []
    probe = 3
    while True:
        st = tr.next_step()
        if st is None:
            break
        x0 = st["x0"].to(dt).cuda()
        for c in (pol, none, mix):
            c.calibrate_step(x0, st["n_unmasked"], st["block_index"], st["block_entry"])
        ref.full_forward(x0)
        if st["t"] == probe:
            mix.full_forward(x0)
        lg = st["logits"].cuda()
        mk = st["masked"].to(torch.uint8).cuda()
        masks = []
        for c in (pol, mix):
            cm = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
            conf = torch.zeros(w.batch, 2 * w.block, device="cuda")
            c.commit(lg, mk, cm, conf)
            masks.append((cm.cpu(), conf.cpu(), c.read(P.BUF_DREL, 0, (w.batch, 2 * w.block), torch.float32)))
        cm_n = torch.zeros(w.batch, 2 * w.block, dtype=torch.uint8, device="cuda")
        none.commit(lg, mk, cm_n)
        torch.cuda.synchronize()
        if st["t"] <= probe:  # identical up to and including the probed commit
            for x, y in zip(masks[0], masks[1]):
                assert torch.equal(x, y)
        # reference cache = the oracle's full-sequence forward of this x0
        kv_ref = _read_kv(ref, w)
        for s in range(w.batch):
            o = orc.full_forward_kv(st["x0"][s].to(dt).double().numpy())
            for l in range(w.n_layers):
                e = np.linalg.norm(kv_ref[l, s] - o[l].reshape(kv_ref[l, s].shape)) / np.linalg.norm(o[l])
                assert e < kv_tol, (l, s, e)
        # device staleness = the oracle's metric on the two caches read back
        for c, acc in ((pol, win_pol), (none, win_none)):
            E = c.staleness(ref).cpu().numpy()
            kv = _read_kv(c, w)
            E_o = O.kv_staleness(kv, kv_ref, w.n_kv_heads, w.head_dim).reshape(E.shape)
            assert np.max(np.abs(E - E_o)) <= E_TOL
            if not st["block_entry"]:
                acc.append(E[:, 0, synth.window_positions(w, st["block_index"])].mean(axis=1))
        if st["t"] == probe:
            Em = mix.staleness(ref).cpu().numpy()
            assert np.max(np.abs(Em)) <= 1e-6  # refreshed cache: bit-equal recompute
    assert len(win_pol) >= 5
    assert np.all(np.mean(win_pol, axis=0) < np.mean(win_none, axis=0))
    for c in (pol, none, ref, mix):
        c.close()
