"""The C-ABI library builds, loads and exports every function include/polestar.h
declares (no GPU needed: nothing here calls into the device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "polestar.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(polestar_[a-z_]+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("polestar_init", "polestar_calibrate_step", "polestar_commit", "polestar_release"):
        assert n in names


def test_library_exports_every_declared_symbol():
    from drift_aware_kv_gb300.build import build
    from drift_aware_kv_gb300 import polestar as P
    lib = ctypes.CDLL(build())
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(P.EXPORTED) <= set(_declared())


def test_init_rejects_bad_config_without_touching_the_device():
    from drift_aware_kv_gb300 import polestar as P
    from drift_aware_kv_gb300 import synth
    lib = P.load()
    cfg = P.make_config(synth.WORKLOADS["tiny_l1_d256_fp32"].replace(K=9))
    arr = (P.polestar_layer_weights * 1)()
    ctx = ctypes.c_void_p()
    st = lib.polestar_init(ctypes.byref(cfg), arr, None, None, ctypes.byref(ctx))
    assert st == P.ERR_INVALID_ARG and not ctx.value
    assert b"K must be" in lib.polestar_last_error(None)
    cfg = P.make_config(synth.WORKLOADS["tiny_l1_d256_fp32"])
    st = lib.polestar_init(ctypes.byref(cfg), arr, None, None, ctypes.byref(ctx))
    assert st == P.ERR_INVALID_ARG and b"NULL weight" in lib.polestar_last_error(None)
    lib.polestar_release(None)


def test_gemm_choice_without_a_device_is_an_error_not_a_crash():
    """The launch choice needs the device's SM count; with no device the call
    returns an error status instead of dividing by zero."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    from drift_aware_kv_gb300 import polestar as P
    with pytest.raises(P.PolestarError):
        P.gemm_choice(2560, [12288], 4096)


def test_staleness_entry_points_reject_bad_arguments_on_the_host():
    """KV-cache staleness (App. C.2) and the full-sequence forward check their
    arguments before any device work: these calls fail on a machine with no GPU
    exactly as on one with a GPU."""
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    E = ctypes.c_void_p(0x1000)
    buf = ctypes.c_void_p(0x2000)
    # head size not a multiple of 8, unknown dtype, negative rows, misaligned cache
    assert lib.polestar_kv_staleness(buf, buf, 4, 2, 12, P.BF16, E, None) == P.ERR_INVALID_ARG
    assert lib.polestar_kv_staleness(buf, buf, 4, 2, 16, 5, E, None) == P.ERR_INVALID_ARG
    assert lib.polestar_kv_staleness(buf, buf, -1, 2, 16, P.BF16, E, None) == P.ERR_INVALID_ARG
    assert lib.polestar_kv_staleness(ctypes.c_void_p(0x2004), buf, 4, 2, 16, P.BF16, E, None) == P.ERR_INVALID_ARG
    assert lib.polestar_kv_staleness(None, buf, 4, 2, 16, P.BF16, E, None) == P.ERR_INVALID_ARG
    # zero rows is an empty call: nothing to launch
    assert lib.polestar_kv_staleness(None, None, 0, 2, 16, P.BF16, None, None) == P.OK
    # more rows than one launch grid holds
    assert lib.polestar_kv_staleness(buf, buf, 1 << 31, 2, 16, P.BF16, E, None) == P.ERR_UNSUPPORTED
    # no context
    assert lib.polestar_full_forward(None, buf) == P.ERR_INVALID_ARG
    assert lib.polestar_cache_staleness(None, None, E) == P.ERR_INVALID_ARG


def _items(a0, na, b0, nb, max_rows, cap=None):
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    lib.polestar_debug_attention_items.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_void_p, ctypes.c_int32]
    lib.polestar_debug_attention_items.restype = ctypes.c_int32
    cap = cap if cap is not None else (na + nb) // max(1, max_rows) + 2
    buf = (ctypes.c_int32 * (4 * max(cap, 1)))()
    n = lib.polestar_debug_attention_items(a0, na, b0, nb, max_rows, buf, cap)
    return n, [tuple(buf[4 * i: 4 * i + 4]) for i in range(max(n, 0))]


@pytest.mark.parametrize("na,nb,max_rows", [(32, 104, 48), (32, 0, 48), (0, 13, 48), (136, 0, 128), (96, 8, 48),
                                            (1, 1, 1), (768, 0, 48), (5, 200, 7)])
def test_attention_work_items_cover_rows_once(na, nb, max_rows):
    """Host-side scheduling of the row attention (no device): the rows of one
    sequence, active rows [a0, a0 + na) then window/proxy rows [b0, b0 + nb), are
    cut into ceil(total / max_rows) items in order, each at most max_rows rows and
    within one row of each other, together covering every row exactly once."""
    a0, b0 = 1000, 5000
    n, items = _items(a0, na, b0, nb, max_rows)
    tot = na + nb
    assert n == -(-tot // max_rows)
    rows = []
    for x, cx, y, cy in items:
        rows += list(range(x, x + cx)) + list(range(y, y + cy))
        assert 1 <= cx + cy <= max_rows
        assert cy == 0 or (x + cx == a0 + na and y == b0)  # only the straddling item has two parts
    assert rows == list(range(a0, a0 + na)) + list(range(b0, b0 + nb))
    sizes = [cx + cy for _, cx, _, cy in items]
    assert max(sizes) - min(sizes) <= 1


def test_attention_work_items_reject_bad_arguments():
    assert _items(0, -1, 0, 4, 48)[0] == -1
    assert _items(0, 4, 0, 4, 0)[0] == -1
    assert _items(0, 200, 0, 0, 48, cap=2)[0] == -1  # needs 5 items
    assert _items(0, 0, 0, 0, 48)[0] == 0


def _window(prompt_len, gen_len, block, pre, suf, b):
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    lib.polestar_debug_window.argtypes = [ctypes.c_int32] * 6 + [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
    lib.polestar_debug_window.restype = ctypes.c_int32
    span = (ctypes.c_int32 * 2)()
    pos = (ctypes.c_int32 * 512)()
    n = lib.polestar_debug_window(prompt_len, gen_len, block, pre, suf, b, span, pos, 512)
    return n, (span[0], span[1]), list(pos[: max(n, 0)])


def test_library_window_equals_oracle_window_for_every_workload_block():
    """Local window (§4.1, clipped at the sequence ends): the library's host
    computation against the oracle's, for every block of every workload."""
    from drift_aware_kv_gb300 import synth
    from oracle import polestar_oracle as O
    for w in synth.WORKLOADS.values():
        orc = O.PolestarOracle.__new__(O.PolestarOracle)
        orc.cfg, orc.N = w, w.seq_len
        for b in range(w.n_blocks):
            n, span, pos = _window(w.prompt_len, w.gen_len, w.block, w.prefix_win, w.suffix_win, b)
            assert span == orc._span(b) and pos == orc.window(b) and n == len(pos)
            assert pos == synth.window_positions(w, b)


def test_window_edges_closed_form():
    # prompt shorter than the prefix window: the prefix is clipped at position 0
    n, span, pos = _window(16, 64, 32, 64, 32, 0)
    assert span == (16, 48) and pos == list(range(0, 16)) + list(range(48, 80))
    # last block: no suffix past the sequence end
    n, span, pos = _window(64, 128, 32, 64, 32, 3)
    assert span == (160, 192) and pos == list(range(96, 160))
    assert _window(64, 128, 32, 64, 32, 4)[0] == -1  # block index out of range


@pytest.mark.parametrize("tau,ns,expect", [
    (3, [1, 1, 1, 1, 1], [0, 0, 0, 1, 0]),      # cumulative count passes tau_upd at the 4th token
    (3, [4, 0, 4], [1, 0, 1]),                   # more than tau_upd in one step
    (3, [3, 0, 1, 3, 3], [0, 0, 1, 0, 1]),       # exactly tau_upd does not fire; reset after firing
    (0, [0, 1, 0, 2], [0, 1, 0, 1]),             # tau_upd = 0: any unmasked token fires
    (10 ** 6, [6] * 8, [0] * 8),                 # out of reach: never
])
def test_trigger_closed_form(tau, ns, expect):
    """The tau_upd trigger of §4.1 "Update Schedule": refresh after a step that
    unmasks more than tau_upd tokens, or once the tokens unmasked since the last
    refresh exceed tau_upd (this step's count included); the count restarts."""
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    lib.polestar_debug_trigger.argtypes = [ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    arr = (ctypes.c_int32 * len(ns))(*ns)
    out = (ctypes.c_uint8 * len(ns))()
    assert lib.polestar_debug_trigger(tau, arr, len(ns), out) == P.OK
    assert list(out) == expect
    neg = (ctypes.c_int32 * 1)(-1)
    assert lib.polestar_debug_trigger(tau, neg, 1, out) == P.ERR_INVALID_ARG


def test_stalled_wait_hook_without_context_is_an_argument_error():
    """Host-side argument check of the bounded-wait test hook (no device work)."""
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    assert lib.polestar_debug_stalled_wait(None, 1000) == P.ERR_INVALID_ARG


def test_closed_loop_entry_points_without_context_are_argument_errors():
    """Host-side argument checks of the closed-loop calls (no device work)."""
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    buf = ctypes.c_void_p(0x2000)
    n = (ctypes.c_int32 * 4)()
    assert lib.polestar_decode_logits(None, buf, buf, 1000, buf) == P.ERR_INVALID_ARG
    assert lib.polestar_decode_tokens(None, buf, 1000, buf, buf, buf, n, n) == P.ERR_INVALID_ARG
    assert lib.polestar_embed(None, buf, 1000, buf, buf, buf, buf) == P.ERR_INVALID_ARG


def test_batched_attention_hook_rejects_bad_arguments_on_the_host():
    """polestar_debug_attention_batch checks its sizes before any device work."""
    from drift_aware_kv_gb300 import polestar as P
    lib = P.load()
    lib.polestar_debug_attention_batch.restype = ctypes.c_int
    buf = ctypes.c_void_p(0x2000)
    args = lambda batch, N, H, Hkv, dh, R: (buf, buf, batch, N, H, Hkv, dh, R, None, None, None, 0, 0, buf, None,
                                            P.BF16, None)
    assert lib.polestar_debug_attention_batch(*args(0, 64, 4, 4, 128, 8)) == P.ERR_INVALID_ARG
    assert lib.polestar_debug_attention_batch(*args(2, 64, 6, 4, 128, 8)) == P.ERR_INVALID_ARG  # H % Hkv
    assert lib.polestar_debug_attention_batch(*args(2, 64, 4, 4, 96, 8)) == P.ERR_UNSUPPORTED   # head size
