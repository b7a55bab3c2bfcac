"""The allocation-free attention entry point (polestar_attention_noalloc) gives
the same results as the allocating one (polestar_debug_attention) on two calls
in a row.  It is meant for callers that cannot let a library allocate device
memory -- applications that own all device memory through their own pool, or
latency-critical loops where cudaMalloc/cudaFree may synchronise the device --
so its scratch lives in fixed device arrays shared by every call.  This file
sorts last so that a run stopping at the first failure has run everything else."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_gb300.build import build
    build()


def test_noalloc_attention_matches_allocating_entry_point_twice():
    from drift_aware_kv_gb300 import polestar as P
    R, N, H, Hkv, dh = 136, 768, 32, 32, 128
    tracked = [r % 3 == 0 for r in range(R)]
    tr_dev = torch.tensor(tracked, dtype=torch.uint8, device="cuda")
    trm = np.array(tracked)
    kv = (1.6 * torch.randn(N, 2, Hkv * dh, generator=torch.Generator().manual_seed(1))).to(torch.bfloat16).cuda()
    q0 = (1.6 * torch.randn(R, H * dh, generator=torch.Generator().manual_seed(2))).to(torch.bfloat16).cuda()
    ref_prev, ref_lse = torch.zeros(R, H, N, device="cuda"), torch.zeros(R, H, device="cuda")
    new_prev, new_lse = torch.zeros(R, H, N, device="cuda"), torch.zeros(R, H, device="cuda")
    out_r = torch.empty(R, H * dh, dtype=torch.bfloat16, device="cuda")
    out_n = torch.empty_like(out_r)
    kl_r = torch.zeros(R, H, device="cuda")
    kl_n = torch.zeros(R, H, device="cuda")
    # baseline scores for the tracked rows through each entry point
    P.debug_attention(q0, kv, H, Hkv, tracked, ref_prev, ref_lse, 0, 1, out_r, kl_r)
    P.attention_noalloc(q0, kv, H, Hkv, tr_dev, new_prev, new_lse, 0, 1, out_n, kl_n)
    for call in range(2):
        g = torch.Generator().manual_seed(10 + call)
        q = (q0.float().cpu() + 0.08 * torch.randn(R, H * dh, generator=g)).to(torch.bfloat16).cuda()
        P.debug_attention(q, kv, H, Hkv, tracked, ref_prev, ref_lse, 1, 1, out_r, kl_r)
        P.attention_noalloc(q, kv, H, Hkv, tr_dev, new_prev, new_lse, 1, 1, out_n, kl_n)
        torch.cuda.synchronize()
        a = out_n.double().cpu().numpy()
        b = out_r.double().cpu().numpy()
        err = np.linalg.norm(a - b, axis=1) / np.linalg.norm(b, axis=1)
        assert err.max() < 8e-3, (call, err.max())
        ka, kb = kl_n.cpu().numpy()[trm], kl_r.cpu().numpy()[trm]
        assert np.all(np.abs(ka - kb) <= 1e-5 + 1e-3 * np.abs(kb)), (call, np.abs(ka - kb).max())
        assert torch.allclose(new_prev, ref_prev, rtol=1e-5, atol=1e-5)
        assert torch.allclose(new_lse, ref_lse, rtol=1e-5, atol=1e-5)


def test_noalloc_rejects_rows_beyond_the_static_table():
    from drift_aware_kv_gb300 import polestar as P
    q = torch.zeros(257, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(16, 2, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(P.PolestarError) as e:
        P.attention_noalloc(q, kv, 1, 1, None, None, None, 0, 0, out, None)
    assert e.value.status == P.ERR_INVALID_ARG
