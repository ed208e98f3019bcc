"""rkv_compress_noalloc, the entry point for callers that cannot allocate device
memory at the call (graph capture, foreign arenas, allocation-free serving loops):
it must produce what rkv_compress produces with a caller workspace, on two calls in a
row (its built-in scratch keeps the previous call's bytes), and refuse problems whose
scratch would not fit.  Kept in a file pytest collects last."""
import numpy as np
import pytest
import torch

import rkv_workload as wl
from reference_residual_kv_gb300 import build, rkv

pytestmark = pytest.mark.gpu

Z_TOL = 2e-2


def _dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _inputs(cfg):
    kv = np.stack([wl.layer_kv(cfg, l) for l in range(cfg.L)])
    w = [wl.layer_weights(cfg, l) for l in range(cfg.L)]
    W = [_dev(np.stack([x[i] for x in w]), cfg.kv_dtype) for i in range(3)]
    return _dev(kv, cfg.kv_dtype), W


@pytest.mark.parametrize("cfg", [
    wl.CONFIGS["llama3.1-8b-kv"].replace(L=1, T=1500),
    wl.CONFIGS["tiny-fp32"],
    wl.CONFIGS["long-131k-fp8ref"].replace(T=3000),
], ids=lambda c: c.name)
def test_noalloc_matches_workspace_entry_point(cfg):
    build.build()
    p = rkv.params_from_config(cfg)
    kv, (W1, W2, W3) = _inputs(cfg)

    ref = rkv.Buffers(p, want_z=True)               # the existing entry point, caller workspace
    ref.build_ref_pool(kv)
    ref.compress(kv, W1, W2, W3)

    for call in range(2):                            # second call reuses dirty scratch
        out = rkv.Buffers(p, want_z=True)
        out.build_ref_pool(kv)
        out.codes.fill_(0xAB)
        out.z.fill_(float("nan"))
        rkv.rkv_compress_noalloc(p, kv, out.pool, W1, W2, W3, out.cache, out.z, out.status)
        torch.cuda.synchronize()
        assert out.device_status() == 0 and ref.device_status() == 0
        assert torch.equal(out.ref_idx, ref.ref_idx)
        zr, zo = ref.z.cpu().numpy(), out.z.cpu().numpy()
        scale = np.maximum(np.abs(zr).max(axis=-1, keepdims=True), 1e-3 * np.abs(zr).max())
        assert np.all(np.abs(zo - zr) <= Z_TOL * scale)
        qr = ref.codes.cpu().numpy()
        qo = out.codes.cpu().numpy()
        assert (qr != qo).mean() <= 1e-3
        np.testing.assert_allclose(out.hdr.cpu().numpy(), ref.hdr.cpu().numpy(),
                                   rtol=0, atol=float(Z_TOL * scale.max()))


def test_noalloc_rejects_problems_beyond_its_scratch():
    build.build()
    cfg = wl.CONFIGS["llama3.1-8b-kv"].replace(L=4)          # ~170 MB of scratch
    p = rkv.params_from_config(cfg)
    _, _, ws = rkv.rkv_query_sizes(p)
    assert ws > 64 << 20
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pool = rkv.rkv_ref_pool(16, 16, 16, 16, 16)
    cache = rkv.rkv_cache(16, 16, 16)
    with pytest.raises(rkv.RkvError) as e:
        rkv.rkv_compress_noalloc(p, 16, pool, 16, 16, 16, cache, None, status)
    assert e.value.code == rkv.RKV_ERR_WORKSPACE
