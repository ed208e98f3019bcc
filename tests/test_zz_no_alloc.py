"""rkv_compress_noalloc, the entry point for callers that cannot allocate device
memory at the call (graph capture, foreign arenas, allocation-free serving loops):
it must produce exactly what rkv_compress produces with a caller workspace (records
and z bit for bit), on two calls in a row (its built-in scratch keeps the previous
call's bytes), and refuse problems whose scratch would not fit.  Kept in a file
pytest collects last."""
import numpy as np
import pytest
import torch

import rkv_workload as wl
from reference_residual_kv_gb300 import build, rkv

pytestmark = pytest.mark.gpu


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
        out.hdr.fill_(float("nan"))
        out.ref_idx.fill_(-7)
        out.z.fill_(float("nan"))
        rkv.rkv_compress_noalloc(p, kv, out.pool, W1, W2, W3, out.cache, out.z, out.status)
        torch.cuda.synchronize()
        assert out.device_status() == 0 and ref.device_status() == 0
        # the same kernels on the same inputs: every record bit for bit (the kernels
        # are deterministic; only where the scratch lives differs)
        assert torch.equal(out.ref_idx, ref.ref_idx)
        assert torch.equal(out.codes, ref.codes)
        assert torch.equal(out.hdr.view(torch.int32), ref.hdr.view(torch.int32))
        assert torch.equal(out.z.view(torch.int32), ref.z.view(torch.int32))


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
