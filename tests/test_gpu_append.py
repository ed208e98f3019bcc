"""GPU parity of the decode-time single-token write: appending the last tokens of a
sequence one at a time gives back the pool entries bit for bit, the reference sets of
the batch write, and records that match the fp64 oracle."""
import numpy as np
import pytest
import torch

import rkv_workload as wl
from reference_residual_kv_gb300 import rkv

from _gpu_common import CODE_BUDGET, check_tokens, gen_inputs, host_records, run_gpu

pytestmark = pytest.mark.gpu

C = wl.CONFIGS


@pytest.mark.parametrize("name,T,n_app", [
    ("tiny-fp32", 256, 24),                  # fp32 path
    ("llama3.1-8b-kv", 1000, 40),            # bf16 pool, INT4, 2 layers
    ("long-131k-fp8ref", 2048, 40),          # FP8 pool (stride 16)
    ("multimodal-8x4096-int2", 1024, 24),    # INT2, 8 sequences
])
def test_append_matches_batch_write_and_oracle(name, T, n_app):
    cfg = C[name].replace(L=min(C[name].L, 2), T=T)
    kv, w = gen_inputs(cfg)
    bufs, (kv_d, W1, W2, W3) = run_gpu(cfg, kv, w, want_z=False)
    before = host_records(cfg, bufs)
    pool_vec = bufs.ref_vec.clone()
    pool_nrm = bufs.ref_sqnorm.clone()
    t0 = T - n_app
    # wipe the records of tokens >= t0 and the pool rows of references at positions >= t0
    bufs.codes[:, t0:] = 0xAB
    bufs.hdr[:, t0:] = float("nan")
    bufs.ref_idx[:, t0:] = -7
    late = np.nonzero(bufs.ref_pos.cpu().numpy()[:bufs.n_ref] >= t0)[0]
    if late.size:
        bufs.ref_vec[:, late] = 0
        bufs.ref_sqnorm[:, late] = -1.0
    LB = cfg.L * cfg.B
    xs = kv_d.view(LB, T, -1)
    for t in range(t0, T):
        bufs.append(xs[:, t].contiguous(), t, W1, W2, W3)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    after = host_records(cfg, bufs)
    # the pool is back bit for bit
    assert torch.equal(bufs.ref_vec.view(torch.uint8), pool_vec.view(torch.uint8))
    assert torch.equal(bufs.ref_sqnorm, pool_nrm)
    # reference sets are the exact top-k in both writes
    assert np.array_equal(after["idx"][:, t0:], before["idx"][:, t0:])
    # records against the oracle
    report = {}
    for l in range(cfg.L):
        for b in range(cfg.B):
            check_tokens(cfg, kv[l][b], w[l], after, l * cfg.B + b, np.arange(t0, T), report=report)
    assert report["flips"] <= CODE_BUDGET * report["coords"], report
    # records of earlier tokens are untouched
    for key in ("idx", "q", "hdr"):
        assert np.array_equal(after[key][:, :t0], before[key][:, :t0])


def test_append_rejects_out_of_range_position():
    cfg = C["llama3.1-8b-kv"].replace(L=1, T=300)
    p = rkv.params_from_config(cfg)
    bufs = rkv.Buffers(p)
    x = torch.zeros((1, cfg.W), dtype=torch.bfloat16, device="cuda")
    for t in (-1, cfg.T):
        with pytest.raises(rkv.RkvError):
            bufs.append(x, t, x, x, x)


def test_append_full_size_sampled():
    # the benchmark's decode write: after the batch write of all 32 x 8192 tokens, the
    # last position of every layer appended in one call; its records equal the batch
    # write's and match the oracle on sampled layers
    cfg = C["llama3.1-8b-kv"]
    kv, w = gen_inputs(cfg)
    bufs, (kv_d, W1, W2, W3) = run_gpu(cfg, kv, w, want_z=False)
    before = host_records(cfg, bufs)
    t = cfg.T - 1
    LB = cfg.L * cfg.B
    bufs.codes[:, t] = 0xAB
    bufs.hdr[:, t] = float("nan")
    bufs.ref_idx[:, t] = -7
    bufs.append(kv_d.view(LB, cfg.T, -1)[:, t].contiguous(), t, W1, W2, W3)
    torch.cuda.synchronize()
    assert bufs.device_status() == 0
    after = host_records(cfg, bufs)
    assert np.array_equal(after["idx"][:, t], before["idx"][:, t])
    report = {}
    for l in (0, 13, 31):
        check_tokens(cfg, kv[l][0], w[l], after, l * cfg.B, np.array([t]), report=report)
    assert report["flips"] <= CODE_BUDGET * report["coords"], report
