"""Pins of the fp64 oracle to facts outside itself: brute force, closed forms, library
routines, exact identities and the numbers the ResidualKV reading notes print.

Each test names the plausible oracle mistake it would catch.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import rkv_workload as wl
from reference_residual_kv_gb300 import storage

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- schedule (§2.6)
def test_fixed_schedule_positions():
    # every s-th token from `first`; catches an off-by-one in the stride loop
    assert oracle.fixed_schedule(20, 8).tolist() == [0, 8, 16]
    assert oracle.fixed_schedule(17, 8, 3).tolist() == [3, 11]
    assert oracle.fixed_schedule(0, 8).tolist() == []
    ref = oracle.fixed_schedule(131072, 16)
    assert ref.size == 8192 and ref[-1] == 131072 - 16


def test_dynamic_schedule_table6_counts():
    # Table VI reference counts at 262K for five alphas, all five reproduced exactly
    # under the fitted reading (262144 - 256 positions); catches a wrong floor
    # argument or recurrence sign.
    g = _golden("table6_ref_counts.json")
    got = [oracle.dynamic_schedule(g["T"], g["s0"], a, g["n_sink"]).size for a in g["alpha"]]
    assert got == g["n_ref"]


def test_dynamic_schedule_table6_unfitted_reading():
    # Table VI [RKV §4.6] over the whole 262144-position context with no positions
    # dropped: every alpha > 0 count is within 1 of the table, and alpha = 0 gives the
    # fixed-stride count ceil(T / s0) (the table prints 26 fewer; only the fitted
    # reading above matches it exactly)
    g = _golden("table6_ref_counts.json")
    T = g["unfitted_T"]
    got = [oracle.dynamic_schedule(T, g["s0"], a, g["n_sink"]).size for a in g["alpha"]]
    assert got[0] == -(-T // g["s0"])
    for n, ref in zip(got[1:], g["n_ref"][1:]):
        assert abs(n - ref) <= 1, (got, g["n_ref"])


def test_dynamic_schedule_alpha0_is_fixed_and_log_growth():
    # alpha = 0 reduces to the fixed stride (§2.6); for alpha > 0 the count follows the
    # page's closed form log_{1+a}(1 + a (T - n_sink)/s0) up to the floor's effect.
    assert np.array_equal(oracle.dynamic_schedule(5000, 10, 0.0), oracle.fixed_schedule(5000, 10))
    for a in (0.01, 0.05, 0.1):
        T = 200000
        approx = math.log(1 + a * T / 10) / math.log(1 + a)
        n = oracle.dynamic_schedule(T, 10, a).size
        assert approx * 0.9 <= n <= approx * 1.3


# ---------------------------------------------------------------- FP8 E4M3 (OCP OFP8)
def test_fp8_format_properties():
    # catches a wrong bias, a wrong subnormal scale or a missing NaN code
    dec = oracle.fp8_decode(np.arange(256, dtype=np.uint8))
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0          # largest finite
    assert dec[0x01] == 2.0 ** -9                                 # smallest subnormal
    assert dec[0x08] == 2.0 ** -6                                 # smallest normal
    assert dec[0x38] == 1.0                                       # exponent bias 7
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert np.isnan(dec).sum() == 2
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0)                               # monotone codes
    # every finite code round-trips
    fin = np.nonzero(~np.isnan(dec))[0].astype(np.uint8)
    assert np.array_equal(oracle.fp8_encode(dec[fin]), fin)       # encode(decode(b)) == b


def test_fp8_rne_ties_and_saturation():
    # ties to even, saturation at 448; catches round-half-up or overflow to NaN
    e = oracle.fp8_encode
    assert e(np.array([1.0625]))[0] == 0x38       # halfway 1 and 1.125 -> even mantissa (1.0)
    assert e(np.array([1.1875]))[0] == 0x3A       # halfway 1.125 and 1.25 -> 1.25
    assert e(np.array([2.0 ** -10]))[0] == 0x00   # halfway 0 and 2^-9 -> 0
    assert e(np.array([3 * 2.0 ** -10]))[0] == 0x02  # halfway 2^-9 and 2^-8 -> 2^-8
    assert e(np.array([1e6]))[0] == 0x7E and e(np.array([-1e6]))[0] == 0xFE
    assert e(np.array([-0.0]))[0] == 0x80


def test_fp8_matches_torch_cast_on_all_bf16():
    # library routine: torch's float8_e4m3fn cast (round to nearest even) on every
    # bf16 bit pattern inside the finite range
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        x = wl.bf16_bits_to_f32(bits).astype(np.float64)
    keep = np.isfinite(x) & (np.abs(x) < 464.0)
    x = x[keep]
    ours = oracle.fp8_encode(x)
    ref = torch.tensor(x, dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------- retrieval (§2.2)
def _brute_topk(x, refs, k):
    """All k-subsets; the unique one whose every member beats every non-member under
    (distance, slot) order.  Exact integer distances."""
    n = len(refs)
    d = [sum((int(a) - int(b)) ** 2 for a, b in zip(x, r)) for r in refs]
    ki = min(k, n)
    best = None
    for S in itertools.combinations(range(n), ki):
        rest = [j for j in range(n) if j not in S]
        if all((d[s], s) < (d[j], j) for s in S for j in rest):
            assert best is None
            best = S
    sums = {S: sum(d[s] for s in S) for S in itertools.combinations(range(n), ki)}
    assert sums[best] == min(sums.values())
    return list(best), d


@pytest.mark.parametrize("seed", range(40))
def test_retrieve_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    W = int(rng.integers(1, 5))
    refs = rng.integers(-3, 4, size=(n, W))      # small integers: many exact ties
    x = rng.integers(-3, 4, size=W)
    k = int(rng.integers(1, 6))
    best, d = _brute_topk(x, refs, k)
    idx, ki, dk = oracle.retrieve(x.astype(float), refs.astype(float), k)
    assert ki == min(k, n)
    assert idx[:ki].tolist() == sorted(best)
    assert all(v == -1 for v in idx[ki:])
    srt = sorted(d)
    assert dk[0] == srt[ki - 1]
    assert dk[1] == (srt[ki] if n > ki else math.inf)


def test_retrieve_duplicate_references_prefer_lower_slot():
    x = np.zeros(3)
    refs = np.array([[5, 0, 0], [1, 0, 0], [1, 0, 0], [0, 1, 0], [1, 0, 0], [0, 0, 1]], float)
    idx, ki, _ = oracle.retrieve(x, refs, 4)
    # distances 25,1,1,1,1,1: the four lowest slots among the equal ones
    assert idx.tolist() == [1, 2, 3, 4]


def test_k_i_is_min_k_pool_on_early_tokens():
    # k_i = min(k, |pool|) (§2.1 symbol table); pool = references strictly before t
    cfg = wl.CONFIGS["tiny-fp32"]
    kv = wl.layer_kv(cfg, 0)[0]
    w = wl.layer_weights(cfg, 0)
    toks = np.arange(0, 40)
    o = oracle.compress_tokens(cfg, kv, w, toks)
    for t, ki, row in zip(toks, o["ki"], o["idx"]):
        if t % 8 == 0:
            assert ki == 1 and row[0] == t // 8          # a reference keeps itself
        else:
            pool = (t + 7) // 8
            assert ki == min(4, pool)
            assert row[:ki].max() < pool                 # causal: only earlier refs
            assert list(row[:ki]) == sorted(row[:ki])


# ---------------------------------------------------------------- mean (§2.2, Thm IV.1)
def test_theorem_iv1_identity_on_oracle_means():
    # rho^2 = ||Delta||^2 + V (Theorem IV.1) holds iff the mean is the arithmetic mean
    # of the chosen references; catches a wrong divisor or a wrong reference subset.
    cfg = wl.CONFIGS["tiny-fp32"]
    kv = wl.layer_kv(cfg, 0)[0]
    w = wl.layer_weights(cfg, 0)
    ref_pos = oracle.schedule(cfg)
    refs, _ = oracle.stored_refs(cfg, kv, ref_pos)
    toks = np.array([t for t in range(cfg.T) if t % 8])
    o = oracle.compress_tokens(cfg, kv, w, toks, want_mean=True)
    x64 = kv.astype(np.float64)
    for n, t in enumerate(toks):
        R = refs[o["idx"][n][: o["ki"][n]]]
        m = o["mean"][n]
        rho2 = np.mean(np.sum((x64[t] - R) ** 2, axis=1))
        V = np.mean(np.sum((R - m) ** 2, axis=1))
        D = np.sum((x64[t] - m) ** 2)
        assert abs(rho2 - (D + V)) <= 1e-12 * rho2
    # and a wrong mean breaks it (the identity is a real check)
    R = refs[[0, 1, 2]]
    bad = R.mean(0) * 1.01
    rho2 = np.mean(np.sum((x64[40] - R) ** 2, axis=1))
    assert abs(rho2 - (np.sum((x64[40] - bad) ** 2) + np.mean(np.sum((R - bad) ** 2, 1)))) > 1e-6


def test_mean_exact_small_cases():
    refs = np.array([[1.0, 2.0], [3.0, 6.0], [5.0, -2.0], [7.0, 10.0]])
    assert np.array_equal(oracle.mean(refs, [1, -1, -1, -1]), [3.0, 6.0])
    assert np.array_equal(oracle.mean(refs, [0, 1, 2, 3]), [4.0, 4.0])
    assert np.array_equal(oracle.mean(refs, [0, 2, -1, -1]), [3.0, 0.0])
    assert np.array_equal(oracle.mean(refs, [-1, -1, -1, -1]), [0.0, 0.0])


# ---------------------------------------------------------------- compressor (§2.3)
def test_fc_scalar_golden():
    g = _golden("fc_scalar.json")
    for c in g["cases"]:
        out = oracle.fc([c["x"]], [[c["w1"]]], [[c["w2"]]], [[c["w3"]]])
        assert out[0] == pytest.approx(c["f"], rel=1e-15, abs=1e-300)


def test_fc_matches_torch_swiglu_nonsquare():
    # library routine: torch.nn.functional.silu + matmul in fp64, with 2d_k != d_ff != d_c
    # so a transposed weight cannot pass
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    W, F, C = 6, 5, 3
    x = rng.standard_normal(W)
    Wc1, Wc2, Wc3 = rng.standard_normal((W, F)), rng.standard_normal((W, F)), rng.standard_normal((F, C))
    got = oracle.fc(x, Wc1.T, Wc2.T, Wc3.T)
    tx = torch.tensor(x)
    ref = (torch.nn.functional.silu(tx @ torch.tensor(Wc1)) * (tx @ torch.tensor(Wc2))) @ torch.tensor(Wc3)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-13, atol=1e-13)


def test_fc_gate_is_on_the_first_projection():
    # Swish gates x W_c1 only: driving x W_c1 very negative silences the output even
    # when x W_c2 is large, while the swapped roles do not.
    W1t = np.array([[-50.0]])
    W2t = np.array([[50.0]])
    W3t = np.array([[1.0]])
    assert abs(oracle.fc([1.0], W1t, W2t, W3t)[0]) < 1e-15
    assert oracle.fc([1.0], W2t, W1t, W3t)[0] < -2000


def test_fc_zero_and_linearity_in_w3():
    rng = np.random.default_rng(3)
    W1t, W2t, W3t = rng.standard_normal((5, 4)), rng.standard_normal((5, 4)), rng.standard_normal((3, 5))
    assert np.all(oracle.fc(np.zeros(4), W1t, W2t, W3t) == 0.0)
    x = rng.standard_normal(4)
    np.testing.assert_allclose(oracle.fc(x, W1t, W2t, 2 * W3t), 2 * oracle.fc(x, W1t, W2t, W3t), rtol=1e-14)


def test_encoder_is_difference_of_encodings():
    # §2.3: z = f_c(kv) - f_c(mean), which is neither f_c(kv - mean) nor the mean of
    # f_c over the references; z = 0 exactly when kv equals its (single) reference.
    cfg = wl.CONFIGS["tiny-fp32"]
    kv = wl.layer_kv(cfg, 0)[0].copy()
    kv[3] = kv[0]                                 # token 3's pool is {ref 0}: k = 1
    w = wl.layer_weights(cfg, 0)
    W1, W2, W3 = oracle.weights_f64(cfg, w)
    ref_pos = oracle.schedule(cfg)
    refs, _ = oracle.stored_refs(cfg, kv, ref_pos)
    toks = np.array([3, 50, 77, 201])
    o = oracle.compress_tokens(cfg, kv, w, toks, want_mean=True)
    assert np.all(o["z"][0] == 0.0) and np.all(o["delta"][0] == 0.0) and np.all(o["zmin"][0] == 0.0)
    x64 = kv.astype(np.float64)
    for n, t in enumerate(toks[1:], start=1):
        m = o["mean"][n]
        z_def = oracle.fc(x64[t], W1, W2, W3) - oracle.fc(m, W1, W2, W3)
        np.testing.assert_allclose(o["z"][n], z_def, rtol=0, atol=1e-12)
        wrong1 = oracle.fc(x64[t] - m, W1, W2, W3)
        R = refs[o["idx"][n][: o["ki"][n]]]
        wrong2 = oracle.fc(x64[t], W1, W2, W3) - np.mean([oracle.fc(r, W1, W2, W3) for r in R], 0)
        scale = np.abs(z_def).max()
        assert np.abs(wrong1 - z_def).max() > 0.05 * scale
        assert np.abs(wrong2 - z_def).max() > 1e-3 * scale


# ---------------------------------------------------------------- quantiser (§2.4)
def test_quantize_golden_cases():
    g = _golden("quant_cases.json")
    for c in g["cases"]:
        q, zmin, delta = oracle.quantize(c["z"], c["group"], c["bits"])
        assert q.tolist() == c["q"]
        np.testing.assert_allclose(zmin, c["zmin"], rtol=0, atol=0)
        np.testing.assert_allclose(delta, c["delta"], rtol=1e-15)
        zq = oracle.dequantize(q, zmin, delta, c["group"])
        np.testing.assert_allclose(zq, c["zq"], rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("d_c,group", [(64, 32), (512, 32), (70, 32), (5, 8)])
def test_quantize_invariants_and_error_bound(bits, d_c, group):
    rng = np.random.default_rng(bits * 1000 + d_c)
    qmax = (1 << bits) - 1
    for rep in range(20):
        z = rng.standard_normal(d_c) * rng.uniform(0.01, 10)
        if rep == 0:
            z[:group] = 1.25                        # a constant group
        q, zmin, delta = oracle.quantize(z, group, bits)
        zq = oracle.dequantize(q, zmin, delta, group)
        assert q.max() <= qmax
        for g in range(zmin.size):
            sl = slice(g * group, min(d_c, (g + 1) * group))
            zg = z[sl]
            if zg.max() == zg.min():
                assert delta[g] == 0 and np.all(q[sl] == 0) and np.all(zq[sl] == zg)
                continue
            assert np.all(np.abs(zg - zq[sl]) <= delta[g] / 2 * (1 + 1e-12))
            assert q[sl][np.argmin(zg)] == 0 and q[sl][np.argmax(zg)] == qmax
        # §2.8 quantisation bound: ||e_q|| <= sqrt(sum |G| range^2)/(2(2^b-1)) <= sqrt(g/2)/(2^b-1) ||z||
        e = np.linalg.norm(zq - z)
        sizes = [min(d_c, (g + 1) * group) - g * group for g in range(zmin.size)]
        ranges = [np.ptp(z[g * group: g * group + s]) for g, s in enumerate(sizes)]
        b1 = math.sqrt(sum(s * r * r for s, r in zip(sizes, ranges))) / (2 * qmax)
        b2 = math.sqrt(group / 2) / qmax * np.linalg.norm(z)
        assert e <= b1 * (1 + 1e-12) and b1 <= b2 * (1 + 1e-12)


# ---------------------------------------------------------------- read path (§2.7)
def test_gather_returns_reference_for_reference_tokens_and_standalone_equals_full():
    cfg = wl.CONFIGS["tiny-fp32"]
    kv = wl.layer_kv(cfg, 0)[0]
    w = wl.layer_weights(cfg, 0)
    ref_pos = oracle.schedule(cfg)
    refs, _ = oracle.stored_refs(cfg, kv, ref_pos)
    toks = np.arange(cfg.T)
    o = oracle.compress_tokens(cfg, kv, w, toks, want_mean=True)
    zq, mn = oracle.gather(cfg, refs, o["q"], o["zmin"], o["delta"], o["idx"], toks)
    # standalone mode = every token restored (§2.7): the means equal the write path's
    np.testing.assert_allclose(mn, o["mean"], rtol=0, atol=1e-15)
    for t in ref_pos:
        assert np.array_equal(mn[t], refs[t // 8]) and np.all(zq[t] == 0)
    # sparse read touches only the selected rows: poisoning others changes nothing
    sel = np.array([5, 17, 100, 255])
    q2, zmin2, d2, idx2 = o["q"].copy(), o["zmin"].copy(), o["delta"].copy(), o["idx"].copy()
    other = np.setdiff1d(toks, sel)
    q2[other] = 255
    zmin2[other] = np.nan
    d2[other] = np.nan
    idx2[other] = 10 ** 6
    a = oracle.gather(cfg, refs, q2, zmin2, d2, idx2, sel)
    b = oracle.gather(cfg, refs, o["q"], o["zmin"], o["delta"], o["idx"], sel)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fp8_reference_round_trip_is_used_for_retrieval():
    # §2.5 (Sec. IV-B): encoder and decoder use the stored references; with FP8 refs
    # the pool the oracle searches is the FP8-decoded one
    cfg = wl.CONFIGS["long-131k-fp8ref"].replace(T=512, L=1)
    kv = wl.layer_kv(cfg, 0)[0]
    ref_pos = oracle.schedule(cfg)
    refs, codes = oracle.stored_refs(cfg, kv, ref_pos)
    assert codes.dtype == np.uint8
    np.testing.assert_array_equal(refs, oracle.fp8_decode(codes))
    assert not np.array_equal(refs, wl.stored_to_f64(kv[ref_pos], "bf16"))


# ---------------------------------------------------------------- KR accounting (§3.3)
def test_keep_ratio_worked_example():
    g = _golden("kr_worked_example.json")
    assert storage.q_b(4) == g["q_b"]["q4"] and storage.q_b(2) == g["q_b"]["q2"]
    e = g["kr_example"]
    kr = storage.paper_keep_ratio(e["beta"], e["rho_ref"], e["dc_over_2dk"], e["bits"])
    assert abs(kr - e["kr"]) <= e["tolerance"]


def test_record_bytes_layout():
    # INT4, d_c = 512: 256 B codes + 16 groups x 8 B extremes + 4 x 4 B slots
    assert storage.record_bytes(512, 4) == 256 + 128 + 16
    assert storage.record_bytes(512, 2) == 128 + 128 + 16


# ------------------------------------------------------------------ restore (f_d, RoPE)
def test_rope_closed_forms_and_pair_layout():
    D = 4
    # position 0 is the identity
    x = np.array([0.3, -1.2, 2.0, 0.7])
    assert np.array_equal(oracle.rope(x, 0.0, 10000.0), x)
    # pair 0 has theta = 1: (1, 0) at position p becomes (cos p, sin p)
    for p in (1.0, 2.0, 7.0):
        r = oracle.rope([1.0, 0.0, 0.0, 0.0], p, 10000.0)
        assert np.allclose(r, [math.cos(p), math.sin(p), 0.0, 0.0], atol=1e-15)
    # base 4, D = 4: pair 1 has theta = 4^(-1/2) = 1/2; (0, 1) -> (-sin, cos)
    r = oracle.rope([0.0, 0.0, 0.0, 1.0], 3.0, 4.0)
    assert np.allclose(r, [0.0, 0.0, -math.sin(1.5), math.cos(1.5)], atol=1e-15)
    # the rotated pairs are consecutive coordinates: energy never leaves its pair
    rng = np.random.default_rng(5)
    v = rng.standard_normal(128)
    r = oracle.rope(v, 1234.0, 10000.0)
    assert np.allclose(r[0::2] ** 2 + r[1::2] ** 2, v[0::2] ** 2 + v[1::2] ** 2, rtol=1e-12)


def test_rope_relative_position_property():
    # <R(m) q, R(n) k> = <R(m - n) q, k>: attention scores depend on m - n only
    rng = np.random.default_rng(6)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n in ((5.0, 3.0), (1000.0, 17.0), (131071.0, 131000.0)):
        lhs = float(oracle.rope(q, m, 10000.0) @ oracle.rope(k, n, 10000.0))
        rhs = float(oracle.rope(q, m - n, 10000.0) @ k)
        assert abs(lhs - rhs) <= 1e-9 * (np.abs(q).sum() * np.abs(k).sum()), (m, n, lhs, rhs)


def test_decoder_unit_vectors_select_weight_columns():
    rng = np.random.default_rng(7)
    Wd = rng.standard_normal((12, 5))        # out-major [W][d_c]
    for j in range(5):
        e = np.zeros(5)
        e[j] = 1.0
        assert np.array_equal(oracle.decode(e, Wd), Wd[:, j])
    assert np.array_equal(oracle.decode(np.zeros(5), Wd), np.zeros(12))
    assert np.array_equal(oracle.decode([2.0, 0, 0, 0, -1.0], Wd), 2.0 * Wd[:, 0] - Wd[:, 4])


def _restore_case(T=6, n_ref=3, seed=8):
    cfg = wl.Config("restore-pin", seed=0, L=1, B=1, T=T, N=2, D=8, d_ff=8, d_c=64, k=4,
                    group=32, bits=4, kv_dtype="f32", ref_dtype="f32", rope_base=10000.0)
    rng = np.random.default_rng(seed)
    refs = rng.standard_normal((n_ref, cfg.W))
    Wd = rng.standard_normal((cfg.W, cfg.d_c)) * 0.1
    q = rng.integers(0, 16, (T, cfg.d_c)).astype(np.uint8)
    zmin = rng.standard_normal((T, 2)) * 0.1
    delta = rng.uniform(0.0, 0.05, (T, 2))
    idx = np.full((T, 4), -1, np.int32)
    return cfg, refs, Wd, q, zmin, delta, idx


def test_restore_reference_token_is_the_rotated_reference():
    cfg, refs, Wd, q, zmin, delta, idx = _restore_case()
    dk = cfg.N * cfg.D
    # token 4 is a reference record: own slot, z = 0 (codes 0, extremes {0, 0})
    idx[4, 0] = 2
    q[4] = 0
    zmin[4] = 0.0
    delta[4] = 0.0
    K, V = oracle.restore(cfg, refs, q, zmin, delta, idx, Wd, np.array([4], np.int32))
    assert np.array_equal(V[0], refs[2, dk:])                   # the value half, unrotated
    for h in range(cfg.N):                                       # each key head, rotated at 4
        want = oracle.rope(refs[2, h * cfg.D:(h + 1) * cfg.D], 4.0, cfg.rope_base)
        assert np.allclose(K[0, h * cfg.D:(h + 1) * cfg.D], want, rtol=0, atol=1e-14)


def test_restore_moves_only_keys_with_position_and_is_affine_in_the_minima():
    cfg, refs, Wd, q, zmin, delta, idx = _restore_case()
    dk = cfg.N * cfg.D
    # tokens 1 and 5 carry the same record: same V, keys rotated by the position gap
    idx[1, :2] = [0, 2]
    idx[5] = idx[1]
    q[5], zmin[5], delta[5] = q[1], zmin[1], delta[1]
    K, V = oracle.restore(cfg, refs, q, zmin, delta, idx, Wd, np.array([1, 5], np.int32))
    assert np.array_equal(V[0], V[1])
    for h in range(cfg.N):
        k1 = K[0, h * cfg.D:(h + 1) * cfg.D]
        assert np.allclose(oracle.rope(k1, 4.0, cfg.rope_base), K[1, h * cfg.D:(h + 1) * cfg.D],
                           rtol=0, atol=1e-12)
    # raising every group minimum by c adds f_d(c 1) = c * (row sums of W_d) before RoPE
    c = 0.25
    K2, V2 = oracle.restore(cfg, refs, q, zmin + c, delta, idx, Wd, np.array([1], np.int32))
    shift = c * Wd.sum(axis=1)
    assert np.allclose(V2[0] - V[0], shift[dk:], rtol=0, atol=1e-12)
    for h in range(cfg.N):
        s = slice(h * cfg.D, (h + 1) * cfg.D)
        got = K2[0, s] - K[0, s]
        assert np.allclose(got, oracle.rope(shift[:dk][s], 1.0, cfg.rope_base), rtol=0, atol=1e-12)
    # the mean of the chosen references enters with weight 1/k_i
    idx2 = idx.copy()
    idx2[1, :2] = [0, 2]
    K3, V3 = oracle.restore(cfg, refs, q, zmin, delta, idx2, Wd, np.array([1], np.int32))
    refs2 = refs.copy()
    refs2[0] += 1.0
    K4, V4 = oracle.restore(cfg, refs2, q, zmin, delta, idx2, Wd, np.array([1], np.int32))
    assert np.allclose(V4[0] - V3[0], 0.5, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ sparse attention
def test_attention_closed_forms():
    rng = np.random.default_rng(9)
    D, N = 8, 2
    V = rng.standard_normal((5, N * D))
    K = rng.standard_normal((5, N * D))
    # uniform scores (q = 0): the mean of the selected values, per KV head
    o = oracle.attention(np.zeros((4, D)), K, V, N)
    for j in range(4):
        h = j // 2
        assert np.allclose(o[j], V[:, h * D:(h + 1) * D].mean(axis=0), rtol=0, atol=1e-14)
    # one selected token: its value row
    valid = np.array([0, 0, 1, 0, 0], np.int32)
    o = oracle.attention(rng.standard_normal((4, D)), K, V, N, valid)
    for j in range(4):
        assert np.array_equal(o[j], V[2, (j // 2) * D:(j // 2 + 1) * D])
    # two tokens, scores a/sqrt(D) and 0: weights e^s / (e^s + 1)
    a = 3.0
    K2 = np.zeros((2, N * D))
    K2[0, 0] = 1.0
    q = np.zeros((4, D))
    q[0, 0] = a
    o = oracle.attention(q, K2, V[:2], N)
    s = a / math.sqrt(D)
    want = (math.exp(s) * V[0, :D] + V[1, :D]) / (math.exp(s) + 1.0)
    assert np.allclose(o[0], want, rtol=0, atol=1e-14)


def test_attention_matches_scipy_softmax_with_grouped_heads_and_padding():
    from scipy.special import softmax
    rng = np.random.default_rng(10)
    H, N, D, n = 8, 2, 16, 11
    q = rng.standard_normal((H, D))
    K = rng.standard_normal((n, N * D))
    V = rng.standard_normal((n, N * D))
    valid = (rng.uniform(size=n) > 0.3).astype(np.int32)
    valid[0] = 1
    o = oracle.attention(q, K, V, N, valid)
    sel = np.nonzero(valid)[0]
    for j in range(H):
        h = j // (H // N)
        s = K[sel, h * D:(h + 1) * D] @ q[j] / math.sqrt(D)
        want = softmax(s) @ V[sel, h * D:(h + 1) * D]
        assert np.allclose(o[j], want, rtol=1e-12, atol=1e-14)
    # padding rows do not matter
    K[valid == 0] += 100.0
    V[valid == 0] -= 50.0
    assert np.array_equal(oracle.attention(q, K, V, N, valid), o)
