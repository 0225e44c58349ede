"""Pins for the float64 oracle, independent of the oracle's own code.

Each test checks the oracle against something other than itself: a pure-Python
brute force written separately (its own bf16 decoding, nibble unpacking, page
walk and two-pass softmax with math.fsum), hand-derived closed forms, exact
invariants of softmax attention, and torch's float64 scaled-dot-product
attention on explicitly gathered keys.
"""
import json
import math
import os
import struct

import numpy as np
import pytest
import torch

from oracle import decode_ref, decode_ref_inputs, dequant_int4, merge_splits, unpack_int4
from oracle.decode_ref import bf16_to_f64
from split_kv_paged_gqa_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


# ---------------------------------------------------------------------------
# Independent brute force (pure Python scalars, no numpy arithmetic)


def _bf16_scalar(bits):
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _elem(kind, cache, scales, page, slot, head, d):
    if kind == "bf16":
        return _bf16_scalar(cache[page][slot][head][d])
    if kind == "int8":
        return float(cache[page][slot][head][d]) * float(scales[page][slot][head][0])
    byte = int(cache[page][slot][head][d // 2])
    nib = (byte >> (4 * (d % 2))) & 0xF
    code = nib - 16 if nib > 7 else nib
    return float(code) * float(scales[page][slot][head][d // 32])


def brute_decode(inp):
    q = inp["q"].tolist()
    kc, vc = inp["k_cache"].tolist(), inp["v_cache"].tolist()
    sc = inp["kv_scales"]
    ks = sc[0].tolist() if sc is not None else None
    vs = sc[1].tolist() if sc is not None else None
    pt = inp["page_table"].tolist()
    L_all = [int(x) for x in inp["cache_seqlens"]]
    kind = inp["kv_dtype"]
    B, Tq, Hq, D = inp["q"].shape
    P, Hkv = inp["k_cache"].shape[1], inp["k_cache"].shape[2]
    scale = inp["softmax_scale"] if inp.get("softmax_scale") is not None else 1 / math.sqrt(D)
    out = [[[[0.0] * D for _ in range(Hq)] for _ in range(Tq)] for _ in range(B)]
    lse = [[[-math.inf] * Hq for _ in range(Tq)] for _ in range(B)]
    for b in range(B):
        for t in range(Tq):
            n = L_all[b] - (Tq - 1) + t
            for h in range(Hq):
                hk = (h * Hkv) // Hq
                qv = [_bf16_scalar(x) for x in q[b][t][h]]
                scores, vrows = [], []
                for j in range(max(n, 0)):
                    page, slot = pt[b][j // P], j % P
                    k = [_elem(kind, kc, ks, page, slot, hk, d) for d in range(D)]
                    vrows.append([_elem(kind, vc, vs, page, slot, hk, d) for d in range(D)])
                    scores.append(scale * math.fsum(qv[d] * k[d] for d in range(D)))
                if not scores:
                    continue
                m = max(scores)
                z = math.fsum(math.exp(s - m) for s in scores)
                lse_v = m + math.log(z)
                lse[b][t][h] = lse_v
                w = [math.exp(s - lse_v) for s in scores]
                out[b][t][h] = [math.fsum(w[j] * vrows[j][d] for j in range(len(w)))
                                for d in range(D)]
    return np.array(out), np.array(lse)


def _tiny(kind, seed, B, Tq, Hq, Hkv, D, P, lengths, extra_pages=0, poison=False):
    shape = wl.DecodeShape("tiny", B, Hq, Hkv, D, P, Tq, kind, "fixed:" + ",".join(map(str, lengths)))
    w = wl.make_workload(shape, seed, "cpu", extra_pages=extra_pages, poison=poison)
    return w, wl.oracle_inputs(w)


BRUTE_CASES = [
    # kind, B, Tq, Hq, Hkv, D, P, lengths
    ("bf16", 2, 1, 8, 2, 64, 16, (100 // 4, 40)),
    ("bf16", 3, 1, 4, 4, 8, 1, (1, 7, 13)),
    ("bf16", 2, 4, 6, 2, 8, 4, (4, 9)),
    ("int8", 2, 1, 4, 2, 64, 4, (17, 33)),
    ("int8", 1, 2, 2, 1, 8, 16, (5,)),
    ("int4", 2, 1, 4, 2, 64, 16, (23, 40)),
    ("int4", 2, 4, 4, 1, 32, 4, (6, 11)),
]


@pytest.mark.parametrize("case", BRUTE_CASES, ids=lambda c: f"{c[0]}-B{c[1]}-T{c[2]}-D{c[5]}-P{c[6]}")
def test_oracle_matches_brute_force(case):
    kind, B, Tq, Hq, Hkv, D, P, lengths = case
    w, inp = _tiny(kind, 7 + B + D, B, Tq, Hq, Hkv, D, P, lengths, extra_pages=3, poison=True)
    out, lse = decode_ref_inputs(inp)
    bout, blse = brute_decode(inp)
    assert np.array_equal(np.isinf(lse), np.isinf(blse))
    np.testing.assert_allclose(out, bout, rtol=0, atol=1e-12)
    fin = np.isfinite(blse)
    np.testing.assert_allclose(lse[fin], blse[fin], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms


def _golden_case(c):
    D = len(c["q"])
    L, P = c["seqlen"], c["page_size"]
    table = np.array(c["page_table"], dtype=np.int32)
    n_pages = int(table.max()) + 1
    k = np.zeros((n_pages, P, 1, D), dtype=np.float32)
    v = np.zeros_like(k)
    for j in range(L):
        page, slot = table[0, j // P], j % P
        k[page, slot, 0] = c["k"][j]
        v[page, slot, 0] = c["v"][j]
    to_bits = lambda a: (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q = to_bits(np.array(c["q"], dtype=np.float32).reshape(1, 1, 1, D))
    return decode_ref(q, to_bits(k), to_bits(v), None, table, np.array([L], np.int32), 1, "bf16",
                      softmax_scale=c["scale"])


def test_golden_closed_forms():
    g = json.load(open(GOLDEN))
    env = {"e": math.e, "log": math.log}
    for c in g["cases"]:
        out, lse = _golden_case(c)
        expect_out = [eval(x, {}, env) for x in c["out_expr"]]
        np.testing.assert_allclose(c["out"], expect_out, rtol=0, atol=1e-15)
        assert abs(eval(c["lse_expr"], {}, env) - c["lse"]) < 1e-15
        np.testing.assert_allclose(out[0, 0, 0], c["out"], rtol=0, atol=1e-14, err_msg=c["name"])
        assert abs(lse[0, 0, 0] - c["lse"]) < 1e-14, c["name"]


def test_int4_hand_bytes():
    g = json.load(open(GOLDEN))["int4_bytes"]
    codes = unpack_int4(np.array(g["bytes"], dtype=np.uint8).reshape(-1, 1))
    assert codes.tolist() == g["codes"]


def test_int4_group_scales():
    packed = np.full((1, 32), 0x21, dtype=np.uint8)        # codes 1, 2 alternating, D = 64
    scale = np.array([[0.5, 3.0]], dtype=np.float32)
    x = dequant_int4(packed, scale)
    assert x[0, :32].tolist() == [0.5, 1.0] * 16
    assert x[0, 32:].tolist() == [3.0, 6.0] * 16


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F80, 0x8000], dtype=np.uint16)
    got = bf16_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 1.0 + 2.0 ** -7
    assert got[3] == 2.0 ** -133 and math.isinf(got[4]) and got[5] == 0.0


def _single_request(kind, L, seed=3, D=64, P=16, Tq=1):
    return _tiny(kind, seed, 1, Tq, 4, 2, D, P, (L,))


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_single_key_returns_its_value(kind):
    w, inp = _single_request(kind, 1)
    out, lse = decode_ref_inputs(inp)
    from oracle import gather_kv
    sc = inp["kv_scales"]
    K = gather_kv(inp["k_cache"], None if sc is None else sc[0], inp["page_table"][0], 1, 16, kind)
    V = gather_kv(inp["v_cache"], None if sc is None else sc[1], inp["page_table"][0], 1, 16, kind)
    q = bf16_to_f64(inp["q"])
    for h in range(4):
        np.testing.assert_array_equal(out[0, 0, h], V[0, h // 2])
        s = sum(q[0, 0, h, d] * K[0, h // 2, d] for d in range(64)) / 8.0
        assert abs(lse[0, 0, h] - s) < 1e-12


def test_identical_keys_give_mean_and_log_count():
    w, inp = _single_request("bf16", 37)
    k = inp["k_cache"]
    page0 = inp["page_table"][0, 0]
    for j in range(37):
        pg, sl = inp["page_table"][0, j // 16], j % 16
        k[pg, sl] = k[page0, 0]
    out, lse = decode_ref_inputs(inp)
    from oracle import gather_kv
    V = gather_kv(inp["v_cache"], None, inp["page_table"][0], 37, 16, "bf16")
    K = gather_kv(k, None, inp["page_table"][0], 37, 16, "bf16")
    q = bf16_to_f64(inp["q"])
    for h in range(4):
        np.testing.assert_allclose(out[0, 0, h], V[:, h // 2].mean(axis=0), rtol=0, atol=1e-12)
        s = float(np.dot(q[0, 0, h], K[0, h // 2])) / 8.0
        assert abs(lse[0, 0, h] - (s + math.log(37))) < 1e-12


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_needle_dominates(kind):
    shape = wl.DecodeShape("n", 2, 4, 2, 64, 16, 1, kind, "fixed:300,41")
    w = wl.make_workload(shape, 11, "cpu", needles=True)
    inp = wl.oracle_inputs(w)
    out, _ = decode_ref_inputs(inp)
    from oracle import gather_kv
    sc = inp["kv_scales"]
    for b, h, j in w.needles:
        V = gather_kv(inp["v_cache"], None if sc is None else sc[1], inp["page_table"][b],
                      int(inp["cache_seqlens"][b]), 16, kind)
        np.testing.assert_allclose(out[b, 0, h * 2], V[j, h], rtol=0, atol=2e-6)


# ---------------------------------------------------------------------------
# Invariants


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_merge_of_any_partition_equals_unsplit(kind):
    w, inp = _tiny(kind, 21, 2, 4, 4, 2, 64, 4, (53, 77))
    full_out, full_lse = decode_ref_inputs(inp)
    rng = np.random.default_rng(5)
    for S in (1, 2, 3, 7, 16, 64):
        cuts = np.sort(rng.integers(0, 78, size=S - 1)) if S > 1 else np.array([], dtype=int)
        bounds = [0] + cuts.tolist() + [78]           # repeated cuts give empty pieces
        parts = [decode_ref_inputs(inp, key_range=(lo, hi)) for lo, hi in zip(bounds[:-1], bounds[1:])]
        o, l = merge_splits(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        np.testing.assert_allclose(o, full_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, full_lse, rtol=0, atol=1e-12)


def test_merge_all_empty_is_zero_and_neg_inf():
    o, l = merge_splits(np.zeros((3, 2, 4)), np.full((3, 2), -math.inf))
    assert np.all(o == 0) and np.all(np.isneginf(l))


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_page_permutation_invariance(kind):
    w, inp = _tiny(kind, 31, 2, 1, 4, 2, 64, 4, (30, 19), extra_pages=5)
    out, lse = decode_ref_inputs(inp)
    n_pages = inp["k_cache"].shape[0]
    perm = np.random.default_rng(9).permutation(n_pages)        # new slot of each old page
    inv = np.empty_like(perm)
    inv[perm] = np.arange(n_pages)
    p2 = dict(inp)
    p2["k_cache"] = inp["k_cache"][inv]
    p2["v_cache"] = inp["v_cache"][inv]
    if inp["kv_scales"] is not None:
        p2["kv_scales"] = inp["kv_scales"][:, inv]
    pt = inp["page_table"].copy()
    pt[pt >= 0] = perm[pt[pt >= 0]]
    p2["page_table"] = pt
    out2, lse2 = decode_ref_inputs(p2)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_gqa_equals_replicated_mha(kind):
    G = 3
    w, inp = _tiny(kind, 41, 2, 2, 6, 2, 64, 16, (20, 35))
    out, lse = decode_ref_inputs(inp)
    rep = dict(inp)
    rep["k_cache"] = np.repeat(inp["k_cache"], G, axis=2)        # head h' = old head h' // G
    rep["v_cache"] = np.repeat(inp["v_cache"], G, axis=2)
    if inp["kv_scales"] is not None:
        rep["kv_scales"] = np.repeat(inp["kv_scales"], G, axis=3)
    out2, lse2 = decode_ref_inputs(rep)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_mtp_token_equals_single_token_call(kind):
    Tq = 4
    w, inp = _tiny(kind, 51, 2, Tq, 4, 2, 64, 16, (29, 64))
    out, lse = decode_ref_inputs(inp)
    for t in range(Tq):
        one = dict(inp)
        one["q"] = inp["q"][:, t:t + 1]
        one["q_per_req"] = 1
        one["cache_seqlens"] = inp["cache_seqlens"] - (Tq - 1) + t
        o1, l1 = decode_ref_inputs(one)
        assert np.array_equal(out[:, t], o1[:, 0]) and np.array_equal(lse[:, t], l1[:, 0])


def test_score_shift_leaves_output_and_shifts_lse():
    w, inp = _single_request("bf16", 45)
    k = inp["k_cache"]
    one_bits = np.uint16(0x3F80)
    k[..., 0] = one_bits                                  # every key has k[0] = 1
    inp["q"] = inp["q"].copy()
    inp["q"][..., 0] = np.uint16(0x3F00)                  # q[0] = 0.5
    base_out, base_lse = decode_ref_inputs(inp)
    q = inp["q"].copy()
    q[..., 0] = np.uint16(0x4090)                         # q[0] = 4.5: every score moves by 4/8
    assert bf16_to_f64(np.array([0x4090], np.uint16))[0] == 4.5
    s_inp = dict(inp)
    s_inp["q"] = q
    out, lse = decode_ref_inputs(s_inp)
    np.testing.assert_allclose(out, base_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, base_lse + 4.0 / 8.0, rtol=0, atol=1e-12)


@pytest.mark.parametrize("Tq", [1, 4])
def test_matches_torch_sdpa_float64(Tq):
    w, inp = _tiny("bf16", 61, 2, Tq, 8, 2, 64, 16, (100, 257))
    out, lse = decode_ref_inputs({**inp, "softmax_scale": None})   # default scale vs SDPA's
    from oracle import gather_kv
    q = torch.from_numpy(bf16_to_f64(inp["q"]))
    for b in range(2):
        L = int(inp["cache_seqlens"][b])
        K = torch.from_numpy(gather_kv(inp["k_cache"], None, inp["page_table"][b], L, 16, "bf16"))
        V = torch.from_numpy(gather_kv(inp["v_cache"], None, inp["page_table"][b], L, 16, "bf16"))
        Kh = K.repeat_interleave(4, dim=1).permute(1, 0, 2)        # [Hq, L, D]
        Vh = V.repeat_interleave(4, dim=1).permute(1, 0, 2)
        qh = q[b].permute(1, 0, 2)                                  # [Hq, Tq, D]
        mask = torch.arange(L)[None, :] < (L - (Tq - 1) + torch.arange(Tq))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qh, Kh, Vh, attn_mask=mask)
        np.testing.assert_allclose(out[b], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        scores = (qh @ Kh.transpose(1, 2)) / 8.0
        ref_lse = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)
        np.testing.assert_allclose(lse[b], ref_lse.T.numpy(), rtol=0, atol=1e-12)


def test_rows_without_keys_are_zero_and_neg_inf():
    w, inp = _tiny("bf16", 71, 2, 4, 4, 2, 8, 4, (2, 0))
    out, lse = decode_ref_inputs(inp)
    # request 0: L=2, Tq=4 -> tokens 0,1 see -1 and 0 keys; request 1 sees none
    assert np.all(out[0, :2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(np.isfinite(lse[0, 2:]))
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


@pytest.mark.parametrize("kind", wl.KV_DTYPES)
def test_poisoned_unowned_memory_is_never_read(kind):
    args = (kind, 81, 2, 2, 4, 2, 64, 16, (21, 50))
    _, clean = _tiny(*args, extra_pages=4, poison=False)
    _, dirty = _tiny(*args, extra_pages=4, poison=True)
    o1, l1 = decode_ref_inputs(clean)
    o2, l2 = decode_ref_inputs(dirty)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.all(np.isfinite(o2))
