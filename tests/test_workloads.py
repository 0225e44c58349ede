"""Host-side checks of the seeded workload generator (quantisers, lengths, pages)."""
import math

import numpy as np
import pytest
import torch

from oracle import dequant_int4, dequant_int8, unpack_int4
from split_kv_paged_gqa_gb300 import workloads as wl


def test_int8_round_half_even_and_clamp():
    x = torch.tensor([[127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -127.0]])
    codes, scale = wl.quantize_int8(x)
    assert scale.item() == 1.0
    assert codes.tolist() == [[127, 2, 4, -2, -4, 0, 2, -127]]


def test_int8_zero_row_has_zero_scale():
    codes, scale = wl.quantize_int8(torch.zeros(1, 8))
    assert scale.item() == 0.0 and codes.abs().sum().item() == 0


def test_int4_bytes_from_quantizer():
    x = torch.zeros(1, 32)
    x[0, :4] = torch.tensor([1.0, -1.0, 7.0, 0.0])
    packed, scale = wl.quantize_int4(x)
    assert scale.tolist() == [[1.0]]
    assert packed[0, :2].tolist() == [0xF1, 0x07]
    x[0, :4] = torch.tensor([2.5, 3.5, -2.5, -7.0])
    packed, _ = wl.quantize_int4(x)
    assert unpack_int4(packed.numpy())[0, :4].tolist() == [2, 4, -2, -7]


@pytest.mark.parametrize("kind", ["int8", "int4"])
def test_round_trip_error_within_half_step(kind):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(64, 8, 128, generator=g)
    if kind == "int8":
        codes, scale = wl.quantize_int8(x)
        deq = dequant_int8(codes.numpy(), scale.numpy())
        step = np.repeat(scale.numpy(), 128, axis=-1).astype(np.float64)
        assert codes.min().item() >= -127 and codes.max().item() <= 127
    else:
        packed, scale = wl.quantize_int4(x)
        deq = dequant_int4(packed.numpy(), scale.numpy())
        step = np.repeat(scale.numpy(), 32, axis=-1).astype(np.float64)
        codes = unpack_int4(packed.numpy())
        assert codes.min() >= -7 and codes.max() <= 7
    err = np.abs(x.double().numpy() - deq)
    assert np.all(err <= step / 2 * (1 + 1e-6))


def test_lengths_recipes():
    rng = np.random.default_rng(0)
    u = wl.draw_lengths("uniform:3,5", 2000, rng)
    assert u.min() == 3 and u.max() == 5
    ln = wl.draw_lengths("lognormal:4096,1.0,16,32768", 4000, rng)
    assert ln.min() >= 16 and ln.max() <= 32768
    assert abs(np.median(ln) - 4096) / 4096 < 0.1
    assert wl.draw_lengths("const:7", 3, rng).tolist() == [7, 7, 7]


def test_page_assignment_is_a_permutation_slice():
    rng = np.random.default_rng(1)
    L = np.array([100, 257])
    table, pool = wl.assign_pages(L, 16, 64, 0, rng)
    assert pool == 64 and table.shape == (2, 17)
    assert (table[0, 7:] == -1).all() and (table[0, :7] >= 0).all() and (table[1] >= 0).all()
    used = np.concatenate([table[0, :7], table[1]])
    assert len(set(used.tolist())) == 24 and used.max() < 64


def test_tiny_config_shapes():
    w = wl.make_workload(wl.CONFIGS["tiny_bf16"], wl.CONFIG_SEEDS["tiny_bf16"])
    assert tuple(w.q.shape) == (2, 1, 8, 64) and w.q.dtype == torch.bfloat16
    assert tuple(w.k_cache.shape) == (64, 16, 2, 64)
    assert w.cache_seqlens.tolist() == [100, 257]
    assert w.kv_bytes() == 357 * 2 * 2 * 64 * 2


def test_workload_is_deterministic():
    s = wl.CONFIGS["tiny_bf16"]
    a = wl.make_workload(s, 5)
    b = wl.make_workload(s, 5)
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.page_table, b.page_table)


def test_kv_bytes_per_token():
    assert wl.kv_bytes_per_token(wl.CONFIGS["long_bf16_b1"]) == 8 * 2 * 256
    assert wl.kv_bytes_per_token(wl.CONFIGS["int8_lognormal"]) == 8 * 2 * (128 + 4)
    assert wl.kv_bytes_per_token(wl.CONFIGS["int4_mtp"]) == 8 * 2 * (64 + 16)


def test_oracle_inputs_subset_relabels_pages():
    s = wl.DecodeShape("t", 3, 4, 2, 64, 4, 1, "int8", "fixed:9,5,13")
    w = wl.make_workload(s, 2, extra_pages=2)
    sub = wl.oracle_inputs(w, requests=[2, 0])
    assert sub["cache_seqlens"].tolist() == [13, 9]
    assert sub["page_table"][0, :4].tolist() == [0, 1, 2, 3]
    assert sub["page_table"][1, :3].tolist() == [4, 5, 6]
    full = wl.oracle_inputs(w)
    p = int(full["page_table"][2, 1])
    assert np.array_equal(sub["k_cache"][1], full["k_cache"][p])
    assert np.array_equal(sub["kv_scales"][:, 1], full["kv_scales"][:, p])
