"""Cache and parameter accounting pinned to the figures the LRKV pages print
(reading notes §2.5-2.6 and §4.4; technical review §4).  Also checks the
cache ratio of every synthetic workload and the `numel * element_size`
measurement of the allocated tensors (reading notes §4.7)."""
import math

import pytest
import torch

from conftest import read_golden
from oracle import lrkv_oracle as O
from compressed_cache_decode_gb300 import inputs


def test_table7_remaining_fractions():
    _, rows = read_golden("notes_s2_5_cache_fractions.txt")
    for row in rows:
        if row[0] == "elems":
            H, dh, r, mha, lrkv = map(int, row[1:])
            assert O.mha_elems_per_token(H, dh) == mha
            assert O.cache_elems_per_token(H, dh, r) == lrkv
            continue
        H, dh, r = map(int, row[:3])
        assert round(100 * O.cache_fraction(H, dh, r), 2) == float(row[3])
        assert O.cache_elems_per_token(H, dh, r) / O.mha_elems_per_token(H, dh) == \
            pytest.approx(O.cache_fraction(H, dh, r), rel=1e-15)


def test_rank_sweep_fractions():
    _, rows = read_golden("notes_s4_4_rank_sweep.txt")
    for H, dh, r, pct in rows:
        assert round(100 * O.cache_fraction(int(H), int(dh), int(r)), 1) == float(pct)
    # rank 128 at H=6 spends more than MHA; the saving condition says so
    assert not O.saves_cache(6, 128, 128) and O.saves_cache(6, 128, 64)


def test_review_s4_worked_numbers():
    _, rows = read_golden("review_s4_accounting.txt")
    MiB = 1 << 20
    for row in rows:
        tag = row[0]
        if tag == "ceiling":
            H, dh, c, want = int(row[1]), int(row[2]), float(row[3]), int(row[4])
            assert O.rank_ceiling(dh, H, c) == want
            assert O.cache_fraction(H, dh, want) <= c < O.cache_fraction(H, dh, want + 1)
        elif tag == "padded":
            H, dh, r, pct = int(row[1]), int(row[2]), int(row[3]), float(row[4])
            assert round(100 * O.cache_fraction(H, dh, r), 2) == pct
        elif tag == "ceiling_third":
            H, dh, want = int(row[1]), int(row[2]), int(row[3])
            assert O.rank_ceiling(dh, H, 1.0 / 3.0) == want
        elif tag == "bytes":
            length = int(row[1])
            if row[2] != "-":
                assert O.mha_cache_bytes(2, 18, 1, length, 18, 128) == int(row[2])
            assert O.mha_cache_bytes(2, 18, 1, length, 18, 128) / MiB == float(row[3])
            assert O.cache_bytes(2, 18, 1, length, 18, 128, 55) / MiB == float(row[4])
        elif tag == "tp":
            H, dh, r, P, single, repl = int(row[1]), int(row[2]), int(row[3]), int(row[4]), \
                float(row[5]), float(row[6])
            assert round(100 * O.cache_fraction(H, dh, r), 1) == single
            assert round(100 * O.tp_replicated_fraction(P, H, dh, r), 1) == repl
            assert O.tp_replicated_fraction(1, H, dh, r) == O.cache_fraction(H, dh, r)
        elif tag == "params":
            d, H, dh, r, pct = int(row[1]), int(row[2]), int(row[3]), int(row[4]), float(row[5])
            assert round(100 * O.kv_param_fraction(d, H, dh, r), 1) == pct
            # closed form of the ratio printed beside Eq. (10)
            assert O.kv_param_fraction(d, H, dh, r) == pytest.approx(1 / H + r / dh * (1 + dh / d))
        elif tag == "flops":
            dh, r, want = int(row[1]), int(row[2]), float(row[3])
            assert round(O.decode_flop_ratio(dh, r, 10 ** 12), 2) == want
        else:
            raise AssertionError(tag)


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_cache_ratio_and_numel(name):
    """The factored cache of each workload holds 2(d_h + H r) elements per
    token; measured as numel * element_size of small copies of the tensors
    (the measurement method of reading notes §4.7)."""
    w = inputs.WORKLOADS[name]
    want = {"decode_f32_b1_h4_d16_r4_L64": 0.5, "decode_bf16_b8_h16_d64_r28_L4096": 0.5,
            "decode_bf16_b32_h32_d128_r56_ragged1k-8k": 0.46875,
            "decode_bf16_b4_h32_d128_r48_L65536_outliers": 0.40625,
            "prefill_bf16_b2_t4096_h32_d128_r64_dmodel4096": 0.53125}[name]
    assert O.cache_fraction(w.heads, w.head_dim, w.rank) == want
    t = inputs.random_decode_case(0, 1, w.heads, w.head_dim, w.rank, 8, w.dtype)
    cache_bytes = sum(t[k].numel() * t[k].element_size() for k in ("k_s", "v_s", "z_k", "z_v"))
    assert cache_bytes == 8 * O.cache_elems_per_token(w.heads, w.head_dim, w.rank) * w.elem_bytes
