"""The oracle's cost model against the numbers the pages print (CPU only),
and the product's own counter (used by the benchmark) against the oracle's."""

import json
import math
import os

import pytest

import oracle
from exact_io_aware_attn_gb300 import cost as prod_cost

MiB = 1 << 20
GiB = 1 << 30
with open(os.path.join(os.path.dirname(__file__), "golden", "page_numbers.json")) as f:
    PAGE = json.load(f)


def test_e8_1_sizes():
    g = PAGE["sizes_e8_1"]
    assert oracle.score_bytes(4096) == g["score_bytes_4096_MiB"] * MiB
    assert oracle.tile_bytes(128) == g["tile_bytes_128"]
    assert oracle.num_blocks(4096, 128) == g["num_blocks_4096_128"]
    # num_blocks is a ceiling; block < 1 is an error
    assert oracle.num_blocks(4097, 128) == 33
    assert oracle.num_blocks(1, 128) == 1
    with pytest.raises(ValueError):
        oracle.num_blocks(10, 0)


def test_io_aware_sizes():
    g = PAGE["sizes_io_aware"]
    assert oracle.score_bytes(4096) * 16 == g["score_bytes_4096_x16_MiB"] * MiB
    assert oracle.tile_bytes(1, 128 * 64 * 4) == g["accumulator_bytes_128x64_f32"]
    assert oracle.num_blocks(4096, 128) == g["query_blocks_4096_128"]


def _parse_size(s):
    num, unit = s.split()
    return float(num) * {"MiB": MiB, "GiB": GiB}[unit]


def test_score_tensor_table():
    g = PAGE["score_tensor_table"]
    for t, printed in g["rows"]:
        size = g["heads"] * oracle.score_bytes(t)
        want = _parse_size(printed)
        decimals = len(printed.split()[0].split(".")[1]) if "." in printed else 0
        unit = MiB if printed.endswith("MiB") else GiB
        assert round(size / unit, decimals) == round(want / unit, decimals), (t, printed)


def test_peak_memory_multiples_use_one_score_tensor():
    g = PAGE["peak_memory_multiples"]
    for t, naive, naive_x, math_mib, math_x in g["rows"]:
        one = 12 * oracle.score_bytes(t) / MiB
        digits = len(str(naive_x).split(".")[1])
        assert round(naive / one, digits) == naive_x, (t, naive / one)
        assert round(math_mib / one, 1) == math_x, (t, math_mib / one)
    # the efficient backend's peak at 16,384 is the output tensor
    out_bytes = 12 * 16384 * g["head_dim"] * 2
    assert out_bytes == g["efficient_peak_16384_MiB"] * MiB


def test_causal_pairs_and_flops_closed_form():
    for t in (1, 2, 3, 128, 1000, 16384):
        assert oracle.causal_pairs(t) == t * (t + 1) // 2
        assert oracle.attention_pairs(t, t, True) == oracle.causal_pairs(t)
        assert oracle.attention_pairs(t, t, False) == t * t
    # one query against a cache sees every key, causal or not
    assert oracle.attention_pairs(1, 777, True) == 777
    assert oracle.attention_flops(2, 3, 5, 7, 8, False) == 4 * 2 * 3 * 5 * 7 * 8


def test_doubling_properties():
    # doubling the prompt quadruples prefill FLOPs and doubles decode FLOPs
    for t in (256, 1024, 4096):
        assert oracle.attention_flops(1, 12, 2 * t, 2 * t, 64) == 4 * oracle.attention_flops(1, 12, t, t, 64)
        assert oracle.attention_flops(1, 12, 1, 2 * t, 64) == 2 * oracle.attention_flops(1, 12, 1, t, 64)


def test_throughput_numbers_count_the_causal_half():
    g = PAGE["throughput"]
    for t, ms, ms_dec, tflops, tf_dec in g["rows"]:
        # the interval of rates the printed (rounded) time allows must meet
        # the interval the printed (rounded) rate allows
        half_t, half_r = 0.5 * 10.0 ** -ms_dec, 0.5 * 10.0 ** -tf_dec
        lo_r, hi_r = tflops - half_r, tflops + half_r

        def overlaps(f):
            lo = f / ((ms + half_t) * 1e-3) / 1e12
            hi = f / ((ms - half_t) * 1e-3) / 1e12
            return lo <= hi_r and hi >= lo_r

        causal = oracle.attention_flops(1, g["heads"], t, t, g["head_dim"], causal=True)
        dense = oracle.attention_flops(1, g["heads"], t, t, g["head_dim"], causal=False)
        assert overlaps(causal), (t, causal / (ms * 1e-3))
        assert not overlaps(dense)


def test_naive_traffic_estimate():
    g = PAGE["naive_traffic"]
    elems = g["heads"] * oracle.score_bytes(g["T"], 1)
    assert round(elems / 1e6) == g["elements_millions"]
    assert round(elems * 12 / 1e9, 1) == g["gigabytes"]
    assert round(elems * 12 / 278e9 * 1e3) == g["ms_at_278_GBps"]


def test_decode_flops():
    g = PAGE["decode_flops"]
    f = oracle.attention_flops(1, g["heads"], 1, g["T"], g["head_dim"])
    assert round(f / 1e6) == g["approx_millions"]


def test_kv_cache_numbers():
    g = PAGE["kv_cache"]
    for t, mib in g["per_sequence"]:
        assert oracle.kv_bytes(g["layers"], g["heads"], t, g["head_dim"]) == mib * MiB
    for b, t, mib in g["per_step_MiB"]:
        assert oracle.kv_bytes(g["layers"], g["heads"], t, g["head_dim"], batch=b) == mib * MiB
    for b, t, gib in g["per_step_GiB"]:
        size = oracle.kv_bytes(g["layers"], g["heads"], t, g["head_dim"], batch=b) / GiB
        assert math.floor(size * 10 + 0.5) / 10 == gib   # printed rounded half up


def test_decode_table_bandwidth():
    g = PAGE["decode_table"]
    for b, t, seconds, mib, gbps in g["rows"]:
        read = oracle.kv_bytes(1, g["heads"], t, g["head_dim"], batch=b)
        digits = 1 if mib < 1 else 0
        assert round(read / MiB, digits) == mib, (b, t)
        assert abs(read / seconds / 1e9 - gbps) <= 1.0, (b, t, read / seconds / 1e9)


@pytest.mark.parametrize("shape", [
    (1, 2, 256, 256, 64, False), (8, 12, 1024, 1024, 64, True), (1, 16, 8192, 8192, 128, True),
    (1, 12, 16384, 16384, 64, True), (32, 12, 1, 16384, 64, False), (2, 3, 100, 700, 64, True),
    (1, 1, 1, 1, 64, True)])
def test_product_counter_matches_oracle(shape):
    B, h, tq, tk, d, causal = shape
    assert prod_cost.flops(B, h, tq, tk, d, causal) == oracle.attention_flops(B, h, tq, tk, d, causal)
    assert prod_cost.kv_cache_bytes(B, h, tk, d) == oracle.kv_bytes(1, h, tk, d, batch=B)
