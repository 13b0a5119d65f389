"""The benchmark's byte arithmetic reproduces the numbers the pages print."""
import os

import pytest

from paged_kv_cache_61_gb300 import traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kv(path):
    out = {}
    with open(os.path.join(GOLDEN, path)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                out[k] = float(v)
    return out


def _table():
    rows = []
    with open(os.path.join(GOLDEN, "kv_cache_arithmetic.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            cols = [c.strip() for c in line.split("|")]
            rows.append(cols)
    return rows


@pytest.mark.parametrize("row", _table(), ids=lambda r: r[0])
def test_kib_per_token_table(row):
    name, layers, qh, kvh, hd, lora, rope, bpe, kib, vs_mha, gb32k, ms_b4, maxbatch = row
    layers, qh, bpe = int(layers), int(qh), int(bpe)
    if kvh != "-":
        per_tok = traffic.gqa_bytes_per_token(layers, int(kvh), int(hd), bpe)
        mha_eq = traffic.gqa_bytes_per_token(layers, qh, int(hd), bpe)
    else:
        per_tok = traffic.mla_bytes_per_token(layers, int(lora), int(rope), bpe)
        mha_eq = traffic.gqa_bytes_per_token(layers, qh, 128, bpe)
    ctx, bw, budget, batch = 32768, 3.35e12, 40 * 2 ** 30, 4
    assert round(per_tok / 1024, 1) == float(kib)
    assert round(mha_eq / per_tok, 1) == float(vs_mha)
    assert round(per_tok * ctx / 1e9, 2) == float(gb32k)
    assert round(per_tok * ctx * batch / bw * 1e3, 2) == float(ms_b4)
    assert int(budget // (per_tok * ctx)) == int(maxbatch)


def test_cache_ratios():
    g = _kv("cache_ratios.txt")
    assert traffic.gqa_bytes_per_token(80, 8, 128, 2) == g["llama2_70b_bytes_per_token"]
    assert traffic.gqa_bytes_per_token(80, 8, 128, 2) / 1024 == g["llama2_70b_kib_per_token"]
    assert traffic.gqa_bytes_per_token(80, 64, 128, 2) / 1024 == g["llama2_70b_mha_kib_per_token"]
    mha_elems = traffic.gqa_bytes_per_token(1, 128, 128, 1)
    mla_elems = traffic.mla_bytes_per_token(1, 512, 64, 1)
    assert round(mha_elems / mla_elems, 2) == g["mha_over_mla_elements"]
    assert mla_elems / (2 * 128) == g["mla_equivalent_gqa_groups"]
    assert round(traffic.gqa_bytes_per_token(1, 8, 128, 1) / mla_elems, 1) == g["gqa405b_over_mla"]
    assert mla_elems / traffic.gqa_bytes_per_token(1, 1, 128, 1) == g["mla_over_mqa"]


def test_drill_decode_bytes():
    g = _kv("drill_decode_bytes.txt")
    ctx = [int(g["ctx"])] * int(g["batch"])
    b = traffic.gqa_kv_bytes(ctx, int(g["kv_heads"]), int(g["head_dim"]), int(g["dtype_bytes"]))
    assert b == g["kv_bytes"]
    # the page's 1520 GB/s is the same byte count over its 176 us, to the two digits it prints
    assert round(b / (g["time_us"] * 1e-6) / 1e9, -1) == pytest.approx(g["gbs"], abs=10)


def test_decode_flops_are_two_per_multiply_add():
    # one token, one head, Dqk = Dv = 1: one multiply-add for the score and one for the value
    assert traffic.decode_flops([1], 1, 1, 1) == 4
    # MLA at the measured workload: 2 * (576 + 512) * Hq * sum(ctx)
    assert traffic.decode_flops([65536] * 16, 16, 576, 512) == 2 * 1088 * 16 * 65536 * 16
    assert traffic.mla_kv_bytes([65536] * 16, 576, 2) == 1207959552
