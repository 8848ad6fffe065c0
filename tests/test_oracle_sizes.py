"""Pins of oracle/sizes.py against the numbers the pages print (tests/golden/sizes.json)."""
import json
import os

import pytest

from oracle import sizes

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sizes.json")))


def test_bytes_per_token_7b():
    g = GOLD["kv_bytes_per_token_7b"]
    i = g["inputs"]
    assert sizes.kv_bytes_per_token(i["layers"], i["hidden"], i["dtype_bytes"]) == g["value"]
    # the same figure from heads x head_dim per layer
    assert 32 * sizes.kv_bytes_per_token_layer(32, 128, 2) == g["value"]


def test_bytes_per_token_13b():
    g = GOLD["kv_bytes_per_token_13b_kib"]
    i = g["inputs"]
    assert sizes.kv_bytes_per_token(i["layers"], i["hidden"], i["dtype_bytes"]) == g["value"] * 1024


def test_request_sizes():
    per_tok = sizes.kv_bytes_per_token(32, 4096, 2)
    assert sizes.request_bytes(4096, per_tok) == sizes.gib(GOLD["request_4096_tokens_7b_gib"]["value"])
    assert sizes.request_bytes(2048, per_tok) == sizes.gib(GOLD["request_2048_tokens_7b_gib"]["value"])


def test_layer_and_page_bytes():
    per_layer = sizes.kv_bytes_per_token_layer(32, 128, 2)
    assert per_layer == GOLD["kv_bytes_per_token_layer_7b"]["value"]
    assert sizes.block_bytes(256, per_layer) == GOLD["page_bytes_256_tokens"]["value"]
    per_tok = sizes.kv_bytes_per_token(32, 4096, 2)
    assert sizes.block_bytes(16, per_tok) == sizes.mib(GOLD["block_bytes_16_tokens_all_layers_mib"]["value"])


def test_pool_arithmetic_80gb_card():
    g = GOLD["pool_80gb_card"]
    per_tok = sizes.kv_bytes_per_token(32, 4096, 2)
    n = sizes.pool_blocks(sizes.gib(g["usable_gib"]), g["block_tokens"], per_tok)
    assert n == g["blocks"]
    assert sizes.pool_tokens(n, g["block_tokens"]) == g["tokens"]
    assert sizes.max_concurrency(n, g["block_tokens"], g["mean_request_tokens"]) == g["concurrency"]


def test_table_entries():
    g = GOLD["table_entries_per_2048_tokens"]
    for b, e in zip(g["block_sizes"], g["entries"]):
        assert sizes.table_entries(2048, b) == e


def test_wasted_slots_small_cases():
    # brute force: count unused slots of the last block by enumeration
    for b in (1, 2, 4, 8, 16, 32):
        for t in range(0, 3 * b + 1):
            used_blocks = 0
            while used_blocks * b < t:
                used_blocks += 1
            assert sizes.wasted_slots(t, b) == used_blocks * b - t
    assert sizes.wasted_slots(17, 16) == 15
    assert sizes.wasted_slots(64, 16) == 0
    assert sizes.internal_waste_fraction([16, 32, 48], 16) == 0.0


def test_waste_closed_form_uniform_residue():
    # lengths k*B .. k*B + B-1 cover every residue once: mean waste (B-1)/2 exactly
    for b in (8, 16, 32, 64):
        lens = list(range(10 * b, 11 * b))
        wasted = sum(sizes.wasted_slots(t, b) for t in lens)
        assert wasted == b * (b - 1) // 2
        assert sizes.expected_waste_uniform_residue(b) == pytest.approx((b - 1) / 2)


def test_waste_table_mean_300():
    # The page prints approximate values ("about"); lengths uniform on 1..599 have
    # mean 300 and every residue equally often, the plainest reading of its case.
    g = GOLD["internal_waste_mean_300"]
    lens = list(range(1, 600))
    assert sum(lens) / len(lens) == g["mean_tokens"]
    for b, pct in zip(g["block_sizes"], g["percent"]):
        got = 100.0 * sizes.internal_waste_fraction(lens, b)
        assert abs(got - pct) <= 0.15 * pct, (b, got, pct)
    # and waste grows with the block size, about half a block per request
    fr = [sizes.internal_waste_fraction(lens, b) for b in g["block_sizes"]]
    assert fr == sorted(fr)
