"""Pins the roofline accounting to the numbers the pages print (no GPU)."""
import json
import os

import numpy as np

from decode_attention_mfa_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "step3_decode_accounting.json")


def _sig(x, digits):
    return float(f"{x:.{digits - 1}e}")


def test_step3_table2_table3_rows():
    g = json.load(open(GOLDEN))
    layers = g["layers"]
    assert acc.kv_bytes_per_token("fp8", include_scales=False) == g["kv_bytes_per_token_per_layer_8bit"]
    for row in g["rows"]:
        kv = row["context"] * layers * acc.kv_bytes_per_token("fp8", include_scales=False)
        fl = row["context"] * layers * acc.attention_flops_per_token()
        assert _sig(kv, g["printed_significant_digits"]) == row["kv_bytes"]
        assert _sig(fl, g["printed_significant_digits"]) == row["attention_flops"]


def test_arithmetic_intensity():
    g = json.load(open(GOLDEN))
    ai8 = acc.attention_flops_per_token() / acc.kv_bytes_per_token("fp8", include_scales=False)
    assert ai8 == g["arithmetic_intensity_8bit"]
    assert acc.attention_flops_per_token() / acc.kv_bytes_per_token("bf16") == 64


def test_step_bytes_counts_each_stream_once():
    b = acc.decode_step_bytes([4096] * 32, "bf16")
    kv = 32 * 4096 * 1024
    assert b == kv + 32 * 64 * 256 * 2 * 2 + 32 * 64 * 4 + 32 * 64 * 4 + 32 * 4
    assert acc.decode_step_flops([4096] * 32) == 32 * 4096 * 65536


def test_block_gather_bytes():
    # 512 selected blocks + a last block of 8 tokens (L = 32768): 4104 tokens attended
    assert list(acc.blocks_attended([32768, 32769, 0, 1], [512, 3, 0, 0])) == [4104, 25, 0, 1]
    b = acc.decode_blocks_step_bytes([32768] * 32, [512] * 32)
    kv = 32 * 4104 * 1024
    assert b == kv + 32 * 64 * 256 * 2 * 2 + 32 * 64 * 4 + 32 * (513 + 512) * 4 + 32 * 8
    # every block selected: the same K/V rows as dense decode
    L = np.array([1, 8, 9, 700])
    assert list(acc.blocks_attended(L, (L - 1) // 8)) == list(L)
