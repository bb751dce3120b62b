"""The byte ledger behind every GB/s figure, pinned to the numbers the
tutorial page prints for Qwen2.5-7B ("18 e2e inference serving", sections
2.4-2.6) and to a step worked by hand."""

import os

import numpy as np

from paged_gqa_decode_reshape_gb300 import ledger

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_ledger.txt")


def golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_kv_ledger_matches_printed_values():
    g = golden()
    per_tok = ledger.kv_bytes_per_token(g["hkv"], g["head_dim"], g["elem_bytes"])
    assert per_tok == g["bytes_per_token_per_layer"]
    assert per_tok * g["layers"] == g["bytes_per_token_all_layers"]
    assert ledger.kv_bytes_per_block(g["hkv"], g["head_dim"], g["block_size"], g["layers"],
                                     g["elem_bytes"]) == g["bytes_per_block_all_layers"]
    assert ledger.decode_arithmetic_intensity(g["hq"], g["hkv"], g["elem_bytes"]) == g["arithmetic_intensity"]


def test_step_bytes_by_hand():
    # 2 sequences, ctx 17 and 3, Hq 4, Hkv 2, D 8, BS 16, topk 1
    ctx = np.array([17, 3])
    slots = np.array([5 * 16 + 0, -1])        # one written token landing at offset 0
    sel = np.array([[[1], [0]], [[0], [-1]]])
    s = ledger.step_bytes(ctx, slots, Hq=4, Hkv=2, D=8, BS=16, topk=1, selected=sel)
    row = 2 * 8 * 2                            # one token's K (or V) over both KV heads: 32 B
    q = 2 * 4 * 8 * 2                          # 128 B
    assert s.reshape == 2 * 2 * row + 16
    assert s.meta == row + 1 * row * 4 + 16
    assert s.dense == (17 + 3) * 2 * row + 2 * q + (2 + 1) * 4 + 8
    assert s.select == (2 + 1) * 2 * row + q + 3 * 4 + 8 + 2 * 2 * 1 * 4
    # selected tokens: seq 0 head 0 block 1 -> 1 token, head 1 block 0 -> 16, seq 1 head 0 -> 3
    assert s.sparse == (1 + 16 + 3) * 2 * 8 * 2 + 2 * q + 4 * 4 + 3 * 4 + 8
    assert s.total == s.reshape + s.meta + s.dense + s.select + s.sparse
