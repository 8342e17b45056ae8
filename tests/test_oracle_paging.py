"""Pins of the oracle's sizing, block counting and block-table gather against the
figures and worked examples the pages print (tests/golden/*.json)."""
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_bytes_per_token_match_pages():
    g = _golden("sizing.json")
    for row in g["per_token"]:
        got = oracle.kv_bytes_per_token(row["num_kv_heads"], row["head_dim"],
                                        row["num_layers"], row["elem_bytes"])
        assert got == row["bytes_per_token"], row["model"]
    pl = g["per_layer_token"]
    # one layer, one KV group as wide as the hidden size
    assert oracle.kv_bytes_per_token(1, pl["hidden"], 1, pl["elem_bytes"]) == pl["bytes"]


def test_budget_tokens_and_sequences_match_pages():
    g = _golden("sizing.json")
    b = g["budget"]
    opt = g["per_token"][0]
    per_tok = oracle.kv_bytes_per_token(opt["num_kv_heads"], opt["head_dim"],
                                        opt["num_layers"], opt["elem_bytes"])
    tokens = b["cache_bytes"] // per_tok
    assert tokens == 15728
    assert abs(tokens - b["tokens_printed"]) / b["tokens_printed"] < 0.01
    assert tokens // b["max_len"] == b["sequences_printed"]
    seq = g["sequence"]
    gib = per_tok * seq["tokens"] / 2 ** 30
    assert abs(gib - seq["gb_printed"]) < 0.05
    bt = g["batch"]
    l7 = g["per_token"][3]
    per7 = oracle.kv_bytes_per_token(l7["num_kv_heads"], l7["head_dim"], l7["num_layers"],
                                     l7["elem_bytes"])
    assert per7 * bt["context"] * bt["batch"] == bt["gb_printed"] * 2 ** 30


def test_blocks_for_tokens_worked_example():
    ex = _golden("paging_examples.json")["block_size_4_reply"]
    n, bs = ex["num_tokens"], ex["block_size"]
    blocks = oracle.blocks_for_tokens(n, bs)
    assert blocks == ex["blocks"]
    assert blocks * bs - n == ex["wasted_paged"]
    assert n - (blocks - 1) * bs == ex["last_block_fill"]
    assert ex["contiguous_reservation"] - n == ex["wasted_contiguous"]


def test_blocks_for_tokens_closed_form_and_waste_bound():
    for bs in (1, 2, 4, 8, 16, 32):
        for n in range(0, 200):
            b = oracle.blocks_for_tokens(n, bs)
            assert b == -(-n // bs)                          # ceil(n / bs)
            assert 0 <= b * bs - n < bs                       # waste < one block


def _place(tokens_kv, table, block_size, num_blocks):
    """Write token rows into a pool, one block-table entry per block."""
    n, hkv, d = tokens_kv.shape
    pool = np.zeros((num_blocks, hkv, block_size, d), dtype=tokens_kv.dtype)
    for t in range(n):
        pool[table[t // block_size], :, t % block_size, :] = tokens_kv[t]
    return pool


def test_gather_worked_block_table():
    ex = _golden("paging_examples.json")["block_size_4_reply"]
    bs, n, table = ex["block_size"], ex["num_tokens"], ex["block_table"]
    # token t carries the value t + 1 in every element (fp16 bits of small ints)
    hkv, d = 2, 3
    vals = np.repeat(np.arange(1, n + 1, dtype=np.float16)[:, None, None], hkv, 1)
    vals = np.repeat(vals, d, 2)
    pool = _place(vals.view(np.uint16), table, bs, num_blocks=16)
    for h in range(hkv):
        got = oracle.gather(pool, oracle.F16, table, n, h)
        assert np.array_equal(got[:, 0], np.arange(1, n + 1))
        assert np.array_equal(got, np.repeat(got[:, :1], d, 1))


def test_gather_reads_only_used_blocks():
    # entries past the last used block may hold anything, even ids outside the pool
    pool = np.arange(4 * 1 * 4 * 2, dtype=np.uint16).reshape(4, 1, 4, 2)
    got = oracle.gather(pool, oracle.F16, [2, 0, 999999, -5], 6, 0)
    assert got.shape == (6, 2)
    try:
        oracle.gather(pool, oracle.F16, [2, 0, 999999], 9, 0)
    except IndexError:
        pass
    else:
        raise AssertionError("an out-of-pool entry inside the context must be reported")


def test_gather_any_placement_equals_contiguous_layout():
    rng = np.random.default_rng(3)
    bs, n, hkv, d, nb = 4, 23, 3, 5, 40
    rows = rng.standard_normal((n, hkv, d)).astype(np.float16)
    table = rng.permutation(nb)[: math.ceil(n / bs)]
    pool = _place(rows.view(np.uint16), table, bs, nb)
    for h in range(hkv):
        got = oracle.gather(pool, oracle.F16, table, n, h)
        assert np.array_equal(got, rows[:, h, :].astype(np.float64))
