"""Pins of the oracle's chained block hashes (prefix caching).

* the hash function: SHA-256 as defined by FIPS 180-4, checked against the
  standard's published example digests (one-block "abc", the empty message,
  and the two-block 448-bit message);
* prefix property: two token streams with equal openings get equal hashes for
  every full block inside the common opening and different hashes from the
  first block that differs onward (each hash covers everything before it);
* only full blocks are hashed; a parent hash continues a chain exactly.
"""
import hashlib

import numpy as np

import oracle

FIPS_EXAMPLES = {
    b"abc": "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad",
    b"": "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855",
    b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq":
        "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1",
}


def test_sha256_matches_the_standard_examples():
    for msg, digest in FIPS_EXAMPLES.items():
        assert hashlib.sha256(msg).hexdigest() == digest


def test_equal_openings_share_hashes_until_they_differ():
    rng = np.random.default_rng(1)
    bs = 16
    common = rng.integers(0, 32000, size=5 * bs + 7)
    a = np.concatenate([common, rng.integers(0, 32000, size=40)])
    b = np.concatenate([common, rng.integers(0, 32000, size=70)])
    toks = np.concatenate([a, b]).astype(np.int32)
    cu = [0, len(a), len(a) + len(b)]
    ha, hb = oracle.block_hashes(toks, cu, bs)
    assert len(ha) == len(a) // bs and len(hb) == len(b) // bs
    assert ha[:5] == hb[:5]                      # blocks inside the common opening
    assert all(x != y for x, y in zip(ha[5:], hb[5:]))
    assert len(set(ha + hb)) == len(ha) + len(hb) - 5


def test_partial_blocks_and_parent_chaining():
    rng = np.random.default_rng(2)
    bs = 8
    seq = rng.integers(-5, 2 ** 31 - 1, size=45).astype(np.int32)
    whole = oracle.block_hashes(seq, [0, 45], bs)[0]
    assert len(whole) == 5                        # 45 tokens: 5 full blocks of 8
    # the first 3 blocks, then the rest continued from the third hash
    head = oracle.block_hashes(seq[:24], [0, 24], bs)[0]
    tail = oracle.block_hashes(seq[24:], [0, 21], bs,
                               parent_hashes=[np.frombuffer(head[-1], np.uint8)])[0]
    assert head + tail == whole
    assert oracle.block_hashes(seq[:7], [0, 7], bs) == [[]]
