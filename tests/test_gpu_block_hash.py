"""Chained SHA-256 block hashes on the GPU against the oracle (hashlib),
byte for byte (「KV 缓存与分页注意力」 §11: a full block's hash covers its
tokens and everything before it)."""
import numpy as np
import pytest
import torch

import harness as H
import oracle
from paged_kv_cache_130_gb300 import binding as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    H.build_library()


def _batch(rng, lens):
    toks = rng.integers(-2 ** 31, 2 ** 31 - 1, size=int(sum(lens)), dtype=np.int64)
    return toks.astype(np.int32), np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_hashes_match_the_oracle(bs):
    rng = np.random.default_rng(bs)
    lens = [0, 5, bs, bs + 1, 7 * bs, 300, 1, 2 * bs - 1] + list(rng.integers(0, 700, 200))
    toks, cu = _batch(rng, lens)
    got = B.pkv_block_hashes(torch.from_numpy(toks).cuda(), torch.from_numpy(cu).cuda(), bs)
    torch.cuda.synchronize()
    want = [h for seq in oracle.block_hashes(toks, cu, bs) for h in seq]
    assert got.shape[0] == len(want)
    assert np.array_equal(got.cpu().numpy(), np.frombuffer(b"".join(want), np.uint8)
                          .reshape(-1, 32))


def test_parent_hashes_and_offsets():
    rng = np.random.default_rng(5)
    bs = 16
    lens = [40, 100, 16]
    toks, cu = _batch(rng, lens)
    parents = rng.integers(0, 256, size=(3, 32), dtype=np.uint8)
    offs = np.array([10, 0, 20], np.int64)          # out of order, with gaps
    hashes = torch.full((24, 32), 7, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.pkv_block_hashes(torch.from_numpy(toks).cuda(), torch.from_numpy(cu).cuda(), bs,
                       block_offsets=torch.from_numpy(offs).cuda(),
                       parent_hashes=torch.from_numpy(parents).cuda(), hashes=hashes,
                       dev_err=err)
    torch.cuda.synchronize()
    got = hashes.cpu().numpy()
    want = oracle.block_hashes(toks, cu, bs, parent_hashes=parents)
    for s, off in enumerate(offs):
        for k, h in enumerate(want[s]):
            assert bytes(got[off + k]) == h
    written = {int(off) + k for s, off in enumerate(offs) for k in range(len(want[s]))}
    for r in range(24):
        if r not in written:
            assert np.all(got[r] == 7)
    assert int(err.item()) == 0


def test_overflowing_offsets_are_flagged():
    rng = np.random.default_rng(6)
    toks, cu = _batch(rng, [64, 64])
    hashes = torch.zeros((5, 32), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    offs = torch.tensor([0, 3], dtype=torch.int64, device="cuda")   # 3 + 4 > 5
    B.pkv_block_hashes(torch.from_numpy(toks).cuda(), torch.from_numpy(cu).cuda(), 16,
                       block_offsets=offs, hashes=hashes, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & B.PKV_DEVERR_CONTEXT
    want = oracle.block_hashes(toks, cu, 16)[0]
    got = hashes.cpu().numpy()
    assert [bytes(got[k]) for k in range(4)] == want
    assert np.all(got[4] == 0)
