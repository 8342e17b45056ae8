"""Block swap between the device cache and pinned host memory against the
oracle, byte for byte (「KV 缓存与分页注意力」 §09: a pre-empted sequence's blocks
go to CPU memory and come back)."""
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


def _pool(rng, layers, nb, shape, dtype, device, pinned=False):
    out = []
    for _ in range(layers):
        a = rng.integers(0, 256, size=(nb,) + shape, dtype=np.uint8)
        t = torch.from_numpy(a)
        if dtype != torch.uint8:
            t = t.view(torch.int16).view(dtype) if a.shape[-1] % 2 == 0 else t
        if device == "cpu":
            t = t.pin_memory() if pinned else t
        else:
            t = t.to(device)
        out.append(t)
    return out


@pytest.mark.parametrize("dtype,shape", [(torch.float16, (8, 16, 64 * 2)),
                                         (torch.uint8, (4, 32, 128)),
                                         (torch.bfloat16, (2, 8, 128 * 2))])
def test_swap_out_and_back_in(dtype, shape):
    rng = np.random.default_rng(7)
    layers, nd, nh = 3, 40, 12
    # byte pools; the element view only changes the descriptor's dtype
    shp = shape[:-1] + (shape[-1] // (1 if dtype == torch.uint8 else 2),)
    dk = _pool(rng, layers, nd, shape, torch.uint8, "cuda")
    dv = _pool(rng, layers, nd, shape, torch.uint8, "cuda")
    hk = [torch.full((nh,) + shape, 0xA5, dtype=torch.uint8).pin_memory() for _ in range(layers)]
    hv = [torch.full((nh,) + shape, 0xA5, dtype=torch.uint8).pin_memory() for _ in range(layers)]
    view = (lambda t: t.view(dtype).view((t.shape[0],) + shp)) if dtype != torch.uint8 else \
        (lambda t: t)
    ddesc = [B.cache_desc(view(a), view(b)) for a, b in zip(dk, dv)]
    hdesc = [B.cache_desc(view(a), view(b)) for a, b in zip(hk, hv)]
    ok = [a.cpu().numpy() for a in dk], [a.cpu().numpy() for a in dv]
    ohk = [a.numpy().copy() for a in hk]
    ohv = [a.numpy().copy() for a in hv]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_pairs = np.array([[3, 0], [39, 7], [17, 11], [0, 2]], np.int64)
    B.pkv_swap_blocks(ddesc, hdesc, torch.from_numpy(out_pairs).cuda(), dev_err=err)
    torch.cuda.synchronize()
    oracle.swap_blocks(ok[0], ok[1], ohk, ohv, out_pairs)
    for l in range(layers):
        assert np.array_equal(hk[l].numpy(), ohk[l]) and np.array_equal(hv[l].numpy(), ohv[l])
    # back into other device blocks, pairs read from pinned host memory
    in_pairs = np.array([[0, 5], [7, 6], [11, 30], [2, 31]], np.int64)
    B.pkv_swap_blocks(hdesc, ddesc, torch.from_numpy(in_pairs).pin_memory(), dev_err=err)
    torch.cuda.synchronize()
    oracle.swap_blocks(ohk, ohv, ok[0], ok[1], in_pairs)
    for l in range(layers):
        assert np.array_equal(dk[l].cpu().numpy(), ok[0][l])
        assert np.array_equal(dv[l].cpu().numpy(), ok[1][l])
    assert int(err.item()) == 0


def test_swap_between_device_pools_and_bad_pairs():
    rng = np.random.default_rng(8)
    shape = (2, 16, 128)
    a = torch.from_numpy(rng.integers(0, 256, size=(10,) + shape, dtype=np.uint8)).cuda()
    b = torch.zeros((6,) + shape, dtype=torch.uint8, device="cuda")
    # the descriptors hold raw pointers: every cache they name stays alive
    # (a local) until the swap has finished
    av = a.view(torch.float16).clone()
    bv = b.view(torch.float16).clone()
    sa = B.cache_desc(a.view(torch.float16), av)
    sb = B.cache_desc(b.view(torch.float16), bv)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pairs = torch.tensor([[9, 5], [10, 0], [2, 6], [4, -1], [1, 1]], dtype=torch.int64,
                         device="cuda")
    B.pkv_swap_blocks(sa, sb, pairs, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == B.PKV_DEVERR_COPY_PAIR
    got = b.cpu().numpy()
    want = np.zeros_like(got)
    src = a.cpu().numpy()
    want[5] = src[9]
    want[1] = src[1]
    assert np.array_equal(got, want)


def test_stream_copy_moves_bytes_both_ways():
    """The SM streaming copy the swap bench measures the link with: device to
    pinned host and back, byte for byte, a size that is not a multiple of the
    grid's round; a misaligned pointer or size is refused."""
    rng = np.random.default_rng(11)
    n = (3 << 20) + 48
    src = torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8)).cuda()
    host = torch.zeros(n, dtype=torch.uint8).pin_memory()
    back = torch.zeros(n, dtype=torch.uint8, device="cuda")
    B.pkv_testing_stream_copy(host, src)
    torch.cuda.synchronize()
    assert torch.equal(host, src.cpu())
    B.pkv_testing_stream_copy(back, host)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    lib = B.load()
    st = lib.pkv_testing_stream_copy(B._ptr(back[1:]), B._ptr(src[1:]), 16, None)
    assert st == B.PKV_ERR_INVALID_ARG
    st = lib.pkv_testing_stream_copy(B._ptr(back), B._ptr(src), 24, None)
    assert st == B.PKV_ERR_INVALID_ARG
