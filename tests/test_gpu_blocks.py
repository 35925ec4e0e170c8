"""GPU parity of the copy-on-write block copy (pkv_copy_blocks) and of a decode
step driven by the host allocator, against the CPU oracle.

The copy must match bit for bit; the decode that follows must stay within the
decode tolerance (max-abs 2e-2, mean-abs 2e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_62_gb300 import pkv
from paged_kv_cache_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def caches(NB, bs, Hkv, D, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    kc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    vc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    return kc, vc


def disjoint_pairs(rng, NB, n):
    ids = rng.permutation(NB)[: 2 * n]
    return np.stack([ids[:n], ids[n:]], axis=1).astype(np.int32)


@pytest.mark.parametrize("NB,bs,Hkv,D,n", [(64, 16, 8, 128, 20), (24, 256, 8, 128, 9), (40, 8, 2, 64, 13),
                                           (10, 32, 1, 64, 1), (300, 16, 8, 128, 140)])
def test_copy_blocks_bit_exact(NB, bs, Hkv, D, n):
    rng = np.random.default_rng(NB + n)
    kc, vc = caches(NB, bs, Hkv, D, seed=n)
    pairs = disjoint_pairs(rng, NB, n)
    if n > 1:
        pairs[0, 1] = pairs[0, 0]  # src == dst: unchanged
    kh, vh = W.bits(kc), W.bits(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() == 0
    oracle.copy_blocks(kh, vh, pairs)
    assert np.array_equal(W.bits(kc), kh) and np.array_equal(W.bits(vc), vh)


def test_copy_blocks_bad_ids_and_empty_call():
    NB, bs, Hkv, D = 16, 16, 2, 64
    kc, vc = caches(NB, bs, Hkv, D, seed=3)
    kh, vh = W.bits(kc), W.bits(vc)
    pairs = np.array([[1, 2], [3, NB], [-1, 4], [5, 6]], np.int32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(kc, vc, torch.from_numpy(pairs).cuda(), err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_BLOCK_RANGE
    oracle.copy_blocks(kh, vh, pairs[[0, 3]])  # the valid pairs only
    assert np.array_equal(W.bits(kc), kh) and np.array_equal(W.bits(vc), vh)
    pkv.copy_blocks(kc, vc, torch.zeros(0, 2, dtype=torch.int32, device="cuda"))  # nothing to do
    torch.cuda.synchronize()
    assert np.array_equal(W.bits(kc), kh)


def test_fork_copy_on_write_store_decode():
    """Parallel sampling through the library end to end: the allocator forks a sequence, the child's
    first token triggers copy-on-write of the shared half-full block, pkv_copy_blocks makes the copy,
    pkv_kv_store writes both sequences' new tokens, and pkv_paged_decode attends -- all against the
    oracle run on the same operations."""
    NB, bs, Hkv, D, Hq = 32, 16, 2, 64, 8
    kc, vc = caches(NB, bs, Hkv, D, seed=21)
    a = pkv.BlockAllocator(NB, bs)
    a.add(0, 40)
    a.fork(0, 1)
    cow0 = a.append(0)          # parent writes first: copy-on-write for the parent
    cow1 = a.append(1)          # the child now owns the original alone: no copy
    assert cow0 != (-1, -1) and cow1 == (-1, -1)
    bt_h, lens_h = a.tables([0, 1], 4)
    bt, lens = bt_h.cuda(), lens_h.cuda()
    g = torch.Generator(device="cuda").manual_seed(5)
    k_new = torch.randn(2, Hkv, D, generator=g, device="cuda").bfloat16()
    v_new = torch.randn(2, Hkv, D, generator=g, device="cuda").bfloat16()
    q = torch.randn(2, Hq, D, generator=g, device="cuda").bfloat16()
    kh, vh = W.bits(kc), W.bits(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    pkv.copy_blocks(kc, vc, torch.tensor([cow0], dtype=torch.int32, device="cuda"), err)
    slots = torch.empty(2, dtype=torch.int32, device="cuda")
    pkv.decode_slot_mapping(bt, lens, bs, NB, slots, err)
    pkv.kv_store(k_new, v_new, slots, kc, vc, err)
    out = torch.empty_like(q)
    ws = pkv.alloc_workspace(2, Hq, Hkv, D)
    pkv.paged_decode(q, kc, vc, bt, lens, 0.125, out, ws, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0

    oracle.copy_blocks(kh, vh, np.array([cow0], np.int32))
    s_h = oracle.decode_slot_mapping(bt_h.numpy(), lens_h.numpy(), bs)
    assert np.array_equal(slots.cpu().numpy(), s_h)
    oracle.kv_store(W.bits(k_new), W.bits(v_new), s_h, kh, vh)
    assert np.array_equal(W.bits(kc), kh) and np.array_equal(W.bits(vc), vh)
    want = oracle.paged_decode(W.bits(q), kh, vh, bt_h.numpy(), lens_h.numpy(), 0.125)
    d = np.abs(out.float().cpu().double().numpy() - want)
    assert d.max() <= 2e-2 and d.mean() <= 2e-3
    # the two sequences share blocks 0 and 1 but wrote their token 40 into different blocks
    assert bt_h[0, :2].tolist() == bt_h[1, :2].tolist() and bt_h[0, 2] != bt_h[1, 2]
