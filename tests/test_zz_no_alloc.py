"""The allocation-free decode entry point (GPU).

pkv_paged_decode_noalloc serves callers that cannot allocate device memory
(an engine whose KV block pool took the free memory, a plugin interface that
passes only inputs and outputs): it uses a fixed scratch array inside the
library instead of a caller workspace.  Every call on a device shares that
array, so each call here finds the previous call's leftovers in it -- of
other sizes, in both orders (a small batch, then a larger one, then small
again), with the default and a fixed split, and a batch large enough that
its arrival counters live outside the array's fixed counter region -- and
must match both pkv_paged_decode on the same inputs and the CPU oracle.

The first call on a device is the set-up call with num_seqs == 0: it loads
the array and looks up its address without launching anything.

Self-contained, so it passes alone in a fresh process as well as after the
rest of the suite.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _problem(lens, Hq, Hkv, D, bs, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    nblk = [-(-int(x) // bs) for x in lens]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    bt = np.full((len(lens), max(nblk)), -1, np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    kc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    vc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    q = torch.randn(len(lens), Hq, D, generator=g, device="cuda").bfloat16()
    return (q, kc, vc, torch.from_numpy(bt).cuda(),
            torch.tensor(lens, dtype=torch.int32, device="cuda"))


def _close(got, want, what):
    d = np.abs(got.float().cpu().double().numpy() - want)
    assert np.isfinite(d).all(), what
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, f"{what}: max {d.max():.3g} mean {d.mean():.3g}"


def test_noalloc_matches_workspace_entry_point_and_oracle_on_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import oracle
    from paged_kv_cache_62_gb300 import pkv, workloads

    torch.cuda.set_device(0)
    lib = pkv.load()
    # set-up call on this device: nothing to compute, nothing launched
    st = lib.pkv_paged_decode_noalloc(None, None, None, None, 1, None, 0, 16, 8, 128, 256, 1, 0, 0.1, None, 0,
                                      None, torch.cuda.current_stream().cuda_stream)
    assert st == pkv.OK
    rng = np.random.default_rng(5)
    qwen3 = ([700, 1500, 33, 1, 4096, 250], 16, 8, 128, 256, 21)      # Qwen3-0.6B-shaped heads, split-K merges
    qwen25 = ([129, 17, 160, 192, 5], 14, 2, 64, 16, 22)              # Qwen2.5-0.5B-shaped heads
    many = ([int(x) for x in rng.integers(1, 48, 2100)], 16, 8, 128, 16, 23)  # 16800 arrival counters
    calls = [(qwen25, 0), (qwen3, 0), (qwen25, 0), (qwen3, 333), (many, 0), (qwen3, 0)]
    for (lens, Hq, Hkv, D, bs, seed), workers in calls:
        what = f"B={len(lens)} Hkv={Hkv} workers={workers}"
        q, kc, vc, bt, ctx = _problem(lens, Hq, Hkv, D, bs, seed)
        scale = 1.0 / math.sqrt(D)
        ref = torch.empty_like(q)
        ws = pkv.alloc_workspace(len(lens), Hq, Hkv, D)
        pkv.paged_decode(q, kc, vc, bt, ctx, scale, ref, ws, max_context_len=max(lens), num_workers=workers)
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.paged_decode_noalloc(q, kc, vc, bt, ctx, scale, out, max_context_len=max(lens), num_workers=workers,
                                 err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0, what
        d = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all(), what
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, what
        if workers > 0:  # a fixed split gives the same partial states in the same order: the same bits
            assert torch.equal(out, ref), what
        want = oracle.paged_decode(workloads.bits(q), workloads.bits(kc), workloads.bits(vc), bt.cpu().numpy(),
                                   ctx.cpu().numpy(), scale, nthreads=16)
        _close(out, want, what)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from paged_kv_cache_62_gb300 import build, pkv
    build.build()
    lib = pkv.load()
    B, Hq, Hkv, D = 16000, 64, 8, 128     # needs far more than the fixed scratch
    assert lib.pkv_paged_decode_workspace_size(B, Hq, Hkv, D) > pkv.NOALLOC_SCRATCH_BYTES
    st = lib.pkv_paged_decode_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 4, 0x10000, B, Hq, Hkv, D, 16, 10,
                                      64, 0.1, 0x10000, 0, None, None)
    assert st == pkv.EWORKSPACE
