"""The allocation-free decode entry point against the regular one (GPU).

pkv_paged_decode_noalloc serves callers that cannot allocate device memory
(an engine whose KV block pool took the free memory, a plugin interface that
passes only inputs and outputs): it uses a fixed scratch array inside the
library instead of a caller workspace.  Two calls in a row, on different
batches, must each match pkv_paged_decode on the same inputs -- the second
call finds the first call's leftovers in the shared array and must not care.

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


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_cache_62_gb300 import pkv

    torch.cuda.set_device(0)
    cases = [
        ([700, 1500, 33, 1, 4096, 250], 16, 8, 128, 256, 21),   # Qwen3-0.6B-shaped heads, split-K merges
        ([129, 17, 160, 192, 5], 14, 2, 64, 16, 22),            # Qwen2.5-0.5B-shaped heads
    ]
    for lens, Hq, Hkv, D, bs, seed in cases:
        q, kc, vc, bt, ctx = _problem(lens, Hq, Hkv, D, bs, seed)
        scale = 1.0 / math.sqrt(D)
        ref = torch.empty_like(q)
        ws = pkv.alloc_workspace(len(lens), Hq, Hkv, D)
        pkv.paged_decode(q, kc, vc, bt, ctx, scale, ref, ws, max_context_len=max(lens))
        out = torch.full_like(q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pkv.paged_decode_noalloc(q, kc, vc, bt, ctx, scale, out, max_context_len=max(lens), err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        d = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS


def test_noalloc_rejects_sizes_beyond_its_scratch():
    from paged_kv_cache_62_gb300 import build, pkv
    build.build()
    lib = pkv.load()
    B, Hq, Hkv, D = 16000, 64, 8, 128     # needs far more than the fixed scratch
    assert lib.pkv_paged_decode_workspace_size(B, Hq, Hkv, D) > pkv.NOALLOC_SCRATCH_BYTES
    st = lib.pkv_paged_decode_noalloc(0x10000, 0x10000, 0x10000, 0x10000, 4, 0x10000, B, Hq, Hkv, D, 16, 10,
                                      64, 0.1, 0x10000, 0, None, None)
    assert st == pkv.EWORKSPACE
