"""GPU parity of pkv_paged_attention (several new tokens per sequence: prefill
chunks over a cached prefix mixed with decode steps) against the CPU oracle,
within the decode tolerance (max-abs 2e-2, mean-abs 2e-3)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_62_gb300 import pkv
from paged_kv_cache_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def check_close(got, want, what):
    g = got.float().cpu().double().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - want)
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, f"{what}: max {d.max():.3g} mean {d.mean():.3g}"


def mixed_batch(lens, news, Hq, Hkv, D, bs, seed):
    """Shuffled bf16 pool with NaN canaries in unowned rows, and queries for each sequence's new tokens."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk) + 4
    perm = rng.permutation(NB)
    bt = np.full((len(lens), max(nblk)), -1, np.int32)
    filled = np.zeros(NB, np.int64)
    cur = 0
    for b, L in enumerate(lens):
        for i in range(nblk[b]):
            bt[b, i] = perm[cur]
            filled[perm[cur]] = min(bs, L - i * bs)
            cur += 1
    kc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    vc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    canary = torch.arange(bs, device="cuda").view(1, bs) >= torch.as_tensor(filled, device="cuda").view(NB, 1)
    kc[canary] = float("nan")
    vc[canary] = float("nan")
    cu = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    q = torch.randn(int(cu[-1]), Hq, D, generator=g, device="cuda").bfloat16()
    return (q, kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(cu).cuda(),
            torch.tensor(lens, dtype=torch.int32, device="cuda"))


def oracle_of(q, kc, vc, bt, cu, lens, scale):
    return oracle.paged_attention(W.bits(q), W.bits(kc), W.bits(vc), bt.cpu().numpy(), cu.cpu().numpy(),
                                  lens.cpu().numpy(), scale, nthreads=16)


def run(q, kc, vc, bt, cu, lens, scale, workers=0, ws=None, err=None):
    T, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    ws = pkv.alloc_attention_workspace(T, Hq, kc.shape[2], D) if ws is None else ws
    pkv.paged_attention(q, kc, vc, bt, cu, lens, scale, out, ws, num_workers=workers, err_word=err)
    return out


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(16, 8, 128, 16), (14, 2, 64, 16), (8, 2, 64, 256), (16, 4, 128, 8)])
def test_mixed_prefill_chunks_and_decodes(Hq, Hkv, D, bs):
    lens = [300, 17, 1, 700, 129, 64, 2000, 5]
    news = [300, 17, 1, 1, 40, 64, 3, 2]      # whole prefills, prefill chunks after a cached prefix, decodes
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, Hq, Hkv, D, bs, seed=Hq + D + bs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(q, kc, vc, bt, cu, lens_t, 0.0884, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884), f"{Hq}/{Hkv} D{D} bs{bs}")


@pytest.mark.parametrize("workers", [1, 7, 500])
def test_forced_splits_and_repeated_calls(workers):
    lens = [900, 33, 400, 1]
    news = [100, 33, 2, 1]
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, 16, 8, 128, 16, seed=workers)
    want = oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884)
    check_close(run(q, kc, vc, bt, cu, lens_t, 0.0884, workers=workers), want, f"workers {workers}")
    ws = pkv.alloc_attention_workspace(q.shape[0], 16, 8, 128)
    for call in range(3):  # the default split over one workspace, call after call
        check_close(run(q, kc, vc, bt, cu, lens_t, 0.0884, ws=ws), want, f"call {call}")


def test_inconsistent_offsets_give_zeros_and_an_error():
    lens = [10, 20]
    news = [3, 4]
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, 8, 2, 64, 16, seed=1)
    bad_lens = torch.tensor([2, 20], dtype=torch.int32, device="cuda")   # 3 new tokens in a length-2 sequence
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(q, kc, vc, bt, cu, bad_lens, 0.125, err=err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_CONTEXT_RANGE
    assert torch.all(out[:3].float() == 0)
    want = oracle.paged_attention(W.bits(q)[3:], W.bits(kc), W.bits(vc), bt.cpu().numpy()[1:],
                                  np.array([0, 4], np.int32), np.array([20], np.int32), 0.125)
    check_close(out[3:], want, "the consistent sequence")
    short = torch.tensor([0, 3, 5], dtype=torch.int32, device="cuda")   # offsets end before the last rows
    err.zero_()
    out = run(q, kc, vc, bt, short, lens_t, 0.125, err=err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_CONTEXT_RANGE
    assert torch.all(out[5:].float() == 0)


@pytest.mark.parametrize("Hq,Hkv,D,bs,workers", [(8, 8, 64, 16, 0), (6, 2, 64, 16, 0), (6, 2, 64, 8, 77),
                                                 (16, 8, 128, 256, 0), (32, 8, 128, 16, 500)])
def test_long_prefill_chunks_share_passes(Hq, Hkv, D, bs, workers):
    """Prefill chunks of many tokens after a cached prefix: consecutive queries of a sequence go in
    chunks of max(1, 8 // G) (G = 1: 8, G = 3: 2, G = 2: 4, G = 4: 2), the last chunk of a sequence
    shorter; every query keeps its own causal bound."""
    lens = [700, 129, 1, 333, 64, 1200]
    news = [250, 129, 1, 7, 33, 5]          # whole prefill, partial chunks, a decode
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, Hq, Hkv, D, bs, seed=Hq * 7 + bs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884)
    ws = pkv.alloc_attention_workspace(q.shape[0], Hq, Hkv, D)
    for call in range(2):
        out = run(q, kc, vc, bt, cu, lens_t, 0.0884, workers=workers, ws=ws, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"{Hq}/{Hkv} bs{bs} call {call}")


@pytest.mark.parametrize("workers", [0, 250])
def test_prefill_batch_past_512_entries(workers):
    """More than 512 query rows (entries): split-K pieces numbered by slice; whole prefills, chunks
    after a prefix and decodes."""
    lens = [900, 400, 333, 64, 1, 2000, 17] + [50 + 7 * i for i in range(40)]
    news = [300, 400, 200, 10, 1, 3, 17] + [1] * 40
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, 16, 8, 64, 16, seed=950 + workers)
    assert q.shape[0] > 512
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(q, kc, vc, bt, cu, lens_t, 0.125, workers=workers, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_of(q, kc, vc, bt, cu, lens_t, 0.125), f"workers {workers}")


@pytest.mark.parametrize("Hq,Hkv,D,workers", [(16, 8, 128, 0), (16, 8, 128, 97), (14, 2, 64, 0), (8, 8, 64, 0)])
def test_short_runs_of_new_tokens_on_regular_ctas(Hq, Hkv, D, workers):
    """A batch of short runs (speculative verify steps and decodes, offsets given, at most two chunks of
    16 / G queries per sequence on average): chunks on regular CTAs, up to 16 (query, head) pairs a warp."""
    rng = np.random.default_rng(Hq + Hkv + workers)
    news = rng.integers(1, 9, size=24).tolist()
    lens = [int(n) + int(x) for n, x in zip(news, rng.integers(0, 1500, size=24))]
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, Hq, Hkv, D, 16, seed=Hq * 3 + workers)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(q, kc, vc, bt, cu, lens_t, 0.0884, workers=workers, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884), f"{Hq}/{Hkv} D{D} workers {workers}")


def test_same_n_with_a_too_short_sequence():
    """new_per_seq = n with a sequence of fewer than n cached tokens: its rows are zero and the
    error word says so; the other sequences are exact (the n queries share one pass)."""
    n = 3
    lens = [40, 2, 0, 90]
    good = [0, 3]
    q, kc, vc, bt, cu, lens_t = mixed_batch([40, 3, 3, 90], [n] * 4, 16, 8, 128, 16, seed=5)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    ws = pkv.alloc_attention_workspace(q.shape[0], 16, 8, 128)
    pkv.paged_attention(q, kc, vc, bt, None, lens_t, 0.0884, out, ws, err_word=err, new_per_seq=n)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_CONTEXT_RANGE
    assert torch.all(out[n:3 * n].float() == 0)
    for b in good:
        rows = slice(b * n, b * n + n)
        want = oracle.paged_attention(W.bits(q)[rows], W.bits(kc), W.bits(vc), bt.cpu().numpy()[b:b + 1],
                                      np.array([0, n], np.int32), np.array([lens[b]], np.int32), 0.0884)
        check_close(out[rows], want, f"sequence {b}")


@pytest.mark.parametrize("n,Hq,Hkv,D,bs,workers", [(2, 16, 8, 128, 16, 0), (3, 16, 8, 128, 256, 0),
                                                   (4, 16, 8, 128, 16, 0), (4, 16, 8, 128, 8, 333),
                                                   (8, 4, 4, 64, 16, 0), (4, 14, 2, 64, 16, 1),
                                                   (5, 16, 8, 128, 16, 0), (8, 16, 8, 128, 16, 0),
                                                   (8, 16, 8, 128, 256, 250), (16, 8, 8, 64, 16, 0),
                                                   (12, 16, 8, 128, 16, 77), (6, 12, 2, 128, 8, 0)])
def test_uniform_new_tokens_share_one_pass(n, Hq, Hkv, D, bs, workers):
    """Every sequence with n new tokens (new_per_seq = n): when n * G <= 16 the n queries are n * G virtual
    heads of a kv head over one pass of its keys (both 8-row halves of the MMA tile past 8), each with its
    own causal bound -- including pieces of a split where some virtual head sees no key at all; longer runs
    go in chunks (of 16 / G queries on regular CTAs, or of 8 x that on query-split CTAs)."""
    rng = np.random.default_rng(n * 100 + Hq + bs)
    lens = rng.integers(n, 1500, size=12).tolist() + [n, n + 1, 16 + n - 1]
    news = [n] * len(lens)
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, Hq, Hkv, D, bs, seed=n + D)
    want = oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884)
    T = q.shape[0]
    ws = pkv.alloc_attention_workspace(T, Hq, Hkv, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention(q, kc, vc, bt, None, lens_t, 0.0884, out, ws, num_workers=workers, err_word=err,
                            new_per_seq=n)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"n {n} call {call}")


# --------------------------------------------------------------------------- tensor-memory query-split CTAs
# Long runs of new tokens with gq = Hq / Hkv a power of two and block_size >= 128 run on the tcgen05 CTAs:
# 128-row entries (128 / gq queries x gq heads) against 128-key tiles, scores and outputs in tensor memory.
@pytest.mark.parametrize("Hq,Hkv,D,bs,workers", [
    (16, 8, 128, 256, 0), (16, 8, 128, 128, 0), (8, 8, 128, 128, 0), (32, 8, 64, 128, 0), (64, 8, 128, 256, 0),
    (16, 1, 64, 512, 0), (16, 8, 128, 256, 7), (16, 8, 128, 256, 333), (16, 8, 128, 128, 2000),
    (16, 8, 128, 1024, 0)])
def test_tensor_memory_prefill_chunks(Hq, Hkv, D, bs, workers):
    """Whole prefills, 64-query chunks and partial chunks after cached prefixes (up to 5000 keys: split over
    several CTAs and merged), decodes; every query with its own causal bound; repeated calls on one
    workspace."""
    lens = [5000, 700, 129, 1, 333, 64, 1200, 2100]
    news = [64, 250, 129, 1, 100, 33, 2, 190]
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, Hq, Hkv, D, bs, seed=Hq * 13 + Hkv + D + bs + workers)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884)
    ws = pkv.alloc_attention_workspace(q.shape[0], Hq, Hkv, D)
    for call in range(3):
        out = run(q, kc, vc, bt, cu, lens_t, 0.0884, workers=workers, ws=ws, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"{Hq}/{Hkv} D{D} bs{bs} workers {workers} call {call}")


def test_tensor_memory_prefill_chunk_of_the_qwen3_shape():
    """The Qwen3-0.6B-shaped layer (16 q / 8 kv heads, head_dim 128, block_size 256): the last 64 tokens of
    each sequence as one prefill chunk over its cached prefix, context lengths U[512, 4096]."""
    rng = np.random.default_rng(64)
    lens = [int(x) for x in rng.integers(512, 4097, 12)]
    news = [64] * len(lens)
    q, kc, vc, bt, cu, lens_t = mixed_batch(lens, news, 16, 8, 128, 256, seed=65)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run(q, kc, vc, bt, cu, lens_t, 0.0884, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_of(q, kc, vc, bt, cu, lens_t, 0.0884), "64-token chunks")
