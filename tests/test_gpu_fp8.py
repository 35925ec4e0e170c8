"""GPU parity of the E4M3 (fp8) KV cache path against the CPU oracle.

pkv_kv_store_fp8 must match the oracle's codes bit for bit; pkv_paged_decode_fp8
must stay within the decode tolerance (max-abs 2e-2, mean-abs 2e-3) of the
oracle's fp64 attention over the same codes and scales.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_62_gb300 import pkv
from paged_kv_cache_62_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
NTHREADS = 16


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


def quantise(x: torch.Tensor, scale: torch.Tensor) -> torch.Tensor:
    """Input generation only: E4M3 codes of x / scale[kv head] via torch's float8 cast, saturated at
    +-448 first (torch's cast turns magnitudes from 464 up into NaN; in range it is the oracle's
    rounding -- see the oracle pins).  NaN stays NaN."""
    y = x.float() / scale.view(1, 1, -1, 1)
    return torch.where(torch.isnan(y), y, y.clamp(-448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8)


def synth_fp8(B, Hq, Hkv, D, bs, seed, lens, extra=5):
    """Random paged problem with E4M3 caches, a shuffled pool and NaN codes in unowned rows."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    nblk = [-(-int(x) // bs) for x in lens]
    NB = sum(nblk) + extra
    perm = rng.permutation(NB)
    bt = np.full((B, max(max(nblk), 1)), -1, np.int32)
    filled = np.zeros(NB, np.int64)
    cur = 0
    for b in range(B):
        for i in range(nblk[b]):
            bt[b, i] = perm[cur]
            filled[perm[cur]] = min(bs, int(lens[b]) - i * bs)
            cur += 1
    ks = torch.as_tensor(rng.uniform(0.004, 0.02, Hkv), dtype=torch.float32, device="cuda")
    vs = torch.as_tensor(rng.uniform(0.004, 0.02, Hkv), dtype=torch.float32, device="cuda")
    kc = quantise(torch.randn(NB, bs, Hkv, D, generator=g, device="cuda"), ks)
    vc = quantise(torch.randn(NB, bs, Hkv, D, generator=g, device="cuda"), vs)
    canary = torch.arange(bs, device="cuda").view(1, bs) >= torch.as_tensor(filled, device="cuda").view(NB, 1)
    kc[canary] = 0x7F
    vc[canary] = 0xFF
    q = torch.randn(B, Hq, D, generator=g, device="cuda").bfloat16()
    return q, kc, vc, ks, vs, torch.from_numpy(bt).cuda(), torch.from_numpy(lens.astype(np.int32)).cuda()


def oracle_fp8(q, kc, vc, ks, vs, bt, lens, scale):
    return oracle.paged_decode_fp8(W.bits(q), kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy(),
                                   bt.cpu().numpy(), lens.cpu().numpy(), scale, nthreads=NTHREADS)


def run_fp8(q, kc, vc, ks, vs, bt, lens, scale, num_workers=0, ws=None, err=None):
    B, Hq, D = q.shape
    out = torch.full_like(q, float("nan"))
    ws = pkv.alloc_workspace(B, Hq, kc.shape[2], D) if ws is None else ws
    pkv.paged_decode_fp8(q, kc, vc, ks, vs, bt, lens, scale, out, ws, num_workers=num_workers, err_word=err)
    return out


@pytest.mark.parametrize("T,Hkv,D", [(7, 8, 128), (33, 2, 64), (3, 1, 64)])
def test_kv_store_fp8_bit_exact(T, Hkv, D):
    NB, bs = 20, 16
    rng = np.random.default_rng(T)
    g = torch.Generator(device="cuda").manual_seed(T)
    k = (torch.randn(T, Hkv, D, generator=g, device="cuda") * 3).bfloat16()
    v = torch.randn(T, Hkv, D, generator=g, device="cuda").bfloat16()
    k[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0]).bfloat16()      # saturation, signed zeros
    ks = torch.as_tensor(rng.uniform(0.003, 0.05, Hkv), dtype=torch.float32, device="cuda")
    vs = torch.as_tensor(rng.uniform(0.003, 0.05, Hkv), dtype=torch.float32, device="cuda")
    slots = rng.permutation(NB * bs)[:T].astype(np.int32)
    slots[T // 2] = -1
    kc = torch.randint(0, 255, (NB, bs, Hkv, D), dtype=torch.uint8, device="cuda")
    vc = torch.randint(0, 255, (NB, bs, Hkv, D), dtype=torch.uint8, device="cuda")
    kh, vh = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_store_fp8(k, v, torch.from_numpy(slots).cuda(), kc, vc, ks, vs, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    oracle.kv_store_fp8(W.bits(k), W.bits(v), slots, kh, vh, ks.cpu().numpy(), vs.cpu().numpy())
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", [(8, 2), (16, 4), (16, 8)])
@pytest.mark.parametrize("bs", [8, 16, 256])
def test_decode_fp8_matrix(D, heads, bs):
    Hq, Hkv = heads
    lens = [1, 15, 16, 17, 128, 511, 1024, 40]
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(len(lens), Hq, Hkv, D, bs, seed=D + bs + Hq, lens=lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884), f"D{D} {heads} bs{bs}")


@pytest.mark.parametrize("G", range(1, 9))
@pytest.mark.parametrize("D", [64, 128])
def test_decode_fp8_every_group_size(G, D):
    Hkv = 2
    lens = [300, 1, 77, 0, 1500]
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(len(lens), G * Hkv, Hkv, D, 16, seed=G * 3 + D, lens=lens)
    out = run_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.125)
    want = oracle_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.125)
    check_close(out, want, f"G{G} D{D}")
    assert torch.all(out[3].float() == 0)


@pytest.mark.parametrize("Hkv", [3, 5, 7])
def test_decode_fp8_head_groups_below_eight_warps(Hkv):
    """Head groups of 3 (x 2 slices), 5 and 7 kv heads: 6, 5 and 7 consumer warps run the set-up."""
    lens = [700, 1, 33, 250, 96]
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(len(lens), 2 * Hkv, Hkv, 128, 16, seed=Hkv * 5, lens=lens)
    want = oracle_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884)
    ws = pkv.alloc_workspace(len(lens), 2 * Hkv, Hkv, 128)
    for call in range(2):  # the second call sizes its slices from the first one's timings
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = run_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884, ws=ws, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"Hkv{Hkv} call{call}")


@pytest.mark.parametrize("workers", [1, 7, 333, 4096])
def test_decode_fp8_forced_splits(workers):
    lens = [1, 15, 17, 40, 300, 0, 1024, 2, 513]
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(len(lens), 16, 8, 128, 16, seed=workers, lens=lens)
    out = run_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884, num_workers=workers)
    check_close(out, oracle_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884), f"workers {workers}")


def test_decode_fp8_repeated_adaptive_calls():
    rng = np.random.default_rng(8)
    lens = rng.integers(1, 3000, size=40).tolist()
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(len(lens), 16, 8, 128, 16, seed=8, lens=lens)
    want = oracle_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884)
    ws = pkv.alloc_workspace(len(lens), 16, 8, 128)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(5):
        out = run_fp8(q, kc, vc, ks, vs, bt, lens_t, 0.0884, ws=ws, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"call {call}")


def test_qwen3_shaped_batch_in_fp8():
    """The Qwen3-0.6B-shaped decode batch with its caches quantised per kv head (scale = max |x| / 448):
    store the step's new rows with pkv_kv_store_fp8, decode with pkv_paged_decode_fp8, compare both
    with the oracle on the same codes."""
    wl = W.make("qwen3_0p6b", "cuda")
    s, lay = wl.spec, wl.layers[0]
    fin = lambda x: torch.nan_to_num(x.float(), nan=0.0)
    ks = (fin(lay.k_cache).abs().amax(dim=(0, 1, 3)) / 448).clamp_min(1e-6).contiguous()
    vs = (fin(lay.v_cache).abs().amax(dim=(0, 1, 3)) / 448).clamp_min(1e-6).contiguous()
    kc, vc = quantise(lay.k_cache, ks).contiguous(), quantise(lay.v_cache, vs).contiguous()
    slots = torch.from_numpy(oracle.decode_slot_mapping(wl.block_tables.cpu().numpy(), wl.lens_host(),
                                                        s.block_size, wl.num_tokens)).cuda()
    kh, vh = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.kv_store_fp8(lay.k_new, lay.v_new, slots, kc, vc, ks, vs, err)
    out = torch.empty_like(lay.q)
    ws = pkv.alloc_workspace(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim)
    pkv.paged_decode_fp8(lay.q, kc, vc, ks, vs, wl.block_tables, wl.context_lens, wl.scale, out, ws,
                         max_context_len=int(wl.lens_host().max()), err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    oracle.kv_store_fp8(W.bits(lay.k_new), W.bits(lay.v_new), slots.cpu().numpy(), kh, vh, ks.cpu().numpy(),
                        vs.cpu().numpy())
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    want = oracle.paged_decode_fp8(W.bits(lay.q), kh, vh, ks.cpu().numpy(), vs.cpu().numpy(),
                                   wl.block_tables.cpu().numpy(), wl.lens_host(), wl.scale, nthreads=NTHREADS)
    check_close(out, want, "qwen3_0p6b fp8")


@pytest.mark.parametrize("workers", [0, 7, 333])
@pytest.mark.parametrize("D,bs", [(128, 16), (64, 8), (128, 256)])
def test_decode_and_store_fp8_in_one_launch(workers, D, bs):
    """pkv_paged_decode_store_fp8: the new rows quantised and stored as pkv_kv_store_fp8 would (codes bit
    for bit, against the oracle), the attention over the stored codes within the decode tolerance, slots
    as the oracle's slot mapping; a padding row (context_len 0) stores nothing and gives zeros."""
    lens = [1, 15, 16, 17, 300, 0, 1024, 2, 513]
    B, Hq, Hkv = len(lens), 16, 8
    q, kc, vc, ks, vs, bt, lens_t = synth_fp8(B, Hq, Hkv, D, bs, seed=workers + D + bs, lens=lens)
    g = torch.Generator(device="cuda").manual_seed(workers + 1)
    k_new = (torch.randn(B, Hkv, D, generator=g, device="cuda") * 0.01).bfloat16()
    v_new = (torch.randn(B, Hkv, D, generator=g, device="cuda") * 0.01).bfloat16()
    k_new[0, 0, :3] = torch.tensor([1e4, -1e4, 0.0]).bfloat16()   # saturation
    kh, vh = kc.cpu().numpy().copy(), vc.cpu().numpy().copy()
    slots = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, float("nan"))
    ws = pkv.alloc_workspace(B, Hq, Hkv, D)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_decode_store_fp8(q, k_new, v_new, kc, vc, ks, vs, bt, lens_t, 0.0884, out, ws, slot_mapping=slots,
                               num_workers=workers, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    want_slots = oracle.decode_slot_mapping(bt.cpu().numpy(), np.asarray(lens, np.int32), bs, B)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    oracle.kv_store_fp8(W.bits(k_new), W.bits(v_new), want_slots, kh, vh, ks.cpu().numpy(), vs.cpu().numpy())
    assert np.array_equal(kc.cpu().numpy(), kh) and np.array_equal(vc.cpu().numpy(), vh)
    want = oracle.paged_decode_fp8(W.bits(q), kh, vh, ks.cpu().numpy(), vs.cpu().numpy(), bt.cpu().numpy(),
                                   np.asarray(lens, np.int32), 0.0884, nthreads=NTHREADS)
    check_close(out, want, f"workers {workers} D{D} bs{bs}")
    assert torch.all(out[lens.index(0)].float() == 0)
