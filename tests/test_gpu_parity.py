"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

kv_store and the slot mapping must match bit for bit; paged_decode must stay
within max-abs 2e-2 and mean-abs 2e-3 of the fp64 oracle (bf16 inputs, fp32
accumulation, bf16 output).
"""
import math

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


def err_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def check_close(got: torch.Tensor, want: np.ndarray, what: str):
    g = got.float().cpu().double().numpy()
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - want)
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, f"{what}: max {d.max():.3g} mean {d.mean():.3g}"
    return d


def run_decode(q, kc, vc, bt, lens, scale, max_ctx=None, num_workers=0, err=None):
    B, Hq, D = q.shape
    Hkv = kc.shape[2]
    out = torch.full_like(q, float("nan"))
    ws = shared_workspace(B, Hq, Hkv, D)  # left by earlier, differently sized calls: must not matter
    pkv.paged_decode(q, kc, vc, bt, lens, scale, out, ws, max_context_len=max_ctx, num_workers=num_workers,
                     err_word=err)
    return out


_WS = {}


def shared_workspace(B, Hq, Hkv, D):
    """One zero-filled workspace per process, grown on demand and reused by every test that
    does not bring its own: each call finds the state the previous (other-sized) call left."""
    need = pkv.paged_decode_workspace_size(B, Hq, Hkv, D)
    ws = _WS.get("ws")
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 64 << 20), dtype=torch.uint8, device="cuda")
        _WS["ws"] = ws
    return ws


def oracle_slots(wl):
    s = oracle.decode_slot_mapping(wl.block_tables.cpu().numpy(), wl.context_lens.cpu().numpy(),
                                   wl.spec.block_size, wl.num_tokens)
    for t in wl.skip_tokens:
        s[t] = -1
    return s


# --------------------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("name", W.ORDER)
def test_slot_mapping_bit_exact(name):
    wl = W.make(name, "cuda", layers=1)
    err = err_word()
    got = torch.full((wl.num_tokens,), 7, dtype=torch.int32, device="cuda")
    pkv.decode_slot_mapping(wl.block_tables, wl.context_lens, wl.spec.block_size, wl.num_blocks, got, err)
    want = oracle.decode_slot_mapping(wl.block_tables.cpu().numpy(), wl.context_lens.cpu().numpy(),
                                      wl.spec.block_size, wl.num_tokens)
    assert np.array_equal(got.cpu().numpy(), want)
    assert err.item() == 0


@pytest.mark.parametrize("name", W.ORDER)
def test_store_then_decode(name):
    """One decode step per layer: kv_store (bit-exact over the whole pool) then paged_decode, on every layer
    (all 28 of the full-depth workload, one after the other on one workspace)."""
    wl = W.make(name, "cuda")
    s = wl.spec
    bt_h, lens_h = wl.block_tables.cpu().numpy(), wl.context_lens.cpu().numpy()
    slots_h = oracle_slots(wl)
    slots = torch.from_numpy(slots_h).cuda()
    err = err_word()
    ws = pkv.alloc_workspace(s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim)
    for li, lay in enumerate(wl.layers):
        kc_h, vc_h = W.bits(lay.k_cache), W.bits(lay.v_cache)
        pkv.kv_store(lay.k_new, lay.v_new, slots, lay.k_cache, lay.v_cache, err)
        out = torch.empty_like(lay.q)
        pkv.paged_decode(lay.q, lay.k_cache, lay.v_cache, wl.block_tables, wl.context_lens, wl.scale, out, ws,
                         max_context_len=int(lens_h.max()), err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0, hex(err.item())
        oracle.kv_store(W.bits(lay.k_new), W.bits(lay.v_new), slots_h, kc_h, vc_h)
        assert np.array_equal(W.bits(lay.k_cache), kc_h), "k_cache differs from the oracle store"
        assert np.array_equal(W.bits(lay.v_cache), vc_h), "v_cache differs from the oracle store"
        want = oracle.paged_decode(W.bits(lay.q), kc_h, vc_h, bt_h, lens_h, wl.scale, nthreads=NTHREADS)
        check_close(out, want, f"{name} layer {li}")
        del kc_h, vc_h


@pytest.mark.parametrize("name", W.ORDER)
def test_fused_decode_store_bit_exact(name):
    """pkv_decode_store (slot of position L - 1, then the store, in one launch) against the oracle's
    slot mapping and store; one sequence turned into a padding row (context_len 0) writes nothing."""
    wl = W.make(name, "cuda", layers=1)
    s, lay = wl.spec, wl.layers[0]
    B = s.num_seqs
    lens = wl.context_lens.clone()
    lens[B // 2] = 0
    lens_h = lens.cpu().numpy()
    bt_h = wl.block_tables.cpu().numpy()
    kc_h, vc_h = W.bits(lay.k_cache), W.bits(lay.v_cache)
    slots = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    err = err_word()
    pkv.decode_store(lay.k_new[:B].contiguous(), lay.v_new[:B].contiguous(), wl.block_tables, lens, lay.k_cache,
                     lay.v_cache, slots, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    want = oracle.decode_slot_mapping(bt_h, lens_h, s.block_size, B)
    assert want[B // 2] == -1
    assert np.array_equal(slots.cpu().numpy(), want)
    oracle.kv_store(W.bits(lay.k_new)[:B], W.bits(lay.v_new)[:B], want, kc_h, vc_h)
    assert np.array_equal(W.bits(lay.k_cache), kc_h) and np.array_equal(W.bits(lay.v_cache), vc_h)


@pytest.mark.parametrize("name", W.ORDER)
def test_decode_and_store_in_one_launch(name):
    """pkv_paged_decode_store: the store (slots and cache bit for bit, as the oracle's slot mapping and
    store) and the attention over the stored token (within the decode tolerance of the oracle's decode
    on the stored caches) in one launch; a padding row (context_len 0) stores nothing and gives zeros."""
    wl = W.make(name, "cuda", layers=1)
    s, lay = wl.spec, wl.layers[0]
    B = s.num_seqs
    lens = wl.context_lens.clone()
    lens[B // 2] = 0
    lens_h = lens.cpu().numpy()
    bt_h = wl.block_tables.cpu().numpy()
    kc_h, vc_h = W.bits(lay.k_cache), W.bits(lay.v_cache)
    k_new, v_new = lay.k_new[:B].contiguous(), lay.v_new[:B].contiguous()
    slots = torch.full((B,), 7, dtype=torch.int32, device="cuda")
    out = torch.full_like(lay.q, float("nan"))
    ws = shared_workspace(B, s.num_q_heads, s.num_kv_heads, s.head_dim)
    err = err_word()
    pkv.paged_decode_store(lay.q, k_new, v_new, lay.k_cache, lay.v_cache, wl.block_tables, lens, wl.scale, out, ws,
                           slot_mapping=slots, max_context_len=int(lens_h.max()), err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0, hex(err.item())
    want_slots = oracle.decode_slot_mapping(bt_h, lens_h, s.block_size, B)
    assert np.array_equal(slots.cpu().numpy(), want_slots)
    oracle.kv_store(W.bits(k_new), W.bits(v_new), want_slots, kc_h, vc_h)
    assert np.array_equal(W.bits(lay.k_cache), kc_h) and np.array_equal(W.bits(lay.v_cache), vc_h)
    want = oracle.paged_decode(W.bits(lay.q), kc_h, vc_h, bt_h, lens_h, wl.scale, nthreads=NTHREADS)
    check_close(out, want, name)
    assert torch.all(out[B // 2].float() == 0)


@pytest.mark.parametrize("name", ["tiny", "qwen25_0p5b"])
def test_bound_decode_step_matches_the_call(name):
    """DecodeStoreStep (the step bound to its buffers once) issues the same pkv_paged_decode_store: over three
    steps whose buffer contents change in place (new q and new K/V rows, lengths grown by one), its outputs and
    caches equal those of paged_decode_store run on copies of the same buffers, bit for bit (fixed split)."""
    wl = W.make(name, "cuda", layers=1)
    s, lay = wl.spec, wl.layers[0]
    B, Hq, Hkv, D = s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_dim
    q = lay.q.clone()
    k_new, v_new = lay.k_new[:B].contiguous(), lay.v_new[:B].contiguous()
    lens = (wl.context_lens - 3).clamp(min=0)  # three steps bring them back to the workload's lengths
    caches = [(lay.k_cache.clone(), lay.v_cache.clone()) for _ in range(2)]
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    wss = [torch.zeros(pkv.paged_decode_workspace_size(B, Hq, Hkv, D), dtype=torch.uint8, device="cuda")
           for _ in range(2)]
    err = err_word()
    cap = int(wl.context_lens.max())
    step = pkv.DecodeStoreStep(q, k_new, v_new, caches[0][0], caches[0][1], wl.block_tables, lens, wl.scale,
                               outs[0], wss[0], max_context_len=cap, num_workers=64, err_word=err)
    g = torch.Generator(device="cuda").manual_seed(3)
    for i in range(3):
        lens += (lens > 0).int()
        q.copy_(torch.randn(q.shape, generator=g, device="cuda").bfloat16())
        k_new.copy_(torch.randn(k_new.shape, generator=g, device="cuda").bfloat16())
        v_new.copy_(torch.randn(v_new.shape, generator=g, device="cuda").bfloat16())
        step.run()
        pkv.paged_decode_store(q, k_new, v_new, caches[1][0], caches[1][1], wl.block_tables, lens, wl.scale,
                               outs[1], wss[1], max_context_len=cap, num_workers=64, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0, hex(err.item())
        assert torch.equal(outs[0], outs[1]), f"{name} step {i}"
        # (bit patterns: the pools hold NaN canaries, which torch.equal never calls equal)
        assert np.array_equal(W.bits(caches[0][0]), W.bits(caches[1][0]))
        assert np.array_equal(W.bits(caches[0][1]), W.bits(caches[1][1]))
    lens_h = lens.cpu().numpy()
    want = oracle.paged_decode(W.bits(q), W.bits(caches[1][0]), W.bits(caches[1][1]), wl.block_tables.cpu().numpy(),
                               lens_h, wl.scale, nthreads=NTHREADS)
    check_close(outs[0], want, name)


@pytest.mark.parametrize("lens", [[1, 15, 40, 96, 0, 128], [1, 15, 600, 700, 5, 0]])
@pytest.mark.parametrize("heads", [(4, 2), (14, 2), (16, 8)])
def test_small_calls_one_cta_per_segment_or_split(lens, heads):
    """Calls with fewer units than SMs: when no (sequence, head group) segment has more than 8 units they
    run one CTA per segment (no split-K pieces); a longer segment sends the call back to one CTA per unit
    (pieces and merges).  Both against the oracle, with zero-length rows, on a workspace other calls used."""
    Hq, Hkv = heads
    for D, bs in ((64, 16), (128, 16)):
        q, kc, vc, bt, lens_t = synth(len(lens), 0, Hq, Hkv, D, bs, seed=sum(lens) + Hq + D, lens=lens)
        err = err_word()
        out = run_decode(q, kc, vc, bt, lens_t, 0.1, max_ctx=max(lens), err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, oracle_of(q, kc, vc, bt, lens_t, 0.1), f"lens {lens} heads {heads} D {D}")
        for b, L in enumerate(lens):
            if L == 0:
                assert torch.all(out[b].float() == 0)


@pytest.mark.parametrize("heads", [(16, 8), (32, 2), (24, 2)])
@pytest.mark.parametrize("workers", [0, 1, 7, 333])
def test_decode_and_store_split_over_workers(workers, heads):
    """The fused store where the new token's unit lands in a later slice than the sequence's first
    units (forced splits), over block sizes 8 and 16 (several boxes per unit); also with 16 and 12 query
    heads per kv head (the 16-row tiles, which load the new row when its tile comes)."""
    Hq, Hkv = heads
    for bs in (8, 16):
        lens = [1, 15, 16, 17, 300, 1024, 2, 513]
        q, kc, vc, bt, lens_t = synth(len(lens), 0, Hq, Hkv, 128, bs, seed=workers * 10 + bs + Hq, lens=lens)
        g = torch.Generator(device="cuda").manual_seed(workers + bs + Hq)
        k_new = torch.randn(len(lens), Hkv, 128, generator=g, device="cuda").bfloat16()
        v_new = torch.randn(len(lens), Hkv, 128, generator=g, device="cuda").bfloat16()
        kc_h, vc_h = W.bits(kc), W.bits(vc)
        ws = shared_workspace(len(lens), Hq, Hkv, 128)
        out = torch.empty_like(q)
        err = err_word()
        pkv.paged_decode_store(q, k_new, v_new, kc, vc, bt, lens_t, 0.0884, out, ws, num_workers=workers, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        slots = oracle.decode_slot_mapping(bt.cpu().numpy(), np.asarray(lens, np.int32), bs, len(lens))
        oracle.kv_store(W.bits(k_new), W.bits(v_new), slots, kc_h, vc_h)
        assert np.array_equal(W.bits(kc), kc_h) and np.array_equal(W.bits(vc), vc_h)
        want = oracle.paged_decode(W.bits(q), kc_h, vc_h, bt.cpu().numpy(), np.asarray(lens, np.int32), 0.0884,
                                   nthreads=NTHREADS)
        check_close(out, want, f"workers {workers} bs {bs} heads {heads}")


# --------------------------------------------------------------------------- mini-vLLM-style matrix
def synth(B, L, Hq, Hkv, D, bs, seed, lens=None, extra=5):
    """Random paged problem with a shuffled pool and NaN canaries in unowned rows."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    rng = np.random.default_rng(seed)
    lens = np.full(B, L, np.int64) if lens is None else np.asarray(lens, np.int64)
    nblk = [-(-int(x) // bs) for x in lens]
    NB = sum(nblk) + extra
    perm = rng.permutation(NB)
    mb = max(max(nblk), 1)
    bt = np.full((B, mb), -1, np.int32)
    cur = 0
    filled = np.zeros(NB, np.int64)
    for b in range(B):
        for i in range(nblk[b]):
            bt[b, i] = perm[cur]
            filled[perm[cur]] = min(bs, int(lens[b]) - i * bs)
            cur += 1
    kc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    vc = torch.randn(NB, bs, Hkv, D, generator=g, device="cuda").bfloat16()
    canary = torch.arange(bs, device="cuda").view(1, bs) >= torch.as_tensor(filled, device="cuda").view(NB, 1)
    kc[canary] = float("nan")
    vc[canary] = float("nan")
    q = torch.randn(B, Hq, D, generator=g, device="cuda").bfloat16()
    return q, kc, vc, torch.from_numpy(bt).cuda(), torch.from_numpy(lens.astype(np.int32)).cuda()


def oracle_of(q, kc, vc, bt, lens, scale):
    return oracle.paged_decode(W.bits(q), W.bits(kc), W.bits(vc), bt.cpu().numpy(), lens.cpu().numpy(), scale,
                               nthreads=NTHREADS)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("heads", [(8, 2), (16, 4)])
@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("B", [1, 4, 16])
def test_kernel_matrix(B, bs, heads, D):
    Hq, Hkv = heads
    for L in (1, 15, 16, 17, 128, 511, 1024):
        q, kc, vc, bt, lens = synth(B, L, Hq, Hkv, D, bs, seed=B * 100000 + bs * 1000 + Hq * 10 + L + D)
        scale = 1 / math.sqrt(D)
        err = err_word()
        out = run_decode(q, kc, vc, bt, lens, scale, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, oracle_of(q, kc, vc, bt, lens, scale), f"B{B} L{L} bs{bs} {Hq}/{Hkv} D{D}")


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_every_group_size(G, D):
    Hkv = 2
    lens = [1, 5, 16, 33, 200, 77]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, G * Hkv, Hkv, D, 16, seed=G * 7 + D, lens=lens)
    out = run_decode(q, kc, vc, bt, lens_t, 0.1)
    check_close(out, oracle_of(q, kc, vc, bt, lens_t, 0.1), f"G{G} D{D}")


@pytest.mark.parametrize("workers", [0, 7])
@pytest.mark.parametrize("G", [1, 2])
@pytest.mark.parametrize("Hkv", [1, 3, 5, 6, 7, 12])
def test_head_groups_of_any_size(Hkv, G, workers):
    """Kv-head counts whose head group (the largest divisor of Hkv up to 8) leaves 5, 6 or 7 consumer
    warps, or one head over 8 token slices: the decode set-up's scan and partition run on the consumer
    warps alone, so their count sets that barrier's size.  Three calls on one workspace: the second and
    third size their slices from the previous call's timings."""
    lens = [1, 17, 300, 64, 1000, 5, 256, 129]
    D = 128 if Hkv in (3, 5) else 64
    q, kc, vc, bt, lens_t = synth(len(lens), 0, G * Hkv, Hkv, D, 16, seed=Hkv * 31 + G + workers, lens=lens)
    want = oracle_of(q, kc, vc, bt, lens_t, 0.2)
    ws = pkv.alloc_workspace(len(lens), G * Hkv, Hkv, D)
    for call in range(3):
        out = torch.full_like(q, float("nan"))
        err = err_word()
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.2, out, ws, num_workers=workers, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0, (call, hex(err.item()))
        check_close(out, want, f"Hkv{Hkv} G{G} workers{workers} call{call}")


@pytest.mark.parametrize("workers", [1, 2, 3, 7, 64, 333, 4096])
def test_forced_splits(workers):
    """Spread the same batch over very different worker counts: exercises the split-K merge."""
    lens = [1, 15, 17, 40, 300, 0, 1024, 2, 513]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 16, seed=workers, lens=lens)
    want = oracle_of(q, kc, vc, bt, lens_t, 0.0884)
    out = run_decode(q, kc, vc, bt, lens_t, 0.0884, num_workers=workers)
    check_close(out, want, f"workers {workers}")
    assert torch.all(out[lens.index(0)].float() == 0)


@pytest.mark.parametrize("workers", [0, 97, 4096])
def test_many_sequences_slice_numbered_pieces(workers):
    """B * (kv head groups) >= 512: split-K pieces are numbered by slice (two per slice) instead of by
    sequence; long and short sequences mixed so that pieces start and end inside slices."""
    rng = np.random.default_rng(640 + workers)
    lens = rng.integers(0, 400, size=640)
    lens[::37] = 1500
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 64, 16, seed=workers + 3, lens=lens)
    want = oracle_of(q, kc, vc, bt, lens_t, 0.125)
    ws = shared_workspace(len(lens), 16, 8, 64)
    err = err_word()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.125, out, ws, num_workers=workers, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want, f"workers {workers} call {call}")


def test_alternating_batches_on_one_workspace():
    """Two different batches (other tables, lengths and pools) decoded in turn on one workspace: each
    call finds the previous call's balance table and L2 warm-up hints, which describe the other batch,
    and must still give exact results."""
    rng = np.random.default_rng(77)
    a = synth(48, 0, 16, 8, 128, 256, seed=5, lens=rng.integers(300, 3000, size=48))
    b = synth(40, 0, 16, 8, 128, 256, seed=6, lens=rng.integers(1, 2500, size=40))
    want = [oracle_of(*x[:5], 0.0884) for x in (a, b)]
    ws = pkv.alloc_workspace(48, 16, 8, 128)
    err = err_word()
    for call in range(6):
        q, kc, vc, bt, lens_t = a if call % 2 == 0 else b
        out = torch.full_like(q, float("nan"))
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.0884, out, ws, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, want[call % 2], f"call {call}")


@pytest.mark.parametrize("bs", [16, 256])
def test_adaptive_split_over_repeated_calls(bs):
    """Default split, eight calls on one workspace: each call sizes its per-SM slices from the
    previous call's timings, so the partition (and the split-K pieces) change from call to call;
    every call must match the oracle, whatever the partition it ended up with."""
    rng = np.random.default_rng(62)
    lens = rng.integers(1, 3000, size=40).tolist() + [0, 1, 8, 9, 127, 128, 129, 4096]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, bs, seed=bs, lens=lens)
    want = oracle_of(q, kc, vc, bt, lens_t, 0.0884)
    B, Hq, D = q.shape
    ws = pkv.alloc_workspace(B, Hq, kc.shape[2], D)
    err = err_word()
    for call in range(8):
        out = torch.full_like(q, float("nan"))
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.0884, out, ws, num_workers=0, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0, hex(err.item())
        check_close(out, want, f"call {call}")


def test_cuda_graph_replay():
    """The call captured once in a CUDA graph and replayed with new queries and lengths: nothing
    per call is baked into the launch (the call epoch lives in the workspace), so every replay
    must match the oracle, adaptive split included."""
    lens0 = [700, 1500, 33, 2047, 1, 300, 999, 64] * 3
    q, kc, vc, bt, lens_t = synth(len(lens0), 0, 16, 8, 128, 16, seed=11, lens=lens0)
    B, Hq, D = q.shape
    ws = pkv.alloc_workspace(B, Hq, kc.shape[2], D)
    err = err_word()
    out = torch.empty_like(q)
    mx = int(max(lens0))
    for _ in range(3):  # warm up (tensor maps, attributes) outside the capture
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.0884, out, ws, max_context_len=mx, err_word=err)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_decode(q, kc, vc, bt, lens_t, 0.0884, out, ws, max_context_len=mx, err_word=err)
    rng = np.random.default_rng(3)
    for rep_i in range(5):
        q.copy_(torch.randn(q.shape, generator=torch.Generator(device="cuda").manual_seed(rep_i), device="cuda")
                .to(torch.bfloat16))
        new = np.minimum(np.asarray(lens0) - rng.integers(0, 20, size=B), mx).clip(min=0)
        lens_t.copy_(torch.as_tensor(new, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        assert err.item() == 0, hex(err.item())
        check_close(out, oracle_of(q, kc, vc, bt, lens_t, 0.0884), f"replay {rep_i}")


def test_workspace_not_zero_filled_is_reported():
    """A workspace whose control block the library did not leave (here: all bytes 0xFF) sets
    PKV_ERR_WORKSPACE; the call still ends normally."""
    lens = [100, 200, 300]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 16, seed=9, lens=lens)
    B, Hq, D = q.shape
    ws = pkv.alloc_workspace(B, Hq, kc.shape[2], D)
    ws.fill_(0xFF)
    err = err_word()
    out = torch.empty_like(q)
    pkv.paged_decode(q, kc, vc, bt, lens_t, 0.0884, out, ws, err_word=err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_WORKSPACE


def test_workers_do_not_change_results_much():
    lens = [700, 1500, 33]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 256, seed=5, lens=lens)
    a = run_decode(q, kc, vc, bt, lens_t, 0.0884, num_workers=1).float()
    b = run_decode(q, kc, vc, bt, lens_t, 0.0884, num_workers=500).float()
    assert (a - b).abs().max().item() <= 2e-2


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), returned as fp64."""
    f = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (f >> 16) & 1
    r = ((f + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("workers", [0, 333])
def test_wide_values_stay_correctly_rounded(workers):
    """V ~ N(0, 8^2) on the Qwen3-0.6B shape.  The output is the fp32 weighted sum rounded once to bf16 (the
    pages' "bf16 storage, fp32 accumulation"): within the usual tolerance, and nearly every element the
    correctly rounded bf16 of the fp64 oracle's value or one bf16 step from it.  With the weights rounded to
    bf16 as the output product's operand (2^-9 each), 58 % of the elements came out correctly rounded and
    80 % within one step (measured on this test's inputs); with the weights carried in two bf16 parts,
    99.7 % and 99.97 % (the rest: outputs near zero, where fp32 summation error passes one bf16 step)."""
    rng = np.random.default_rng(11)
    lens = rng.integers(512, 4097, 16)
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 256, seed=12, lens=lens)
    vc.mul_(8.0)                            # exact: a power-of-two scale of bf16 values (NaN canaries stay NaN)
    out = run_decode(q, kc, vc, bt, lens_t, 1.0 / math.sqrt(128), num_workers=workers)
    torch.cuda.synchronize()
    want = oracle_of(q, kc, vc, bt, lens_t, 1.0 / math.sqrt(128))
    check_close(out, want, "V ~ N(0, 64)")
    got = out.float().cpu().double().numpy()
    near = float((np.abs(got - want) <= bf16_ulp(want)).mean())
    exact = float((got == bf16_round(want)).mean())
    assert near >= 0.999, f"only {near:.4f} of the elements within one bf16 step of the oracle value"
    assert exact >= 0.97, f"only {exact:.3f} of the elements are the correctly rounded bf16 of the oracle value"


def test_fixed_split_is_bit_reproducible():
    """A fixed split (num_workers > 0) gives the same partial states merged in the same order, so two calls on
    the same inputs give the same bits, whatever ran on the workspace in between."""
    lens = [700, 1500, 33, 4096, 1, 250]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 256, seed=6, lens=lens)
    a = run_decode(q, kc, vc, bt, lens_t, 0.0884, num_workers=333)
    other = [129, 17, 160]
    q2, kc2, vc2, bt2, lens2 = synth(len(other), 0, 14, 2, 64, 16, seed=7, lens=other)
    run_decode(q2, kc2, vc2, bt2, lens2, 0.125)
    b = run_decode(q, kc, vc, bt, lens_t, 0.0884, num_workers=333)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    check_close(a, oracle_of(q, kc, vc, bt, lens_t, 0.0884), "fixed split")


def test_counters_outside_the_fixed_region_after_other_calls():
    """A batch with more than 16384 (sequence, kv head) arrival counters keeps them where earlier, smaller
    calls on the same workspace left partial states; they are cleared before its launch."""
    lens = [700, 1500, 33, 4096, 1, 250]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 16, 8, 128, 256, seed=8, lens=lens)
    run_decode(q, kc, vc, bt, lens_t, 0.0884)
    rng = np.random.default_rng(9)
    many = rng.integers(1, 80, 2100)
    q2, kc2, vc2, bt2, lens2 = synth(len(many), 0, 16, 8, 128, 16, seed=10, lens=many)
    err = err_word()
    for _ in range(2):
        out = run_decode(q2, kc2, vc2, bt2, lens2, 0.0884, err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        check_close(out, oracle_of(q2, kc2, vc2, bt2, lens2, 0.0884), "2100 sequences")
        run_decode(q, kc, vc, bt, lens_t, 0.0884)


# --------------------------------------------------------------------------- closed forms on the GPU
def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """A wait that nothing completes gives up at its time limit with PKV_ERR_WAIT_TIMEOUT (no hang, no
    fault), and the next calls on the device work as before."""
    err = err_word()
    pkv.diag_wait_timeout(err)
    torch.cuda.synchronize()
    assert err.item() == pkv.ERR_WAIT_TIMEOUT
    lens = [1, 40, 300]
    q, kc, vc, bt, lens_t = synth(len(lens), 0, 8, 2, 64, 16, seed=9, lens=lens)
    err.zero_()
    out = run_decode(q, kc, vc, bt, lens_t, 0.125, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    check_close(out, oracle_of(q, kc, vc, bt, lens_t, 0.125), "after the timed-out wait")


def test_worked_example_on_gpu():
    """Lab manual appendix B.1.2 example, zero-padded to D=64, scattered through a shuffled table."""
    D = 64
    q = torch.zeros(1, 2, D); q[0, :, :2] = torch.tensor([1.0, 1.0])
    k = torch.zeros(3, 1, D); k[:, 0, :2] = torch.tensor([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    v = torch.zeros(3, 1, D); v[:, 0, :2] = torch.tensor([[1.0, 0.0], [0.0, 2.0], [1.0, 2.0]])
    NB, bs = 6, 8
    kc = torch.full((NB, bs, 1, D), float("nan")); vc = kc.clone()
    kc[4, :3] = k; vc[4, :3] = v
    bt = torch.tensor([[4]], dtype=torch.int32)
    out = run_decode(q.bfloat16().cuda(), kc.bfloat16().cuda(), vc.bfloat16().cuda(), bt.cuda(),
                     torch.tensor([3], dtype=torch.int32).cuda(), 1 / math.sqrt(2))
    o = out.float().cpu()
    for h in range(2):
        assert abs(o[0, h, 0].item() - 0.75174492) < 4e-3   # bf16 output rounding
        assert abs(o[0, h, 1].item() - 1.50348984) < 8e-3
        assert torch.all(o[0, h, 2:] == 0)


def test_context_one_returns_v_row_exactly():
    q, kc, vc, bt, lens = synth(5, 1, 16, 8, 128, 16, seed=3)
    out = run_decode(q, kc, vc, bt, lens, 0.0884)
    for b in range(5):
        p = bt[b, 0].item()
        want = vc[p, 0].repeat_interleave(2, dim=0)
        assert torch.equal(out[b].view(torch.int16), want.view(torch.int16))


def test_uniform_v_gives_v():
    q, kc, vc, bt, lens = synth(3, 300, 8, 2, 64, 16, seed=4)
    row = torch.randn(2, 64, device="cuda").bfloat16()
    vc[:] = row
    out = run_decode(q, kc, vc, bt, lens, 0.125)
    want = row.float().repeat_interleave(4, dim=0)
    assert (out.float() - want).abs().max().item() <= 1e-2


def test_shared_prefix_equals_duplicated_blocks():
    lens = [100, 120]
    q, kc, vc, bt, lens_t = synth(2, 0, 16, 8, 128, 16, seed=6, lens=lens)
    # make seq 1's first 3 blocks copies of seq 0's, then point its table at seq 0's blocks
    for i in range(3):
        kc[bt[1, i]] = kc[bt[0, i]]
        vc[bt[1, i]] = vc[bt[0, i]]
    dup = run_decode(q, kc, vc, bt, lens_t, 0.0884)
    bt2 = bt.clone()
    bt2[1, :3] = bt[0, :3]
    shared = run_decode(q, kc, vc, bt2, lens_t, 0.0884)
    assert torch.equal(dup.view(torch.int16), shared.view(torch.int16))


def test_zero_and_padding_rows():
    lens = [0, 5, 0]
    q, kc, vc, bt, lens_t = synth(3, 0, 8, 2, 64, 16, seed=9, lens=lens)
    out = run_decode(q, kc, vc, bt, lens_t, 0.125)
    assert torch.all(out[0].float() == 0) and torch.all(out[2].float() == 0)
    check_close(out, oracle_of(q, kc, vc, bt, lens_t, 0.125), "zero rows")


# --------------------------------------------------------------------------- device-side range errors
def test_bad_slot_sets_error_and_writes_nothing_else():
    NB, bs, Hkv, D = 8, 16, 2, 64
    kc = torch.randn(NB, bs, Hkv, D, device="cuda").bfloat16(); vc = torch.randn_like(kc)
    k = torch.randn(3, Hkv, D, device="cuda").bfloat16(); v = torch.randn_like(k)
    before_k, before_v = kc.clone(), vc.clone()
    slots = torch.tensor([NB * bs, -1, -7], dtype=torch.int32, device="cuda")
    err = err_word()
    pkv.kv_store(k, v, slots, kc, vc, err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_SLOT_RANGE
    assert torch.equal(kc, before_k) and torch.equal(vc, before_v)


def test_bad_block_id_sets_error_without_fault():
    q, kc, vc, bt, lens = synth(2, 40, 8, 2, 64, 16, seed=10)
    bt[1, 1] = kc.shape[0] + 100
    err = err_word()
    run_decode(q, kc, vc, bt, lens, 0.125, err=err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_BLOCK_RANGE
    # the context is still healthy
    bt[1, 1] = bt[0, 0]
    run_decode(q, kc, vc, bt, lens, 0.125)
    torch.cuda.synchronize()


def test_context_beyond_limit_sets_error_and_zeros():
    q, kc, vc, bt, lens = synth(2, 40, 8, 2, 64, 16, seed=11)
    err = err_word()
    out = run_decode(q, kc, vc, bt, lens, 0.125, max_ctx=39, err=err)
    torch.cuda.synchronize()
    assert err.item() & pkv.ERR_CONTEXT_RANGE
    assert torch.all(out.float() == 0)


def test_slot_mapping_range_errors():
    bt = torch.tensor([[3, -1], [99, 1]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([40, 3], dtype=torch.int32, device="cuda")
    slots = torch.empty(2, dtype=torch.int32, device="cuda")
    err = err_word()
    pkv.decode_slot_mapping(bt, lens, 16, 10, slots, err)
    torch.cuda.synchronize()
    assert slots.tolist() == [-1, -1]
    assert err.item() & pkv.ERR_CONTEXT_RANGE and err.item() & pkv.ERR_BLOCK_RANGE
