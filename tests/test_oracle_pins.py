"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test fixes the oracle against a value printed on the pages (tests/golden),
a closed form, a library routine (torch's scaled_dot_product_attention in fp64
on contiguous K/V), brute force, or an invariant that a plausible mistake (a
dropped scale, a wrong block index, a wrong GQA head, an off-by-one context
length, a bad merge weight) breaks.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_62_gb300 import workloads as W


# --------------------------------------------------------------------------- helpers
def to_bits(x: np.ndarray) -> np.ndarray:
    """Values exactly representable in bf16 -> uint16 bit patterns."""
    t = torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.from_numpy(np.asarray(x, np.float32))), "value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def rand_bits(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged_from_contiguous(seqs_k, seqs_v, block_size, rng, extra_blocks=3):
    """Place contiguous per-sequence K/V [L, Hkv, D] into a shuffled block pool.

    Block-granular numpy slicing only: logical block i of a sequence is copied
    whole into physical block table[i].  Unused rows are NaN canaries.
    """
    Hkv, D = seqs_k[0].shape[1:]
    nblk = [-(-s.shape[0] // block_size) for s in seqs_k]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB)
    nan = np.uint16(0x7FC0)          # bf16 quiet NaN
    kc = np.full((NB, block_size, Hkv, D), nan, np.uint16)
    vc = np.full((NB, block_size, Hkv, D), nan, np.uint16)
    bt = np.full((len(seqs_k), max(max(nblk), 1)), -1, np.int32)
    cur = 0
    for b, (sk, sv) in enumerate(zip(seqs_k, seqs_v)):
        for i in range(nblk[b]):
            p = perm[cur]
            cur += 1
            bt[b, i] = p
            chunk_k = sk[i * block_size:(i + 1) * block_size]
            kc[p, :chunk_k.shape[0]] = chunk_k
            kc_rows = chunk_k.shape[0]
            vc[p, :kc_rows] = sv[i * block_size:(i + 1) * block_size]
    return kc, vc, bt


def sdpa_reference(q_bits, seqs_k, seqs_v, scale):
    """torch SDPA in fp64 on contiguous K/V, GQA by repeat_interleave."""
    B, Hq, D = q_bits.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = seqs_k[b].shape[0]
        if L == 0:
            continue
        Hkv = seqs_k[b].shape[1]
        q = torch.from_numpy(bits_to_f64(q_bits[b])).view(1, Hq, 1, D)
        k = torch.from_numpy(bits_to_f64(seqs_k[b])).permute(1, 0, 2).unsqueeze(0)
        v = torch.from_numpy(bits_to_f64(seqs_v[b])).permute(1, 0, 2).unsqueeze(0)
        k = k.repeat_interleave(Hq // Hkv, dim=1)
        v = v.repeat_interleave(Hq // Hkv, dim=1)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
        out[b] = o[0, :, 0, :].numpy()
    return out


def random_problem(rng, lens, Hq, Hkv, D, bs):
    seqs_k = [rand_bits(rng, (L, Hkv, D)) for L in lens]
    seqs_v = [rand_bits(rng, (L, Hkv, D)) for L in lens]
    q = rand_bits(rng, (len(lens), Hq, D))
    kc, vc, bt = paged_from_contiguous(seqs_k, seqs_v, bs, rng)
    return q, seqs_k, seqs_v, kc, vc, bt


# --------------------------------------------------------------------------- page values
def test_softmax_pin(golden):
    g = golden("softmax_2_1_0.txt")[""]
    scores = g["scores"][0]
    probs = g["probs"][0]
    tol = g["tol"][0][0]
    # softmax through the oracle: one query, keys chosen so that scale * q.k_j = scores[j]
    D = 2
    q = to_bits(np.array([[[1.0, 0.0]]]))
    k = [to_bits(np.array([[s, 0.0] for s in scores]).reshape(3, 1, D))]
    v = [to_bits(np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]]).reshape(3, 1, D))]  # out = (p0, p1)
    rng = np.random.default_rng(0)
    kc, vc, bt = paged_from_contiguous(k, v, 2, rng)
    out = oracle.paged_decode(q, kc, vc, bt, np.array([3], np.int32), 1.0)
    assert abs(out[0, 0, 0] - probs[0]) < tol
    assert abs(out[0, 0, 1] - probs[1]) < tol
    # the remaining probability is the third one
    assert abs((1 - out[0, 0, 0] - out[0, 0, 1]) - probs[2]) < tol
    assert int(np.argmax([out[0, 0, 0], out[0, 0, 1], 1 - out[0, 0, 0] - out[0, 0, 1]])) == int(g["greedy"][0][0])


@pytest.mark.parametrize("case", ["v_differs", "qkv_same"])
@pytest.mark.parametrize("block_size", [1, 2, 4])
def test_attention_worked_example(golden, case, block_size):
    g = golden("attention_b12.txt")[case]
    q = to_bits(np.array([g["q"][0]]).reshape(1, 1, 2))
    k = to_bits(np.array(g["k"]).reshape(3, 1, 2))
    v = to_bits(np.array(g["v"]).reshape(3, 1, 2))
    scale = 1.0 / math.sqrt(g["scale_inv_sq"][0][0])
    rng = np.random.default_rng(block_size)
    kc, vc, bt = paged_from_contiguous([k], [v], block_size, rng)
    out = oracle.paged_decode(q, kc, vc, bt, np.array([3], np.int32), scale)
    np.testing.assert_allclose(out[0, 0], g["out"][0], atol=g["tol"][0][0], rtol=0)
    # weights: single-token partial states give m_j = s_j, and exp(s_j - M) / sum gives the weights
    ms = [oracle.partial_state(q, kc, vc, bt, 0, 0, scale, j, j + 1)[0] for j in range(3)]
    M = max(ms)
    w = np.exp(np.array(ms) - M)
    w /= w.sum()
    np.testing.assert_allclose(w, g["weights"][0], atol=g["tol"][0][0], rtol=0)
    if "scores" in g:
        np.testing.assert_allclose(ms, g["scores"][0], atol=g["scores_tol"][0][0], rtol=0)


def test_attention_worked_example_embedded_d64(golden):
    """The same example zero-padded to head_dim 64 inside a 2-head GQA group."""
    g = golden("attention_b12.txt")["v_differs"]
    D = 64
    q = np.zeros((1, 2, D)); q[0, :, :2] = g["q"][0]
    k = np.zeros((3, 1, D)); k[:, 0, :2] = np.array(g["k"])
    v = np.zeros((3, 1, D)); v[:, 0, :2] = np.array(g["v"])
    rng = np.random.default_rng(7)
    kc, vc, bt = paged_from_contiguous([to_bits(k)], [to_bits(v)], 8, rng)
    out = oracle.paged_decode(to_bits(q), kc, vc, bt, np.array([3], np.int32), 1 / math.sqrt(2))
    for h in range(2):
        np.testing.assert_allclose(out[0, h, :2], g["out"][0], atol=g["tol"][0][0], rtol=0)
        assert np.all(out[0, h, 2:] == 0)


def test_slot_teaching_example(golden):
    g = golden("slots_b23.txt")[""]
    bs = int(g["block_size"][0][0])
    row = np.array(g["block_table"][0], np.int32)
    for pos, want in zip(g["positions"][0], g["slots"][0]):
        assert oracle.slot_of(row, bs, int(pos)) == int(want)


def test_block_count_boundaries(golden):
    g = golden("slots_b23.txt")[""]
    bs = int(g["count_block_size"][0][0])
    row = np.array([7, 3], np.int32)
    for n, nblocks in zip(g["count_lengths"][0], g["count_blocks"][0]):
        last = oracle.slot_of(row, bs, int(n) - 1)
        used_block = row[int(nblocks) - 1]
        assert last // bs == used_block
        # every position of the sequence falls in the first `nblocks` table entries
        blocks_touched = {oracle.slot_of(row, bs, p) // bs for p in range(int(n))}
        assert blocks_touched == set(int(x) for x in row[:int(nblocks)])


def test_decode_slots_page_example(golden):
    g = golden("slots_decode_s44.txt")[""]
    bs = int(g["block_size"][0][0])
    bt = np.array(g["block_tables"], np.int32)
    ctx = np.array(g["context_lens"][0], np.int32)
    got = oracle.decode_slot_mapping(bt, ctx, bs)
    assert got.tolist() == [int(x) for x in g["slot_mapping"][0]]
    # padding rows (beyond the batch, or context_len 0) get -1
    got = oracle.decode_slot_mapping(bt, np.array([431, 0], np.int32), bs, num_tokens=4)
    assert got.tolist() == [430, -1, -1, -1]


def test_prefill_slots_page_example(golden):
    g = golden("slots_prefill_s35.txt")[""]
    bs = int(g["block_size"][0][0])
    row5 = np.array(g["seq5_block_table"][0], np.int32)
    p0 = int(g["seq5_first_position"][0][0])
    n5 = int(g["seq5_count"][0][0])
    slots5 = [oracle.slot_of(row5, bs, p) for p in range(p0, p0 + n5)]
    assert slots5[:10] == [int(x) for x in g["seq5_first_slots"][0]]
    assert slots5[-1] == int(g["seq5_last_slot"][0][0])
    row4 = np.array(g["seq4_block_table"][0], np.int32)
    n4 = int(g["seq4_count"][0][0])
    slots4 = [oracle.slot_of(row4, bs, p) for p in range(n4)]
    assert slots4 == list(range(n4)) and slots4[-1] == int(g["seq4_last_slot"][0][0])


# --------------------------------------------------------------------------- library routine / brute force
@pytest.mark.parametrize("D,Hq,Hkv,bs", [(64, 4, 2, 16), (128, 16, 8, 8), (64, 14, 2, 32), (128, 8, 2, 16),
                                         (64, 4, 4, 8)])
def test_paged_equals_sdpa_contiguous(D, Hq, Hkv, bs):
    rng = np.random.default_rng(D * 1000 + Hq * 10 + bs)
    lens = [1, 15, 16, 17, 40, 0, 129]
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, Hq, Hkv, D, bs)
    scale = 1 / math.sqrt(D)
    got = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), scale, nthreads=3)
    want = sdpa_reference(q, sk, sv, scale)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-10)
    assert np.all(got[lens.index(0)] == 0)


def test_identity_table_is_contiguous():
    """Block table [0, 1, 2, ...]: the pool *is* the contiguous sequence."""
    rng = np.random.default_rng(3)
    L, Hkv, D, bs, Hq = 100, 2, 64, 16, 4
    nb = -(-L // bs)
    kc = rand_bits(rng, (nb, bs, Hkv, D))
    vc = rand_bits(rng, (nb, bs, Hkv, D))
    q = rand_bits(rng, (1, Hq, D))
    bt = np.arange(nb, dtype=np.int32).reshape(1, nb)
    got = oracle.paged_decode(q, kc, vc, bt, np.array([L], np.int32), 0.125)
    want = sdpa_reference(q, [kc.reshape(-1, Hkv, D)[:L]], [vc.reshape(-1, Hkv, D)[:L]], 0.125)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-10)


def test_workload_tiny_against_sdpa():
    """The tiny workload from the generator, after the oracle store, against SDPA."""
    wl = W.make("tiny", "cpu")
    lay = wl.layers[0]
    kc, vc = W.bits(lay.k_cache), W.bits(lay.v_cache)
    bt = wl.block_tables.numpy()
    lens = wl.context_lens.numpy()
    slots = oracle.decode_slot_mapping(bt, lens, wl.spec.block_size, wl.num_tokens)
    for t in wl.skip_tokens:
        slots[t] = -1
    oracle.kv_store(W.bits(lay.k_new), W.bits(lay.v_new), slots, kc, vc)
    q = W.bits(lay.q)
    got = oracle.paged_decode(q, kc, vc, bt, lens, wl.scale)
    assert np.isfinite(got).all(), "a canary row was read: store or gather is wrong"
    # contiguous copy by whole blocks (torch indexing), truncated to L
    seqs_k, seqs_v = [], []
    for b, L in enumerate(lens):
        nb = -(-int(L) // wl.spec.block_size)
        ids = torch.from_numpy(bt[b, :nb].astype(np.int64))
        seqs_k.append(torch.from_numpy(kc.view(np.int16))[ids].reshape(-1, *kc.shape[2:])[:L].numpy().view(np.uint16))
        seqs_v.append(torch.from_numpy(vc.view(np.int16))[ids].reshape(-1, *vc.shape[2:])[:L].numpy().view(np.uint16))
    want = sdpa_reference(q, seqs_k, seqs_v, wl.scale)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-10)


def test_decode_slots_brute_force():
    rng = np.random.default_rng(11)
    for bs in (8, 16, 256):
        B, mb = 9, 6
        bt = rng.integers(0, 500, size=(B, mb)).astype(np.int32)
        lens = rng.integers(0, mb * bs + 1, size=B).astype(np.int32)
        got = oracle.decode_slot_mapping(bt, lens, bs, num_tokens=B + 3)
        for t in range(B + 3):
            if t >= B or lens[t] == 0:
                assert got[t] == -1
            else:
                pos = int(lens[t]) - 1
                # brute force: walk positions block by block
                blk, off = 0, pos
                while off >= bs:
                    blk, off = blk + 1, off - bs
                assert got[t] == bt[t, blk] * bs + off


# --------------------------------------------------------------------------- closed forms and invariants
def test_uniform_v_gives_v():
    rng = np.random.default_rng(5)
    L, Hkv, D, Hq, bs = 77, 2, 64, 4, 16
    k = rand_bits(rng, (L, Hkv, D))
    row = rand_bits(rng, (1, Hkv, D))
    v = np.repeat(row, L, axis=0)
    q = rand_bits(rng, (1, Hq, D))
    kc, vc, bt = paged_from_contiguous([k], [v], bs, rng)
    got = oracle.paged_decode(q, kc, vc, bt, np.array([L], np.int32), 0.125)
    for h in range(Hq):
        np.testing.assert_allclose(got[0, h], bits_to_f64(row[0, h // 2]), rtol=1e-14, atol=1e-15)


def test_context_one_gives_v_row_exactly():
    rng = np.random.default_rng(6)
    k = rand_bits(rng, (1, 2, 128))
    v = rand_bits(rng, (1, 2, 128))
    q = rand_bits(rng, (1, 16, 128))
    kc, vc, bt = paged_from_contiguous([k], [v], 16, rng)
    got = oracle.paged_decode(q, kc, vc, bt, np.array([1], np.int32), 0.088)
    for h in range(16):
        assert np.array_equal(got[0, h], bits_to_f64(v[0, h // 8]))


@pytest.mark.parametrize("bs,lens", [(16, [15, 16, 17]), (256, [255, 256, 257])])
def test_block_boundary_contexts(bs, lens):
    rng = np.random.default_rng(bs)
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, 4, 2, 64, bs)
    got = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), 0.125)
    want = sdpa_reference(q, sk, sv, 0.125)
    np.testing.assert_allclose(got, want, atol=1e-12, rtol=1e-10)


def test_permuting_physical_blocks_changes_nothing():
    rng = np.random.default_rng(8)
    lens = [33, 70, 5]
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, 4, 2, 64, 16)
    base = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), 0.1)
    NB = kc.shape[0]
    perm = rng.permutation(NB)          # new position of old block p is perm[p]
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    moved = oracle.paged_decode(q, kc2, vc2, bt2, np.array(lens, np.int32), 0.1)
    assert np.array_equal(base, moved)


def test_gqa_equals_repeat_interleave_mha():
    rng = np.random.default_rng(9)
    lens = [20, 41]
    Hq, Hkv, D = 8, 2, 64
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, Hq, Hkv, D, 16)
    gqa = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), 0.125)
    kc_m = np.repeat(kc, Hq // Hkv, axis=2)
    vc_m = np.repeat(vc, Hq // Hkv, axis=2)
    mha = oracle.paged_decode(q, kc_m, vc_m, bt, np.array(lens, np.int32), 0.125)
    assert np.array_equal(gqa, mha)


def test_shared_prefix_equals_duplicated_blocks():
    rng = np.random.default_rng(10)
    Hkv, D, bs, Hq = 2, 64, 16, 4
    prefix_k = rand_bits(rng, (2 * bs, Hkv, D))
    prefix_v = rand_bits(rng, (2 * bs, Hkv, D))
    tails = [(rand_bits(rng, (n, Hkv, D)), rand_bits(rng, (n, Hkv, D))) for n in (5, 19)]
    seqs_k = [np.concatenate([prefix_k, t[0]]) for t in tails]
    seqs_v = [np.concatenate([prefix_v, t[1]]) for t in tails]
    lens = np.array([s.shape[0] for s in seqs_k], np.int32)
    q = rand_bits(rng, (2, Hq, D))
    # duplicated: every sequence has private copies of the prefix blocks
    kc, vc, bt = paged_from_contiguous(seqs_k, seqs_v, bs, rng)
    dup = oracle.paged_decode(q, kc, vc, bt, lens, 0.125)
    # shared: point sequence 1's first two table entries at sequence 0's blocks
    bt_sh = bt.copy()
    bt_sh[1, :2] = bt[0, :2]
    kc_sh, vc_sh = kc.copy(), vc.copy()
    nan = np.uint16(0x7FC0)
    kc_sh[bt[1, :2]] = nan       # the now-unreferenced copies become canaries
    vc_sh[bt[1, :2]] = nan
    shared = oracle.paged_decode(q, kc_sh, vc_sh, bt_sh, lens, 0.125)
    assert np.array_equal(dup, shared)


def test_scale_multiplies_the_dot_product():
    rng = np.random.default_rng(12)
    lens = [30]
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, 4, 2, 64, 16)
    a = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), 0.25)
    q2 = to_bits(2.0 * bits_to_f64(q))
    b = oracle.paged_decode(q2, kc, vc, bt, np.array(lens, np.int32), 0.125)
    assert np.array_equal(a, b)


def test_merge_of_partial_states_equals_whole():
    rng = np.random.default_rng(13)
    lens = [203]
    q, sk, sv, kc, vc, bt = random_problem(rng, lens, 4, 2, 64, 16)
    whole = oracle.paged_decode(q, kc, vc, bt, np.array(lens, np.int32), 0.125)
    for cuts in ([0, 203], [0, 1, 203], [0, 16, 100, 101, 203], [0, 50, 50, 203]):
        for h in range(4):
            st = [oracle.partial_state(q, kc, vc, bt, 0, h, 0.125, a, b) for a, b in zip(cuts[:-1], cuts[1:])]
            ms, ls, accs = zip(*st)
            merged = oracle.merge_states(ms, ls, np.stack(accs))
            np.testing.assert_allclose(merged, whole[0, h], atol=1e-13, rtol=1e-11)
            rev = oracle.merge_states(ms[::-1], ls[::-1], np.stack(accs[::-1]))
            np.testing.assert_allclose(rev, whole[0, h], atol=1e-13, rtol=1e-11)
    # every state empty -> zeros
    assert np.all(oracle.merge_states([-np.inf], [0.0], np.zeros((1, 64))) == 0)


def test_kv_store_bit_copy_and_skip():
    rng = np.random.default_rng(14)
    NB, bs, Hkv, D, T = 10, 8, 2, 64, 6
    kc = rand_bits(rng, (NB, bs, Hkv, D)); vc = rand_bits(rng, (NB, bs, Hkv, D))
    k = rand_bits(rng, (T, Hkv, D)); v = rand_bits(rng, (T, Hkv, D))
    slots = np.array([3, -1, 79, 40, -1, 0], np.int32)
    kc0, vc0 = kc.copy(), vc.copy()
    oracle.kv_store(k, v, slots, kc, vc)
    want_k, want_v = kc0.reshape(NB * bs, Hkv, D).copy(), vc0.reshape(NB * bs, Hkv, D).copy()
    keep = slots >= 0
    want_k[slots[keep]] = k[keep]
    want_v[slots[keep]] = v[keep]
    assert np.array_equal(kc.reshape(NB * bs, Hkv, D), want_k)
    assert np.array_equal(vc.reshape(NB * bs, Hkv, D), want_v)
    with pytest.raises(oracle.OracleError):
        oracle.kv_store(k, v, np.array([80, -1, -1, -1, -1, -1], np.int32), kc, vc)


def test_copy_blocks_bit_copy_and_copy_on_write_semantics():
    """Block copies (copy-on-write, nano-vllm KV-cache post §2.2): numpy whole-block assignment decides
    the bytes; a sequence whose table points at the copy attends exactly like one pointing at the
    original; src == dst changes nothing; a bad id is refused while the other pairs still apply."""
    rng = np.random.default_rng(15)
    NB, bs, Hkv, D = 12, 8, 2, 64
    kc = rand_bits(rng, (NB, bs, Hkv, D)); vc = rand_bits(rng, (NB, bs, Hkv, D))
    kc0, vc0 = kc.copy(), vc.copy()
    pairs = np.array([[3, 7], [5, 5], [0, 11]], np.int32)
    oracle.copy_blocks(kc, vc, pairs)
    want_k, want_v = kc0.copy(), vc0.copy()
    want_k[[7, 11]] = kc0[[3, 0]]
    want_v[[7, 11]] = vc0[[3, 0]]
    assert np.array_equal(kc, want_k) and np.array_equal(vc, want_v)
    # attention through [..., 3] equals attention through [..., 7] bit for bit
    q = rand_bits(rng, (1, 4, D))
    L = np.array([2 * bs + 5], np.int32)
    a = oracle.paged_decode(q, kc, vc, np.array([[1, 2, 3]], np.int32), L, 0.125)
    b = oracle.paged_decode(q, kc, vc, np.array([[1, 2, 7]], np.int32), L, 0.125)
    assert np.array_equal(a, b)
    kc1 = kc.copy()
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(kc, vc, np.array([[2, 12], [4, 9]], np.int32))
    assert np.array_equal(kc[9], kc1[4]) and np.array_equal(np.delete(kc, 9, 0), np.delete(kc1, 9, 0))


def test_e4m3_codes_are_the_ocp_format():
    """Published constants of OCP E4M3 ("float8_e4m3fn"): 0x7E = 448 (largest), 0x08 = 2^-6 (smallest
    normal), 0x01 = 2^-9 (smallest subnormal), 0x38 = 1, 0x7F / 0xFF NaN, no infinities; the 127
    non-negative finite codes increase strictly; encode(decode(c)) == c for every finite code."""
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0 and v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x00] == 0.0 and np.signbit(v[0x80])
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isfinite(np.delete(v, [0x7F, 0xFF])).all()
    assert np.all(np.diff(v[:0x7F]) > 0)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(v[finite].astype(np.float32)), finite)


def test_e4m3_encode_is_torchs_rounding_in_range_and_saturates_beyond():
    """In range the oracle's rounding equals torch's float8_e4m3fn cast (a library routine), ties
    included; beyond 448 it saturates to +-448 (the GPU conversion's satfinite mode), where torch's
    cast gives NaN from 464 on."""
    rng = np.random.default_rng(16)
    x = np.concatenate([(rng.standard_normal(100000) * 40).astype(np.float32),
                        (rng.standard_normal(20000) * 2.0 ** -8).astype(np.float32),
                        np.array([1.0625, 1.1875, -1.0625, 2 ** -10, 3 * 2 ** -10, 272, 304, 447.9, 448],
                                 np.float32)])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), want)
    big = np.array([448.5, 463.9, 464.0, 1e9, -500.0, np.inf, -np.inf], np.float32)
    assert oracle.e4m3_encode(big).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]


def test_kv_store_fp8_quantises_by_head_scale():
    """Each stored code is torch's float8 cast of the binary32 quotient x / scale[kv head]; slot -1
    writes nothing; a row is written whole."""
    rng = np.random.default_rng(17)
    NB, bs, Hkv, D, T = 6, 8, 2, 64, 5
    kc = rng.integers(0, 255, (NB, bs, Hkv, D), dtype=np.uint8); vc = kc.copy()
    k = rand_bits(rng, (T, Hkv, D)); v = rand_bits(rng, (T, Hkv, D))
    ks = np.array([0.01, 0.75], np.float32); vs = np.array([0.3, 2.0 ** -3], np.float32)
    slots = np.array([3, -1, 47, 12, 0], np.int32)
    kc0, vc0 = kc.copy(), vc.copy()
    oracle.kv_store_fp8(k, v, slots, kc, vc, ks, vs)
    f32 = lambda b: torch.from_numpy(b.astype(np.int32) << 16).view(torch.float32)
    qk = (f32(k) / torch.from_numpy(ks).view(1, Hkv, 1)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    qv = (f32(v) / torch.from_numpy(vs).view(1, Hkv, 1)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    want_k, want_v = kc0.reshape(NB * bs, Hkv, D).copy(), vc0.reshape(NB * bs, Hkv, D).copy()
    keep = slots >= 0
    want_k[slots[keep]] = qk[keep]
    want_v[slots[keep]] = qv[keep]
    assert np.array_equal(kc.reshape(NB * bs, Hkv, D), want_k)
    assert np.array_equal(vc.reshape(NB * bs, Hkv, D), want_v)


def test_fp8_decode_is_attention_over_the_dequantised_cache():
    """With power-of-two scales every dequantised value is exact in bf16, so the fp8 decode must equal
    the bf16 oracle on the dequantised caches; doubling k_scale while halving the attention scale changes
    nothing, doubling v_scale doubles the output -- exactly."""
    rng = np.random.default_rng(18)
    NB, bs, Hkv, D, B, G = 9, 16, 2, 64, 3, 4
    kc = rng.integers(0, 0x7F, (NB, bs, Hkv, D), dtype=np.uint8) | (rng.integers(0, 2, (NB, bs, Hkv, D),
                                                                                  dtype=np.uint8) << 7)
    vc = rng.integers(0, 0x7F, (NB, bs, Hkv, D), dtype=np.uint8)
    kc[kc == 0xFF] = 0xFE
    ks = np.array([2.0 ** -4, 0.5], np.float32); vs = np.array([1.0, 2.0 ** -2], np.float32)
    q = rand_bits(rng, (B, G * Hkv, D))
    bt = rng.permutation(NB)[:B * 3].reshape(B, 3).astype(np.int32)
    lens = np.array([40, 1, 33], np.int32)
    got = oracle.paged_decode_fp8(q, kc, vc, ks, vs, bt, lens, 0.125)
    deq = lambda c, s: torch.from_numpy((oracle.e4m3_decode(c) * s.reshape(1, 1, Hkv, 1)).astype(np.float32))
    kb = deq(kc, ks).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    vb = deq(vc, vs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.e4m3_decode(kc) * ks.reshape(1, 1, Hkv, 1),
                          torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).double().numpy())
    want = oracle.paged_decode(q, kb, vb, bt, lens, 0.125)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
    assert np.array_equal(oracle.paged_decode_fp8(q, kc, vc, ks * 2, vs, bt, lens, 0.0625), got)
    assert np.array_equal(oracle.paged_decode_fp8(q, kc, vc, ks, vs * 2, bt, lens, 0.125), 2 * got)


@pytest.mark.parametrize("Hq,Hkv,D,bs", [(4, 2, 64, 16), (8, 8, 128, 8)])
def test_paged_attention_is_causal_sdpa_over_the_sequence(Hq, Hkv, D, bs):
    """Chunked prefill / mixed batch: the last n tokens of each sequence attend causally over all its
    L cached tokens.  Against torch's scaled_dot_product_attention (fp64, is_causal) run on the whole
    contiguous sequence with every token as a query, keeping the last n query rows; n = L (a whole
    prefill), 1 < n < L (a chunk after a cached prefix) and n = 1 (a decode) are all in the batch."""
    rng = np.random.default_rng(Hq + D)
    lens = [37, 16, 50, 1, 29]
    news = [37, 5, 1, 1, 12]
    seqs_k = [rand_bits(rng, (L, Hkv, D)) for L in lens]
    seqs_v = [rand_bits(rng, (L, Hkv, D)) for L in lens]
    kc, vc, bt = paged_from_contiguous(seqs_k, seqs_v, bs, rng)
    cu = np.concatenate([[0], np.cumsum(news)]).astype(np.int32)
    qs = [rand_bits(rng, (L, Hq, D)) for L in lens]            # a query for every token; the last n are used
    q = np.concatenate([qq[L - n:] for qq, L, n in zip(qs, lens, news)])
    got = oracle.paged_attention(q, kc, vc, bt, cu, np.array(lens, np.int32), 0.125)
    for b, (L, n) in enumerate(zip(lens, news)):
        qq = torch.from_numpy(bits_to_f64(qs[b])).permute(1, 0, 2).unsqueeze(0)          # [1, Hq, L, D]
        k = torch.from_numpy(bits_to_f64(seqs_k[b])).permute(1, 0, 2).unsqueeze(0).repeat_interleave(Hq // Hkv, 1)
        v = torch.from_numpy(bits_to_f64(seqs_v[b])).permute(1, 0, 2).unsqueeze(0).repeat_interleave(Hq // Hkv, 1)
        want = torch.nn.functional.scaled_dot_product_attention(qq, k, v, scale=0.125, is_causal=True)
        want = want[0, :, L - n:, :].permute(1, 0, 2).numpy()                            # [n, Hq, D]
        np.testing.assert_allclose(got[cu[b]:cu[b + 1]], want, rtol=1e-10, atol=1e-12)
    # one new token per sequence is the decode definition
    ones = np.arange(len(lens) + 1, dtype=np.int32)
    qd = rand_bits(rng, (len(lens), Hq, D))
    assert np.array_equal(oracle.paged_attention(qd, kc, vc, bt, ones, np.array(lens, np.int32), 0.125),
                          oracle.paged_decode(qd, kc, vc, bt, np.array(lens, np.int32), 0.125))
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(q[:2], kc, vc, bt, np.array([0, 2, 2, 2, 2, 2], np.int32),
                               np.array([1, 1, 1, 1, 1], np.int32), 0.125)   # 2 new tokens in a length-1 sequence


def test_generator_structure():
    """Generator invariants the parity tests rely on (no arithmetic under test involved)."""
    for name in ("tiny", "qwen25_0p5b"):
        wl = W.make(name, "cpu")
        bt = wl.block_tables.numpy()
        lens = wl.context_lens.numpy()
        used = bt[bt >= 0]
        assert used.max() < wl.num_blocks and len(set(used.tolist())) == used.size  # no sharing here
        assert wl.layers[0].k_cache.shape == (wl.num_blocks, wl.spec.block_size, wl.spec.num_kv_heads,
                                               wl.spec.head_dim)
        assert (lens >= 1).all()
    assert W.make("tiny").context_lens.tolist() == [1, 15, 17, 40]
    a, b = W.make("qwen25_0p5b"), W.make("qwen25_0p5b")
    assert torch.equal(a.layers[0].q.view(torch.int16), b.layers[0].q.view(torch.int16))
