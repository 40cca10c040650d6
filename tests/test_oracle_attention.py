"""Pins for the oracle's decode attention (CPU only).

What fixes the result independently of the oracle's own code:
  * dense attention on a contiguous layout, written with numpy (different
    code path: array slicing and matmul instead of the block-table loop);
  * a pure-Python brute force on tiny cases;
  * closed forms: L = 1 gives V_0 exactly; q = 0 or equal keys give mean(V);
    a key c*q with large c gives that token's V;
  * invariants the pages state: physical placement is arbitrary (permuting
    blocks with the table changes nothing), shared blocks read the same as
    copies, entries past cdiv(L, block_size) are never read, and query head
    h reads KV head h // G;
  * planted mistakes (dropped last partial block, off-by-one offset inside a
    block, wrong GQA grouping) are caught by the dense comparison.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_69_gb300 import inputs


def _problem(wl):
    return oracle.Problem(wl.q, oracle.DTYPE_CODES[wl.q_dtype], wl.k_cache, wl.v_cache,
                          oracle.DTYPE_CODES[wl.kv_dtype], wl.block_tables, wl.seq_lens,
                          wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                          wl.num_blocks, wl.scale, wl.k_scale, wl.v_scale)


def _written(wl):
    """Apply the workload's setup and step writes with the oracle (host copy)."""
    k = oracle.as_raw(wl.k_cache).copy()
    v = oracle.as_raw(wl.v_cache).copy()
    kvd, sd = oracle.DTYPE_CODES[wl.kv_dtype], oracle.DTYPE_CODES[wl.src_dtype]
    args = (wl.num_kv_heads, wl.head_dim, wl.block_size, wl.num_blocks)
    for kind, payload in wl.setup:
        if kind == "copy":
            oracle.copy_blocks(k, v, kvd, oracle.as_raw(payload), *args)
        else:
            oracle.reshape_and_cache(k, v, kvd, oracle.as_raw(payload.key), oracle.as_raw(payload.value),
                                     sd, oracle.as_raw(payload.slots), *args, wl.k_scale, wl.v_scale)
    oracle.reshape_and_cache(k, v, kvd, oracle.as_raw(wl.new_key), oracle.as_raw(wl.new_value), sd,
                             oracle.as_raw(wl.slot_mapping), *args, wl.k_scale, wl.v_scale)
    return k, v


def _dense_from_contiguous(q, K, V, scale, G):
    """numpy dense attention. q [Hq, D]; K, V [L, Hkv, D] contiguous."""
    Kr = np.repeat(K, G, axis=1)            # [L, Hq, D]
    Vr = np.repeat(V, G, axis=1)
    s = np.einsum("hd,lhd->hl", q, Kr) * scale
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return np.einsum("hl,lhd->hd", p, Vr)


def _contiguous_workload(seq_lens, Hq, Hkv, D, bs, dtype, seed):
    """A workload whose block tables are the identity, so sequence i's tokens
    are contiguous rows of the pool starting at its first block."""
    wl = inputs.make_random(seq_lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                            block_size=bs, kv_dtype=dtype, seed=seed)
    nblk = [-(-L // bs) for L in seq_lens]
    start = np.cumsum([0] + nblk[:-1])
    bt = wl.block_tables.clone()
    for i, n in enumerate(nblk):
        bt[i, :n] = torch.arange(start[i], start[i] + n, dtype=torch.int32)
    # rebuild the pool through the new tables from the old one's contents
    k, v = _written(wl)
    old_bt = wl.block_tables.numpy()
    k2 = np.full_like(k, 0); v2 = np.full_like(v, 0)
    for i, n in enumerate(nblk):
        for j in range(n):
            k2[start[i] + j] = k[old_bt[i, j]]
            v2[start[i] + j] = v[old_bt[i, j]]
    return wl, bt, k2, v2


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_oracle_matches_dense_contiguous(dtype):
    lens = [1, 15, 16, 17, 33, 64, 100]
    Hq, Hkv, D, bs = 8, 2, 64, 16
    wl, bt, k2, v2 = _contiguous_workload(lens, Hq, Hkv, D, bs, dtype, seed=11)
    wl.block_tables = bt
    p = oracle.Problem(wl.q, oracle.DTYPE_CODES[wl.q_dtype], k2, v2, oracle.DTYPE_CODES[dtype],
                       bt, wl.seq_lens, Hq, Hkv, D, bs, wl.num_blocks, wl.scale)
    got = oracle.decode(p)
    qd = oracle.decode_array(oracle.as_raw(wl.q), oracle.DTYPE_CODES[wl.q_dtype])
    kd = oracle.decode_array(k2, oracle.DTYPE_CODES[dtype]).reshape(-1, Hkv, D)
    vd = oracle.decode_array(v2, oracle.DTYPE_CODES[dtype]).reshape(-1, Hkv, D)
    start = 0
    for i, L in enumerate(lens):
        want = _dense_from_contiguous(qd[i], kd[start * 1: start + L], vd[start: start + L],
                                      float(np.float32(wl.scale)), Hq // Hkv)
        np.testing.assert_allclose(got[i], want, rtol=1e-12, atol=1e-13)
        start += -(-L // bs) * bs


def _pure_python(q, K, V, scale):
    """Brute force with Python floats. q [D]; K, V lists of [D]."""
    s = [scale * sum(a * b for a, b in zip(q, k)) for k in K]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    Z = sum(e)
    return [sum(e[t] / Z * V[t][d] for t in range(len(K))) for d in range(len(q))]


@pytest.mark.parametrize("bs", [8, 16])
def test_oracle_matches_brute_force_tiny(bs):
    lens = [1, 2, bs - 1, bs, bs + 1]
    Hq, Hkv, D = 4, 2, 8
    wl = inputs.make_random(lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                            kv_dtype="f32", seed=3, spare_blocks=5)
    k, v = _written(wl)
    got = oracle.decode(oracle.Problem(wl.q, oracle.F32, k, v, oracle.F32, wl.block_tables,
                                       wl.seq_lens, Hq, Hkv, D, bs, wl.num_blocks, wl.scale))
    bt = wl.block_tables.numpy()
    qn = wl.q.numpy().astype(np.float64)
    for i, L in enumerate(lens):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            K = [[float(x) for x in k[bt[i, t // bs], t % bs, g]] for t in range(L)]
            V = [[float(x) for x in v[bt[i, t // bs], t % bs, g]] for t in range(L)]
            want = _pure_python(list(qn[i, h]), K, V, float(np.float32(wl.scale)))
            np.testing.assert_allclose(got[i, h], want, rtol=1e-12, atol=1e-14)


def test_closed_form_single_token_is_v0_exactly():
    wl = inputs.make_random([1, 1, 1], num_q_heads=4, num_kv_heads=1, head_dim=16, block_size=16,
                            kv_dtype="bf16", seed=4)
    k, v = _written(wl)
    got = oracle.decode(oracle.Problem(wl.q, oracle.BF16, k, v, oracle.BF16, wl.block_tables,
                                       wl.seq_lens, 4, 1, 16, 16, wl.num_blocks, wl.scale))
    vd = oracle.decode_array(v, oracle.BF16)
    bt = wl.block_tables.numpy()
    for i in range(3):
        for h in range(4):
            assert np.array_equal(got[i, h], vd[bt[i, 0], 0, 0])


def test_closed_form_zero_query_gives_mean_v():
    wl = inputs.make_random([37, 5], num_q_heads=2, num_kv_heads=2, head_dim=32, block_size=8,
                            kv_dtype="f32", seed=5)
    k, v = _written(wl)
    q = np.zeros_like(oracle.as_raw(wl.q))
    got = oracle.decode(oracle.Problem(q, oracle.F32, k, v, oracle.F32, wl.block_tables,
                                       wl.seq_lens, 2, 2, 32, 8, wl.num_blocks, wl.scale))
    bt = wl.block_tables.numpy()
    for i, L in enumerate([37, 5]):
        for h in range(2):
            rows = np.stack([v[bt[i, t // 8], t % 8, h] for t in range(L)]).astype(np.float64)
            np.testing.assert_allclose(got[i, h], rows.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_closed_form_equal_keys_give_mean_v():
    wl = inputs.make_random([20], num_q_heads=1, num_kv_heads=1, head_dim=16, block_size=8,
                            kv_dtype="f32", seed=6)
    k, v = _written(wl)
    bt = wl.block_tables.numpy()
    for t in range(20):
        k[bt[0, t // 8], t % 8, 0] = k[bt[0, 0], 0, 0]
    got = oracle.decode(oracle.Problem(wl.q, oracle.F32, k, v, oracle.F32, wl.block_tables,
                                       wl.seq_lens, 1, 1, 16, 8, wl.num_blocks, wl.scale))
    rows = np.stack([v[bt[0, t // 8], t % 8, 0] for t in range(20)]).astype(np.float64)
    np.testing.assert_allclose(got[0, 0], rows.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_closed_form_planted_key_selects_its_value():
    wl = inputs.make_random([50], num_q_heads=1, num_kv_heads=1, head_dim=16, block_size=16,
                            kv_dtype="f32", seed=7)
    k, v = _written(wl)
    bt = wl.block_tables.numpy()
    t_star = 29
    q = oracle.as_raw(wl.q)
    k[bt[0, t_star // 16], t_star % 16, 0] = 200.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    got = oracle.decode(oracle.Problem(q, oracle.F32, k, v, oracle.F32, wl.block_tables,
                                       wl.seq_lens, 1, 1, 16, 16, wl.num_blocks, wl.scale))
    np.testing.assert_allclose(got[0, 0], v[bt[0, t_star // 16], t_star % 16, 0], rtol=0, atol=1e-12)


def test_invariant_block_permutation():
    wl = inputs.make_random([3, 16, 17, 45, 70], num_q_heads=6, num_kv_heads=3, head_dim=32,
                            block_size=16, kv_dtype="f16", seed=8, spare_blocks=9)
    k, v = _written(wl)
    base = oracle.decode(_problem_raw(wl, k, v, wl.block_tables))
    perm = np.random.default_rng(0).permutation(wl.num_blocks)     # new id of old block b
    k2 = np.empty_like(k); v2 = np.empty_like(v)
    k2[perm] = k; v2[perm] = v
    bt = wl.block_tables.numpy().copy()
    for i, L in enumerate(wl.seq_lens.tolist()):
        n = -(-L // 16)
        bt[i, :n] = perm[bt[i, :n]]
    moved = oracle.decode(_problem_raw(wl, k2, v2, torch.from_numpy(bt)))
    assert np.array_equal(base, moved)


def _problem_raw(wl, k, v, bt):
    return oracle.Problem(wl.q, oracle.DTYPE_CODES[wl.q_dtype], k, v, oracle.DTYPE_CODES[wl.kv_dtype],
                          bt, wl.seq_lens, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                          wl.block_size, wl.num_blocks, wl.scale, wl.k_scale, wl.v_scale)


def test_invariant_shared_blocks_equal_copies():
    """Aliased table entries (ref_cnt > 1) read exactly like duplicated blocks."""
    wl = inputs.prefix_share_fp16(prompt_len=40, num_prompts=2, branches=4, max_div=20,
                                  num_q_heads=4, num_kv_heads=2, head_dim=32)
    k, v = _written(wl)
    shared = oracle.decode(_problem_raw(wl, k, v, wl.block_tables))
    # give every sequence private copies of all its blocks in fresh pool space
    bt = wl.block_tables.numpy().copy()
    lens = wl.seq_lens.tolist()
    need = sum(-(-L // 16) for L in lens)
    NB2 = wl.num_blocks + need
    k2 = np.concatenate([k, np.zeros((need,) + k.shape[1:], k.dtype)])
    v2 = np.concatenate([v, np.zeros((need,) + v.shape[1:], v.dtype)])
    nxt = wl.num_blocks
    for i, L in enumerate(lens):
        for j in range(-(-L // 16)):
            k2[nxt] = k[bt[i, j]]; v2[nxt] = v[bt[i, j]]
            bt[i, j] = nxt; nxt += 1
    p = oracle.Problem(wl.q, oracle.F16, k2, v2, oracle.F16, bt, wl.seq_lens, 4, 2, 32, 16, NB2,
                       wl.scale)
    assert np.array_equal(shared, oracle.decode(p))
    # and branches of one prompt really do alias blocks
    assert (bt is not None) and len(set(wl.block_tables[:4, 0].tolist())) == 1


def test_invariant_entries_past_cdiv_never_read():
    wl = inputs.make_random([16, 17, 31, 32, 33], num_q_heads=2, num_kv_heads=1, head_dim=16,
                            block_size=16, kv_dtype="f32", seed=9, max_blocks_per_seq=6)
    k, v = _written(wl)
    a = oracle.decode(_problem_raw(wl, k, v, wl.block_tables))
    bt = wl.block_tables.clone()
    for i, L in enumerate(wl.seq_lens.tolist()):
        bt[i, -(-L // 16):] = 10 ** 6      # out of range: reading it would fail
    assert np.array_equal(a, oracle.decode(_problem_raw(wl, k, v, bt)))
    bt[0, 0] = 10 ** 6                    # a needed entry out of range is an error
    with pytest.raises(ValueError):
        oracle.decode(_problem_raw(wl, k, v, bt))


def test_gqa_groups_are_consecutive_heads():
    """Head h uses KV head h // G: distinct KV heads make the grouping visible."""
    wl, bt, k2, v2 = _contiguous_workload([24], 6, 3, 16, 8, "f32", seed=12)
    p = oracle.Problem(wl.q, oracle.F32, k2, v2, oracle.F32, bt, wl.seq_lens, 6, 3, 16, 8,
                       wl.num_blocks, wl.scale)
    got = oracle.decode(p)[0]
    q = oracle.as_raw(wl.q)[0].astype(np.float64)
    K = k2.reshape(-1, 3, 16)[:24].astype(np.float64)
    V = v2.reshape(-1, 3, 16)[:24].astype(np.float64)
    for h in range(6):
        want = _dense_from_contiguous(q[h:h + 1], K[:, h // 2:h // 2 + 1], V[:, h // 2:h // 2 + 1],
                                      float(np.float32(wl.scale)), 1)[0]
        np.testing.assert_allclose(got[h], want, rtol=1e-12, atol=1e-13)
        wrong = _dense_from_contiguous(q[h:h + 1], K[:, h % 3:h % 3 + 1], V[:, h % 3:h % 3 + 1],
                                       float(np.float32(wl.scale)), 1)[0]
        if h // 2 != h % 3:
            assert not np.allclose(got[h], wrong, rtol=1e-3, atol=1e-3)


@pytest.mark.parametrize("mistake", ["drop_last_partial_block", "offset_off_by_one"])
def test_planted_mistakes_are_caught(mistake):
    """A plausible indexing mistake planted in the oracle's inputs (on the
    CPU) must fail the dense comparison."""
    lens = [5, 17, 40, 77]
    wl, bt, k2, v2 = _contiguous_workload(lens, 4, 2, 32, 16, "f32", seed=13)
    seq_lens = wl.seq_lens.clone()
    kk, vv = k2, v2
    if mistake == "drop_last_partial_block":
        seq_lens = (seq_lens // 16) * 16
        seq_lens[seq_lens == 0] = 1
    else:
        kk = np.roll(k2, 1, axis=1); vv = np.roll(v2, 1, axis=1)
    bad = oracle.decode(oracle.Problem(wl.q, oracle.F32, kk, vv, oracle.F32, bt, seq_lens, 4, 2,
                                       32, 16, wl.num_blocks, wl.scale))
    good = oracle.decode(oracle.Problem(wl.q, oracle.F32, k2, v2, oracle.F32, bt, wl.seq_lens, 4,
                                        2, 32, 16, wl.num_blocks, wl.scale))
    diff = np.abs(bad - good).max(axis=-1)      # per (seq, head); NaN counts as caught
    assert (~(diff <= 1e-3)).all(axis=-1).all(), diff


def test_zero_length_gives_zeros():
    wl = inputs.make_random([4, 9], num_q_heads=2, num_kv_heads=1, head_dim=8, block_size=8,
                            kv_dtype="f32", seed=14)
    k, v = _written(wl)
    sl = wl.seq_lens.clone(); sl[1] = 0
    out = oracle.decode(oracle.Problem(wl.q, oracle.F32, k, v, oracle.F32, wl.block_tables, sl, 2,
                                       1, 8, 8, wl.num_blocks, wl.scale))
    assert np.array_equal(out[1], np.zeros((2, 8)))
    assert np.isfinite(out).all()


# ---------------------------------------------------------------------------
# fp8 caches: dequantise on read ("kv-cache-memory-core", section 4.4, and
# "vLLM intro part 2", section 7: the cache stores fp8 codes, a read widens a
# code and multiplies it by the tensor's scale).  The reference side decodes
# the codes with torch's float8 types -- not the oracle's codec -- and the K
# and V scales differ by a factor of 85, so using one for the other, or
# dropping either, moves the result far outside the comparison bound.
# ---------------------------------------------------------------------------
FP8_TORCH = {"fp8_e4m3": torch.float8_e4m3fn, "fp8_e5m2": torch.float8_e5m2}
K_SCALE, V_SCALE = 0.02, 1.7


def _fp8_codes(kind, shape, gen):
    """Codes of N(0, 16^2) values cast by torch (round to nearest, finite
    for both formats at this magnitude)."""
    x = torch.randn(shape, generator=gen) * 16.0
    return x.to(FP8_TORCH[kind]).view(torch.uint8).numpy()


def _fp8_contiguous(kind, lens, Hq, Hkv, D, bs, seed):
    """A pool of fp8 codes whose tables are the identity, and bf16 queries;
    returns (q raw, k codes, v codes, tables, seq_lens, NB)."""
    gen = torch.Generator().manual_seed(seed)
    nblk = [-(-L // bs) for L in lens]
    NB = sum(nblk)
    k = _fp8_codes(kind, (NB, bs, Hkv, D), gen)
    v = _fp8_codes(kind, (NB, bs, Hkv, D), gen)
    MB = max(nblk)
    bt = np.full((len(lens), MB), -1, dtype=np.int32)
    start = 0
    for i, n in enumerate(nblk):
        bt[i, :n] = np.arange(start, start + n)
        start += n
    q = torch.randn(len(lens), Hq, D, generator=gen).to(torch.bfloat16)
    return oracle.as_raw(q), k, v, bt, np.array(lens, dtype=np.int32), NB


def _fp8_dense_reference(kind, q_raw, k, v, lens, Hq, Hkv, D, bs, k_scale, v_scale):
    """Dense attention over the contiguous pool: codes widened by torch,
    times the scale, then numpy."""
    to64 = lambda a: torch.from_numpy(a).view(FP8_TORCH[kind]).to(torch.float64).numpy()
    qd = torch.from_numpy(q_raw.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    # the interface passes the scales as float32
    K = to64(k).reshape(-1, Hkv, D) * float(np.float32(k_scale))
    V = to64(v).reshape(-1, Hkv, D) * float(np.float32(v_scale))
    out, start = [], 0
    for i, L in enumerate(lens):
        out.append(_dense_from_contiguous(qd[i], K[start:start + L], V[start:start + L],
                                          float(np.float32(1.0 / math.sqrt(D))), Hq // Hkv))
        start += -(-int(L) // bs) * bs
    return np.stack(out)


def _fp8_oracle(kind, q_raw, k, v, bt, lens, Hq, Hkv, D, bs, NB, k_scale, v_scale):
    p = oracle.Problem(q_raw, oracle.BF16, k, v, oracle.DTYPE_CODES[kind], bt, lens, Hq, Hkv, D, bs, NB,
                       1.0 / math.sqrt(D), k_scale, v_scale)
    return oracle.decode(p)


@pytest.mark.parametrize("kind", ["fp8_e4m3", "fp8_e5m2"])
def test_oracle_fp8_dequantise_on_read_matches_dense(kind):
    lens = [1, 15, 16, 17, 40, 100]
    Hq, Hkv, D, bs = 8, 2, 64, 16
    q, k, v, bt, sl, NB = _fp8_contiguous(kind, lens, Hq, Hkv, D, bs, seed=31)
    got = _fp8_oracle(kind, q, k, v, bt, sl, Hq, Hkv, D, bs, NB, K_SCALE, V_SCALE)
    want = _fp8_dense_reference(kind, q, k, v, lens, Hq, Hkv, D, bs, K_SCALE, V_SCALE)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # L = 1 reads exactly v_scale times the one value code
    assert np.array_equal(got[0], want[0])


@pytest.mark.parametrize("kind", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("mistake", ["scales_swapped", "k_scale_dropped", "v_scale_dropped"])
def test_oracle_fp8_planted_scale_mistakes_are_caught(kind, mistake):
    """The dense check above fails when the oracle is handed the scales the
    way a plausible mistake would use them."""
    lens = [9, 33, 70]
    Hq, Hkv, D, bs = 4, 2, 64, 16
    q, k, v, bt, sl, NB = _fp8_contiguous(kind, lens, Hq, Hkv, D, bs, seed=32)
    ks, vs = {"scales_swapped": (V_SCALE, K_SCALE), "k_scale_dropped": (1.0, V_SCALE),
              "v_scale_dropped": (K_SCALE, 1.0)}[mistake]
    bad = _fp8_oracle(kind, q, k, v, bt, sl, Hq, Hkv, D, bs, NB, ks, vs)
    want = _fp8_dense_reference(kind, q, k, v, lens, Hq, Hkv, D, bs, K_SCALE, V_SCALE)
    err = np.abs(bad - want).max(axis=-1)                  # per (sequence, head)
    bound = 6e-2 + 6e-2 * np.abs(want).max(axis=-1)       # the GPU comparison's fp8 bound
    assert (err > bound).all(), (mistake, err.min(), bound.max())


def test_threaded_oracle_equals_decode():
    """The full-size GPU comparisons run oracle.attend_one per (sequence,
    head) on several host threads; that gives oracle.decode's values bit for
    bit."""
    from _harness import oracle_decode_threaded
    wl = inputs.make_random([1, 17, 300, 45, 1000], num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                            kv_dtype="fp8_e4m3", q_dtype="bf16", seed=33, v_mult=16.0)
    k, v = _written(wl)
    p = _problem_raw(wl, k, v, wl.block_tables)
    assert np.array_equal(oracle_decode_threaded(p, threads=4), oracle.decode(p))
