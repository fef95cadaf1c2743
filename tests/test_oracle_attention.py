"""Pins for the fp64 attention oracle, each against something other than itself.

* brute force in pure Python on tiny inputs;
* a library routine: torch's scaled_dot_product_attention in fp64 on the CPU,
  with GQA expressed through torch.repeat_interleave and the chunk mask built
  from positions;
* closed forms: one key, identical keys, constant values, zero scale, one
  dominant key;
* invariants the pages state: paging does not change the result (any block
  permutation, any block size), a shared-prefix block table equals duplicated
  copies, copy-on-write leaves the other sharer untouched, decode is the n = 1
  case of a chunk.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import model
from oracle.allocator import PoolModel, blocks_for
from synth.workloads import small_workload


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _paged(wl, **kw):
    tb = model.build_tables(wl)
    caches = model.build_cache(wl, tb)
    return model.expected_paged(wl, tb, caches, **kw)


def _contiguous_inputs(wl, s):
    L = int(wl.context_lens[s])
    k = wl.seq_kv("k", s).to(torch.float64)
    v = wl.seq_kv("v", s).to(torch.float64)
    cu = wl.cu_q_lens
    q = wl.q_values(np.arange(cu[s], cu[s + 1])).to(torch.float64)
    return q, k, v, L


# --------------------------------------------------------------- brute force
@pytest.mark.parametrize("D,bs", [(8, 4), (128, 16)])
def test_brute_force_tiny(D, bs):
    wl = small_workload(11, lens=[5, 40, 17], q_lens=[1, 3, 2], hq=4, hkv=2, head_dim=D,
                        block_size=bs)
    out = _paged(wl)
    G = wl.group
    cu = wl.cu_q_lens
    for s in range(wl.num_seqs):
        q, k, v, L = _contiguous_inputs(wl, s)
        n = int(wl.q_lens[s])
        for i in range(n):
            p = L - n + i
            for h in range(wl.num_q_heads):
                g = h // G
                z = []
                for t in range(p + 1):
                    acc = 0.0
                    for d in range(D):
                        acc += float(q[i, h, d]) * float(k[t, g, d])
                    z.append(acc / math.sqrt(D))
                mx = max(z)
                e = [math.exp(x - mx) for x in z]
                den = sum(e)
                for d in range(D):
                    o = sum(e[t] / den * float(v[t, g, d]) for t in range(p + 1))
                    assert abs(o - out[cu[s] + i, h, d]) <= 1e-12


# --------------------------------------------------------- library routine
@pytest.mark.parametrize("hq,hkv", [(8, 2), (8, 8), (8, 1), (64, 8)])
def test_matches_torch_sdpa_fp64(hq, hkv):
    wl = small_workload(12, lens=[33, 70, 129], q_lens=[1, 16, 5], hq=hq, hkv=hkv)
    out = _paged(wl)
    cu = wl.cu_q_lens
    G = hq // hkv
    for s in range(wl.num_seqs):
        q, k, v, L = _contiguous_inputs(wl, s)
        n = q.shape[0]
        kk = k.permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq][L][D]
        vv = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        pos_q = torch.arange(L - n, L)[:, None]
        pos_k = torch.arange(L)[None, :]
        mask = pos_k <= pos_q                                    # [n][L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.permute(1, 0, 2), kk, vv, attn_mask=mask, scale=1.0 / math.sqrt(128))
        got = out[cu[s]:cu[s + 1]]
        assert np.abs(ref.permute(1, 0, 2).numpy() - got).max() <= 1e-12


def test_matches_numpy_dense_softmax():
    wl = small_workload(13, lens=[100, 257], q_lens=[1, 1], hq=8, hkv=2)
    out = _paged(wl)
    for s in range(2):
        q, k, v, L = _contiguous_inputs(wl, s)
        for h in range(8):
            g = h // 4
            z = (k[:, g, :].numpy() @ q[0, h].numpy()) / math.sqrt(128)
            w = np.exp(z - z.max())
            w /= w.sum()
            ref = w @ v[:, g, :].numpy()
            assert np.abs(ref - out[s, h]).max() <= 1e-12


# -------------------------------------------------------------- closed forms
def _contig(q, k, v, scale=None):
    return oracle.contiguous_attention(q, k, v, scale=scale)


def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 4, 16))
    k = rng.standard_normal((1, 2, 16))
    v = rng.standard_normal((1, 2, 16))
    out = _contig(q, k, v)
    for h in range(4):
        assert np.array_equal(out[0, h], v[0, h // 2])


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    L = 37
    q = rng.standard_normal((1, 2, 16))
    k = np.repeat(rng.standard_normal((1, 1, 16)), L, axis=0)
    v = rng.standard_normal((L, 1, 16))
    out = _contig(q, k, v)
    assert np.abs(out[0, 0] - v[:, 0].mean(0)).max() <= 1e-13
    out0 = _contig(q, rng.standard_normal((L, 1, 16)), v, scale=0.0)
    assert np.abs(out0[0, 1] - v[:, 0].mean(0)).max() <= 1e-13


def test_weights_sum_to_one():
    """With V = 1 everywhere the output is the sum of the softmax weights."""
    rng = np.random.default_rng(2)
    L = 300
    q = rng.standard_normal((4, 8, 128)) * 3
    k = rng.standard_normal((L, 2, 128))
    out = _contig(q, k, np.ones((L, 2, 128)))
    assert np.abs(out - 1.0).max() <= 1e-12


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(3)
    L = 50
    k = rng.standard_normal((L, 1, 16)) * 0.01
    v = rng.standard_normal((L, 1, 16))
    q = np.zeros((1, 1, 16))
    q[0, 0, 0] = 1.0
    k[17, 0, 0] = 4000.0                 # score 1000 above the rest
    out = _contig(q, k, v, scale=0.25)
    assert np.abs(out[0, 0] - v[17, 0]).max() <= 1e-12


def test_causal_row_ignores_later_keys():
    rng = np.random.default_rng(4)
    L, n = 40, 6
    q = rng.standard_normal((n, 2, 16))
    k = rng.standard_normal((L, 1, 16))
    v = rng.standard_normal((L, 1, 16))
    a = _contig(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[L - 1] += 100.0
    v2[L - 1] -= 50.0                    # only the last query row may see token L-1
    b = _contig(q, k2, v2)
    assert np.array_equal(a[:n - 1], b[:n - 1])
    assert not np.array_equal(a[n - 1], b[n - 1])


# ---------------------------------------------------- invariants from the pages
@pytest.mark.parametrize("bs", [1, 4, 16, 32])
def test_paged_equals_contiguous_any_permutation(bs):
    wl_ref = small_workload(21, lens=[1, 15, 16, 17, 100], q_lens=[1, 1, 4, 1, 9], hq=8, hkv=2,
                            block_size=bs)
    for perm_seed in (5, 6, 7):
        # same value streams (same workload seed), different physical placement
        wl = small_workload(21, lens=[1, 15, 16, 17, 100], q_lens=[1, 1, 4, 1, 9], hq=8, hkv=2,
                            block_size=bs)
        wl.free_order = np.random.default_rng(perm_seed).permutation(wl.num_blocks).astype(np.int32)
        got = _paged(wl)
        cu = wl.cu_q_lens
        for s in range(wl.num_seqs):
            q, k, v, L = _contiguous_inputs(wl_ref, s)
            ref = oracle.contiguous_attention(q.numpy(), k.numpy(), v.numpy())
            assert np.array_equal(got[cu[s]:cu[s + 1]], ref)


def test_shared_prefix_equals_duplicated_copies():
    lens = [40, 57, 33]
    shared = small_workload(31, lens=lens, hq=8, hkv=2, prefix_tokens=32)
    tb = model.build_tables(shared)
    # every sequence points at the same physical prefix blocks
    pb = blocks_for(32)
    assert (tb.tables[:, :pb] == tb.tables[0, :pb]).all()
    assert tb.pool.stats()["shared"] == pb
    got = model.expected_paged(shared, tb)
    # duplicated copies: each sequence gets private blocks holding the same prefix
    dup = small_workload(31, lens=lens, hq=8, hkv=2, prefix_tokens=32)
    dup_tb_pool = PoolModel(dup.num_blocks, dup.free_order)
    tables = np.full((3, dup.max_blocks_per_seq), -1, np.int32)
    for s in range(3):
        tables[s, :blocks_for(lens[s])] = dup_tb_pool.alloc(blocks_for(lens[s]))
    kc = np.zeros((dup.num_blocks, 2, 16, 128), np.uint16)
    vc = np.zeros_like(kc)
    for s in range(3):
        slots = model.slots_for(tables[s], 0, lens[s])
        oracle.reshape_and_cache(_bits(dup.seq_kv("k", s)), _bits(dup.seq_kv("v", s)), kc, vc, slots)
    ref = oracle.paged_attention(_bits(dup.q_values()), kc, vc, tables, dup.context_lens)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("prefix", [32, 40])
def test_copy_on_write_leaves_other_sharer_untouched(prefix):
    """Sequence 0 forks the last prefix block and writes its tail; sequence 1's
    bytes and output do not change.  prefix=40 puts the fork on a partial block."""
    lens = [prefix + 20, prefix + 9]
    wl = small_workload(41, lens=lens, hq=8, hkv=2, prefix_tokens=prefix)
    pool = PoolModel(wl.num_blocks, wl.free_order)
    pb = blocks_for(prefix)
    pre = pool.alloc(pb)
    pool.share(pre)
    t0 = np.full(wl.max_blocks_per_seq, -1, np.int32)
    t1 = t0.copy()
    t0[:pb] = pre
    t1[:pb] = pre
    kc = np.zeros((wl.num_blocks, 2, 16, 128), np.uint16)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(_bits(wl.seq_kv("k", 0, 0, prefix)), _bits(wl.seq_kv("v", 0, 0, prefix)),
                             kc, vc, model.slots_for(t0, 0, prefix))
    # sequence 1 (the other sharer) finishes its own tokens first
    n1 = blocks_for(lens[1]) - pb
    own1 = pool.alloc(n1)
    t1[pb:pb + n1] = own1
    if prefix % 16:
        nb, need = pool.copy_on_write(t1[pb - 1])
        assert need
        kc[nb], vc[nb] = kc[t1[pb - 1]], vc[t1[pb - 1]]
        t1[pb - 1] = nb
    oracle.reshape_and_cache(_bits(wl.seq_kv("k", 1, prefix, lens[1])), _bits(wl.seq_kv("v", 1, prefix, lens[1])),
                             kc, vc, model.slots_for(t1, prefix, lens[1]))
    q1 = _bits(wl.q_values([1]))
    before = oracle.paged_attention(q1, kc, vc, t1[None], [lens[1]])
    snap_k, snap_v = kc.copy(), vc.copy()
    # sequence 0 forks the last prefix block and writes its tail into its copy
    old = int(t0[pb - 1])
    nb, need = pool.copy_on_write(old)
    if prefix % 16:
        # sequence 1 already took its own copy, so sequence 0 is the sole owner
        assert not need and nb == old
    else:
        assert need and nb != old
        kc[nb], vc[nb] = kc[old], vc[old]
    t0[pb - 1] = nb
    n0 = blocks_for(lens[0]) - pb
    t0[pb:pb + n0] = pool.alloc(n0)
    oracle.reshape_and_cache(_bits(wl.seq_kv("k", 0, prefix, lens[0])), _bits(wl.seq_kv("v", 0, prefix, lens[0])),
                             kc, vc, model.slots_for(t0, prefix, lens[0]))
    after = oracle.paged_attention(q1, kc, vc, t1[None], [lens[1]])
    assert np.array_equal(before, after)
    for b in t1[:blocks_for(lens[1])]:
        assert np.array_equal(kc[b], snap_k[b]) and np.array_equal(vc[b], snap_v[b])
    # and sequence 0 still equals contiguous attention on its logical tokens
    q0 = wl.q_values([0]).to(torch.float64).numpy()
    ref0 = oracle.contiguous_attention(q0, wl.seq_kv("k", 0).double().numpy(), wl.seq_kv("v", 0).double().numpy())
    got0 = oracle.paged_attention(_bits(wl.q_values([0])), kc, vc, t0[None], [lens[0]])
    assert np.array_equal(ref0, got0)


def test_decode_is_the_n1_case_of_a_chunk():
    wl = small_workload(51, lens=[90], q_lens=[7], hq=8, hkv=2)
    chunk = _paged(wl)
    q, k, v, L = _contiguous_inputs(wl, 0)
    for i in range(7):
        p = L - 7 + i
        one = oracle.contiguous_attention(q[i:i + 1].numpy(), k[:p + 1].numpy(), v[:p + 1].numpy())
        assert np.array_equal(one[0], chunk[i])


def test_expected_rows_matches_full_paged_oracle():
    wl = small_workload(61, lens=[300, 64, 129], q_lens=[24, 1, 3], hq=16, hkv=4)
    full = _paged(wl)
    cu = wl.cu_q_lens
    got = model.expected_rows(wl, 0, rows=[0, 1, 2, 10, 23])
    assert np.array_equal(got, full[cu[0] + np.array([0, 1, 2, 10, 23])])
    assert np.array_equal(model.expected_rows(wl, 2), full[cu[2]:cu[3]])


def test_fp8_paged_matches_dequantised_contiguous():
    wl = small_workload(71, lens=[50, 130], q_lens=[1, 5], hq=8, hkv=2, kv_dtype="fp8")
    full = _paged(wl)
    cu = wl.cu_q_lens
    for s in range(2):
        assert np.array_equal(model.expected_rows(wl, s), full[cu[s]:cu[s + 1]])


def test_sequence_without_query_rows_has_no_output_and_changes_nothing():
    """A sequence contributing no rows to a mixed batch (n = 0, the chunk-row
    definition over an empty range) leaves every other row as it is without it."""
    import numpy as np
    from oracle import model as om
    from synth.workloads import small_workload
    wl = small_workload(77, lens=[100, 50, 300, 17], q_lens=[5, 0, 1, 0], hq=8, hkv=2)
    full = om.expected_paged(wl)
    assert full.shape[0] == 6
    assert np.array_equal(full[0:5], om.expected_rows(wl, 0))
    assert np.array_equal(full[5:6], om.expected_rows(wl, 2))


def test_expected_rows_dequant_override_models_wrong_scales_on_the_right_bytes():
    """expected_rows(dequant=...) decodes the same fp8 bytes with other scales:
    with the workload's own scales it is the paged oracle bit for bit, and with
    K and V scales swapped it equals the paged oracle called with swapped
    scales over the same cache."""
    from synth.workloads import DISTINCT_FP8_FACTORS
    wl = small_workload(72, lens=[60, 33], q_lens=[1, 4], hq=8, hkv=2, kv_dtype="fp8",
                        fp8_scale_factors=DISTINCT_FP8_FACTORS)
    tb = model.build_tables(wl)
    kc, vc = model.build_cache(wl, tb)
    ks, vs = wl.fp8_scales()
    q = wl.q_values().contiguous().view(torch.int16).numpy().view(np.uint16)
    cu = wl.cu_q_lens
    for dq in ((ks, vs), (vs, ks)):
        full = oracle.paged_attention(q, kc, vc, tb.tables, wl.context_lens, cu, dtype=oracle.FP8,
                                      k_scale=dq[0], v_scale=dq[1], scale=wl.scale)
        for s in range(2):
            assert np.array_equal(model.expected_rows(wl, s, dequant=dq), full[cu[s]:cu[s + 1]])
