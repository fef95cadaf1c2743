"""The seeded input generator: bit-exact to its published definition, and the
workload recipes have the stated shapes."""

import numpy as np
import torch

from synth import GAMMA, MASK64, NORMAL_MAX_ABS, mix13_t, normal_bf16, splitmix64_py, stream_key
from synth.workloads import WORKLOADS, make_workload


def test_splitmix64_reference_values():
    # first outputs of SplitMix64 seeded with 0 (state advanced by GAMMA before mixing)
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    got = [splitmix64_py((i + 1) * GAMMA & MASK64) for i in range(3)]
    assert got == expect


def test_torch_mix_matches_python_bigints():
    rng = np.random.default_rng(1)
    vals = [int(x) for x in rng.integers(0, 1 << 63, size=2000, dtype=np.int64)]
    vals += [0, 1, (1 << 63) - 1]
    t = torch.tensor(vals, dtype=torch.int64)
    got = mix13_t(t).numpy().astype(np.uint64)
    ref = np.array([splitmix64_py(v) for v in vals], dtype=np.uint64)
    assert np.array_equal(got, ref)


def test_normal_moments_and_bound():
    key = stream_key(2630, 1)
    x = normal_bf16(key, torch.arange(1 << 21)).float()
    assert abs(x.mean().item()) < 0.005
    assert abs(x.var().item() - 1.0) < 0.005
    assert x.abs().max().item() <= NORMAL_MAX_ABS * (1 + 2 ** -8)
    assert abs(NORMAL_MAX_ABS - 6 * 65535 / 65536) < 1e-12
    # tails past 3.5 sigma exist (a standard normal puts 4.7e-4 there; the
    # twelve-lane sum slightly less): about 800 of 2M
    tail = (x.abs() > 3.5).float().mean().item()
    assert 2e-4 < tail < 6e-4


def test_normal_values_follow_their_definition():
    """A few values recomputed from the definition with Python integers: three
    SplitMix64 words, the sum of their twelve 16-bit lanes, centred, times 2^-16,
    rounded to bf16 (round to nearest even)."""
    import struct
    key = stream_key(77, 3)
    ctr = [0, 1, 2, 12345, (1 << 40) + 17]
    got = normal_bf16(key, torch.tensor(ctr)).view(torch.int16).numpy().astype(np.uint16)
    for c, g in zip(ctr, got):
        s = 0
        for j in range(3):
            w = splitmix64_py((key + (3 * c + j) * GAMMA) & MASK64)
            s += sum((w >> (16 * i)) & 0xFFFF for i in range(4))
        f = (s - 6 * 65535) / 65536.0                      # exact in fp64 and in fp32
        u = struct.unpack("<I", struct.pack("<f", f))[0]
        rne = (u + 0x7FFF + ((u >> 16) & 1)) >> 16         # bf16, round to nearest even
        assert int(g) == rne, (c, hex(int(g)), hex(rne))


def test_counter_based_values_are_position_independent():
    key = stream_key(5, 2)
    full = normal_bf16(key, torch.arange(1000))
    part = normal_bf16(key, torch.arange(500, 700))
    assert torch.equal(full[500:700], part)


def test_workload_recipes():
    for name in WORKLOADS:
        wl = make_workload(name)
        assert wl.num_q_heads % wl.num_kv_heads == 0
        assert sorted(wl.free_order.tolist()) == list(range(wl.num_blocks))
    wl = make_workload("tiny")
    assert wl.context_lens.tolist() == [300, 2000, 600, 4400] and wl.num_blocks == 512
    wl = make_workload("llama8b")
    assert len(wl.context_lens) == 64 and wl.context_lens.min() >= 512 and wl.context_lens.max() <= 4096
    assert (wl.num_q_heads, wl.num_kv_heads, wl.num_blocks) == (32, 8, 65536)
    wl = make_workload("llama70b_prefix")
    tails = wl.context_lens - 2000
    assert len(tails) == 128 and tails.min() >= 1024 and tails.max() <= 32768
    need = 125 + 128 + sum(-(-int(t) // 16) for t in tails)
    assert wl.num_blocks >= need
    wl = make_workload("mixed_prefill")
    assert wl.q_lens[0] == 1024 and wl.context_lens[0] == 101024 and (wl.q_lens[1:] == 1).all()
    assert wl.context_lens[1:].min() >= 1024 and wl.context_lens[1:].max() <= 8192
    wl = make_workload("split_fp8")
    assert (wl.context_lens == 131072).all() and wl.kv_dtype == "fp8" and wl.num_splits == 16


def test_prefix_tokens_share_keys():
    wl = make_workload("llama70b_prefix")
    a = wl.token_keys(0, 0, 2010)
    b = wl.token_keys(5, 0, 2010)
    assert np.array_equal(a[:2000], b[:2000]) and not np.array_equal(a[2000:], b[2000:])


def test_fp8_scales_are_per_head_amax_over_every_token():
    """The fp8 scales of a workload: per KV head, separately for K and V, the
    largest |value| over every token of every sequence (the shared prefix once)
    divided by 448 in fp32.  Checked by brute force: each sequence's K/V
    gathered token by token through its own keys, then an elementwise max."""
    import numpy as np
    from synth.workloads import DISTINCT_FP8_FACTORS, small_workload
    wl = small_workload(21, lens=[40, 77, 300], hq=8, hkv=4, kv_dtype="fp8", prefix_tokens=40, cow_block=2)
    ka = np.zeros(4, np.float32)
    va = np.zeros(4, np.float32)
    for s in range(wl.num_seqs):
        k = wl.seq_kv("k", s).float().abs().numpy()
        v = wl.seq_kv("v", s).float().abs().numpy()
        ka = np.maximum(ka, k.max(axis=(0, 2)))
        va = np.maximum(va, v.max(axis=(0, 2)))
    ks, vs = wl.fp8_scales(device="cpu")
    assert np.array_equal(ks, (ka / np.float32(448)).astype(np.float32))
    assert np.array_equal(vs, (va / np.float32(448)).astype(np.float32))
    assert ks.dtype == np.float32 and len(set(ks.tolist())) > 1 and not np.array_equal(ks, vs)
    # with the test factors each scale is multiplied by its own factor
    wl2 = small_workload(21, lens=[40, 77, 300], hq=8, hkv=4, kv_dtype="fp8", prefix_tokens=40, cow_block=2,
                         fp8_scale_factors=DISTINCT_FP8_FACTORS)
    ks2, vs2 = wl2.fp8_scales(device="cpu")
    assert np.array_equal(ks2, (ks * DISTINCT_FP8_FACTORS[0][:4]).astype(np.float32))
    assert np.array_equal(vs2, (vs * DISTINCT_FP8_FACTORS[1][:4]).astype(np.float32))
