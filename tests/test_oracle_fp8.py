"""Pins for the oracle's E4M3 codec.

The cache format is one byte per element, E4M3 ("Waste, and three ways to
reclaim it", section "Quantising the cache"; "M.65 Inference serving",
quantisation (b): 4 exponent bits, 3 mantissa bits).  The oracle's encoder is
written from the format definition; here it is checked against torch's
float8_e4m3fn conversion (a library routine) wherever both define the result:
torch rounds to nearest-even but returns NaN past the largest finite value,
while the cache write saturates (satfinite), so values of magnitude above 464
are checked against the saturation rule instead.
"""
import numpy as np
import pytest
import torch

import oracle


def test_decode_all_256_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert np.array_equal(mine[~nan], ref[~nan])
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


@pytest.mark.parametrize("sign", [0, 1])
def test_encode_exhaustive_over_the_e4m3_range(sign):
    """Every fp32 value whose magnitude lies in [2^-12, 2^10) (all 2^23 mantissas
    of each of those 22 binades), which covers every rounding decision of the
    format: the round-to-zero region, the subnormals, every normal binade,
    and saturation."""
    mant = np.arange(1 << 23, dtype=np.uint32)
    for e in range(127 - 12, 127 + 10):
        bits = (np.uint32(sign) << 31) | (np.uint32(e) << 23) | mant
        x = bits.view(np.float32)
        mine = oracle.e4m3_encode(x)
        ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        a = np.abs(x)
        inside = a <= 464.0
        assert np.array_equal(mine[inside], ref[inside]), e
        sat = np.uint8(0xFE if sign else 0x7E)
        assert (mine[~inside] == sat).all()


def test_encode_random_bit_patterns():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    mine = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    a = np.abs(x)
    ok = (a <= 464.0) & ~np.isnan(x)
    assert np.array_equal(mine[ok], ref[ok])
    assert ((mine[np.isnan(x)] & 0x7F) == 0x7F).all()
    big = (a > 464.0) & ~np.isnan(x)
    assert ((mine[big] & 0x7F) == 0x7E).all()


@pytest.mark.parametrize("x,code", [
    (448.0, 0x7E), (464.0, 0x7E), (465.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E),
    (-float("inf"), 0xFE), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (1.5 * 2.0 ** -10, 0x01),
    (3 * 2.0 ** -10, 0x02), (2.0 ** -6, 0x08), (1.0, 0x38), (1.0625, 0x38), (1.1875, 0x3A),
    (-2.5, 0xC2), (0.0, 0x00), (-0.0, 0x80),
])
def test_encode_hand_checked(x, code):
    # 1.0625 is halfway between 1.0 and 1.125 -> even mantissa (1.0);
    # 1.1875 halfway between 1.125 (m=1) and 1.25 (m=2) -> even (m=2)
    assert oracle.lib().oracle_e4m3_from_f32(x) == code


def test_roundtrip_of_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_cache_write_quantises_with_fp32_division():
    """fp8 cache write = e4m3(fp32(x) / scale), per KV head."""
    rng = np.random.default_rng(9)
    T, H, D = 5, 2, 128
    x = torch.from_numpy(rng.standard_normal((T, H, D)).astype(np.float32) * 40).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    ks = np.array([0.05, 0.3], np.float32)
    vs = np.array([1.7, 0.011], np.float32)
    kc = np.zeros((4, H, 16, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.array([0, 17, -1, 63, 5], np.int64)
    oracle.reshape_and_cache(bits, bits, kc, vc, slots, oracle.FP8, ks, vs)
    xf = x.float().numpy()
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = divmod(int(sl), 16)
        for h in range(H):
            assert np.array_equal(kc[b, h, o], oracle.e4m3_encode(xf[t, h] / ks[h]))
            assert np.array_equal(vc[b, h, o], oracle.e4m3_encode(xf[t, h] / vs[h]))
    # the skipped token wrote nothing
    assert kc[0, :, 2].sum() == 0 and (kc[1, :, 0:1].sum() == 0)


def test_paged_attention_dequantises_with_each_heads_own_k_and_v_scale():
    """Closed form for the fp8 cache with per-KV-head scales that differ between
    K and V and across heads ("Quantising the cache": the stored byte times its
    scale is the value).  Sequence 0 has one key: every query head h of KV head
    g = h // G returns e4m3(v) * v_scale[g].  Sequence 1 has two keys: the
    weights are the two-way softmax of scale * q . (e4m3(k_t) * k_scale[g]),
    written out by hand here.  The decode of the bytes is torch's.  A swapped
    pair of scales, or head 0's scale used for every head, fails the check."""
    Hq, Hkv, D, G = 6, 3, 128, 2
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 256, size=(4, Hkv, 16, D), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30                      # no NaN codes
    kc, vc = codes[:2].copy(), codes[2:].copy()              # 2 blocks each
    ks = np.array([0.37, 2.9, 0.011], np.float32)
    vs = np.array([5.0, 0.11, 0.8], np.float32)
    tables = np.array([[1], [0]], np.int32)
    lens = np.array([1, 2], np.int32)
    q = torch.randn(2, Hq, D, dtype=torch.float64).to(torch.bfloat16)
    q_bits = q.view(torch.int16).numpy().view(np.uint16)
    scale = 1.0 / np.sqrt(D)

    def dec(c):
        return torch.from_numpy(np.ascontiguousarray(c)).view(torch.float8_e4m3fn).to(torch.float64).numpy()

    def run(k_scale, v_scale):
        return oracle.paged_attention(q_bits, kc, vc, tables, lens, dtype=oracle.FP8, k_scale=k_scale,
                                      v_scale=v_scale, scale=scale)

    out = run(ks, vs)
    qd = q.to(torch.float64).numpy()
    exp = np.zeros_like(out)
    for h in range(Hq):
        g = h // G
        exp[0, h] = dec(vc[1, g, 0]) * float(vs[g])                       # one key: its value
        k0, k1 = dec(kc[0, g, 0]) * float(ks[g]), dec(kc[0, g, 1]) * float(ks[g])
        z0, z1 = scale * qd[1, h] @ k0, scale * qd[1, h] @ k1
        w1 = 1.0 / (1.0 + np.exp(z0 - z1))
        exp[1, h] = (1.0 - w1) * dec(vc[0, g, 0]) * float(vs[g]) + w1 * dec(vc[0, g, 1]) * float(vs[g])
    assert np.abs(out - exp).max() <= 1e-12 * max(1.0, np.abs(exp).max())
    # the check has teeth: plausible scale mistakes move the result far away
    for wk, wv in ((vs, ks), (np.full(3, ks[0], np.float32), np.full(3, vs[0], np.float32))):
        assert np.abs(run(wk, wv) - exp).max() > 0.1
