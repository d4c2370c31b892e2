"""Pins of the oracle's per-token K scales ("e4m3_tok": E4M3 codes with one fp32 scale per
(token, KV head) row).

Untitled KV-cache article at ldpk.cn/news/58971 §5.2: K develops outlier channels, so one scale
per tensor (or per head) leaves most tokens with a small part of the code range on long
contexts, and finer granularity (per channel or per token) is needed.  The reading taken: per
token's head row, s = max|x| / 448 in IEEE fp32 (448 = the largest finite E4M3 value), codes
e4m3(x / s) with the same rounding as the per-head path, value = code * s.

Pins: the row's largest element lands on the top code (+-448) and nothing saturates below it;
every code is the brute-force nearest E4M3 value of x / s (ties to even); torch's own
float8_e4m3fn cast of x / s gives the same codes; the relative reconstruction bound of E4M3;
zero rows, NaN elements and infinities; an outlier channel in one token leaves the other tokens'
error where it was (the per-head scale does not); the paged cache stores and gathers exactly the
decoded rows and copies the scales with the block; and planted mistakes (a per-head scale, a
truncating division, a dropped scale) that these pins catch.
"""

import numpy as np
import torch

import oracle as O


def _rows(seed, n=300, d=128):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d)).astype(np.float32)
    x[::7] *= 10.0 ** rng.uniform(-5, 5, (len(x[::7]), 1)).astype(np.float32)   # every magnitude
    x[3::11, 17] = 60.0                                                            # outlier channel
    x[5::13, :64] = 0.0                                                            # half-zero rows
    return O.f32_to_bf16_bits(x)


def _f32(bits):
    return O.bf16_bits_to_f64(bits).astype(np.float32)


def test_scale_is_the_row_absmax_over_448_in_fp32():
    bits = _rows(1)
    s = O.e4m3_token_scale(bits)
    x = _f32(bits)
    for i in range(len(bits)):
        a = np.float32(np.max(np.abs(x[i])))
        assert s[i] == np.float32(a / np.float32(448.0))
        assert s[i].dtype == np.float32


def test_largest_element_takes_the_top_code_and_nothing_else_saturates():
    bits = _rows(2)
    codes, s = O.quantize_token_rows(bits)
    x = _f32(bits)
    for i in range(len(bits)):
        j = int(np.argmax(np.abs(x[i])))
        assert codes[i, j] & 0x7F == 0x7E                        # +-448
        others = np.abs(x[i]) < np.abs(x[i, j]) * np.float32(0.93)
        assert np.all(codes[i][others] & 0x7F < 0x7E)


def test_codes_are_the_bruteforce_nearest_under_the_stored_scale():
    bits = _rows(3, n=40)
    codes, s = O.quantize_token_rows(bits)
    x = _f32(bits)
    for i in range(len(bits)):
        e = (x[i] / s[i]).astype(np.float32)
        for j in range(0, 128, 5):
            assert int(codes[i, j]) == O.e4m3_encode_bruteforce(float(e[j]))


def test_codes_match_torch_float8_cast_of_the_scaled_row():
    bits = _rows(4)
    codes, s = O.quantize_token_rows(bits)
    e = (_f32(bits) / s[:, None]).astype(np.float32)
    # torch's cast does not saturate: clamp first (|e| exceeds 448 only by a rounding step)
    ref = torch.from_numpy(np.clip(e, -448.0, 448.0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


def test_reconstruction_error_bound():
    bits = _rows(5)
    codes, s = O.quantize_token_rows(bits)
    x = _f32(bits).astype(np.float64)
    dec = O.e4m3_decode(codes) * s.astype(np.float64)[:, None]
    # E4M3: half a unit in the last place is 2^-4 relative for normals; subnormal spacing 2^-9
    bound = np.abs(x) * 2.0 ** -4 + s.astype(np.float64)[:, None] * 2.0 ** -10 + 1e-30
    assert np.all(np.abs(dec - x) <= bound * (1 + 1e-6))


def test_zero_rows_nan_and_infinity():
    z = np.zeros((2, 128), dtype=np.uint16)
    z[1, :] = 0x8000  # -0.0
    codes, s = O.quantize_token_rows(z)
    assert np.all(s == 1.0)
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0x80)
    x = np.ones(128, dtype=np.float32)
    x[5] = np.nan
    codes, s = O.quantize_token_rows(O.f32_to_bf16_bits(x)[None])
    assert s[0] == np.float32(1.0 / 448.0)          # NaN is left out of the maximum
    assert codes[0, 5] & 0x7F == 0x7F and codes[0, 0] == 0x7E
    allnan = O.f32_to_bf16_bits(np.full(128, np.nan, np.float32))[None]
    assert O.e4m3_token_scale(allnan)[0] == 1.0
    x = np.ones(128, dtype=np.float32)
    x[0] = np.inf
    _, s = O.quantize_token_rows(O.f32_to_bf16_bits(x)[None])
    assert np.isinf(s[0])


def test_outlier_channel_of_one_token_leaves_the_other_tokens_alone():
    """The point of the per-token scale: a per-head scale set by one token's outlier (here 10^5
    times the other tokens' values, beyond E4M3's 2^15 span of normal values) pushes every other
    token of the head into the subnormal codes; per token it does not."""
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((64, 128)) * 0.002).astype(np.float32)
    x[9, 40] = 300.0
    bits = O.f32_to_bf16_bits(x)
    xf = _f32(bits).astype(np.float64)
    codes, s = O.quantize_token_rows(bits)
    err_tok = np.abs(O.e4m3_decode(codes) * s.astype(np.float64)[:, None] - xf)
    head = np.float32(np.max(np.abs(_f32(bits))) / np.float32(448.0))
    err_head = np.abs(O.e4m3_decode(np.stack([O.quantize_row(b, head, "e4m3") for b in bits])) * float(head) - xf)
    others = np.arange(64) != 9
    assert err_tok[others].mean() < err_head[others].mean() / 5
    assert np.array_equal(err_tok[9], err_tok[9])  # the outlier row itself is encoded either way


def test_paged_cache_stores_codes_and_scales_and_copies_them_with_the_block():
    rng = np.random.default_rng(7)
    H, d = 4, 128
    vs = np.float32([0.03, 0.04, 0.02, 0.05])
    cache = O.PagedKVCache(6, H, d, k_dtype="e4m3_tok", v_dtype="int8", v_scales=vs, num_seqs=1, num_sink=2)
    row = np.array([4, 1, 3])
    x = O.f32_to_bf16_bits((rng.standard_normal((40, H, d)) * rng.uniform(0.1, 9, (40, H, 1))).astype(np.float32))
    for p in range(40):
        cache.append(0, row, p, x[p], x[p])
    K, V = cache.gather(0, row, 40)
    assert np.array_equal(K[:2], O.bf16_bits_to_f64(x[:2]))  # sinks stay bf16
    for p in range(2, 40):
        codes, sc = O.quantize_token_rows(x[p])
        assert np.array_equal(K[p], O.e4m3_decode(codes) * sc.astype(np.float64)[:, None])
        slot = O.locate(row, p)
        assert np.array_equal(cache.k_tscale[slot], sc)
    cache.block_copy(1, 5)
    assert np.array_equal(cache.k_tscale[80:96], cache.k_tscale[16:32])
    assert np.array_equal(cache.k[80:96], cache.k[16:32])


def test_planted_mistakes_are_caught():
    bits = _rows(8, n=60)
    codes, s = O.quantize_token_rows(bits)
    x = _f32(bits)
    # 1) a per-head scale (absmax over all tokens) instead of per token: the top-code pin fails
    head = np.float32(np.max(np.abs(x)) / np.float32(448.0))
    wrong = np.stack([O.quantize_row(b, head, "e4m3") for b in bits])
    top = [int(np.argmax(np.abs(x[i]))) for i in range(len(bits))]
    assert any(wrong[i, top[i]] & 0x7F != 0x7E for i in range(len(bits)))
    # 2) truncation toward zero instead of round-to-nearest: the brute-force pin fails
    e = (x / s[:, None]).astype(np.float32)
    trunc = np.sign(e) * np.floor(np.abs(e) * 8) / 8
    assert not np.array_equal(O.e4m3_encode(trunc.astype(np.float32)), codes)
    # 3) a dropped scale: decoding without it misses the rows by far more than the bound
    dec_wrong = O.e4m3_decode(codes)
    assert np.abs(dec_wrong - x).max() > 1.0
