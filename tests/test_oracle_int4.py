"""Pins of the oracle's INT4 quantiser (asymmetric, scale + zero point per 32-dim group).

Untitled KV-cache article at ldpk.cn/news/58971 §5.2: int4 needs a scale and a zero point
besides the 0.5-byte codes (0.55-0.65 bytes per element in practice), and K's outlier channels
call for per-channel or per-token granularity instead of one scale per tensor.

Pins: every unclamped code is the nearest of the 16 levels under the stored scale (brute
force); 0 encodes exactly; the reconstruction error bound; torch's own per-tensor quint4x2
quantiser (a library routine) agrees given the same scale and zero point; degenerate groups
(all zero, all positive, all negative, a single outlier); the storage cost the page quotes;
the paged INT4 cache gathering exactly the decoded rows; and planted mistakes (codes taken
with the unrounded scale, a range that leaves out 0, truncation instead of rounding).
"""

import numpy as np
import pytest
import torch

import oracle as O


def _groups(seed, n=400):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        kind = i % 6
        if kind == 0:
            x = rng.standard_normal(32)
        elif kind == 1:
            x = rng.standard_normal(32) * 10 ** rng.uniform(-6, 4)
        elif kind == 2:
            x = np.abs(rng.standard_normal(32)) + 0.5           # all positive
        elif kind == 3:
            x = -np.abs(rng.standard_normal(32)) - 0.5          # all negative
        elif kind == 4:
            x = rng.standard_normal(32) * 0.1
            x[rng.integers(0, 32)] = rng.choice([-1, 1]) * 40   # one outlier channel
        else:
            x = rng.standard_normal(32)
            x[rng.integers(0, 32, 5)] = 0.0
        out.append(O.f32_to_bf16_bits(x.astype(np.float32)))
    return out


def _f32(bits):
    return O.bf16_bits_to_f64(np.asarray(bits, dtype=np.uint16)).astype(np.float32)


def test_codes_are_the_nearest_level_and_zero_is_exact():
    for bits in _groups(1):
        q, sb, z = O.int4_encode_group(bits)
        x = _f32(bits)
        s = np.float32(O.bf16_bits_to_f64(np.array([sb], dtype=np.uint16))[0])
        assert 0 <= z <= 15 and q.min() >= 0 and q.max() <= 15
        levels = s.astype(np.float64) * (np.arange(16) - z)
        for xi, qi in zip(x.astype(np.float64), q):
            t = xi / float(s) + z
            if -0.5 < t < 15.5:  # not clamped: nearest level (a tie may go either way only at .5)
                d = np.abs(levels - xi)
                assert d[qi] <= d.min() + 1e-6 * abs(float(s)), (xi, qi, z, s)
        dec = O.int4_decode_row(q, np.array([sb | (z << 16)], dtype=np.uint32))
        assert np.all(dec[x == 0] == 0.0)


def test_reconstruction_error_bound():
    for bits in _groups(2):
        q, sb, z = O.int4_encode_group(bits)
        x = _f32(bits).astype(np.float64)
        s = float(O.bf16_bits_to_f64(np.array([sb], dtype=np.uint16))[0])
        dec = O.int4_decode_row(q, np.array([sb | (z << 16)], dtype=np.uint32))
        lo, hi = min(0.0, x.min()), max(0.0, x.max())
        slack = max(0.0, (hi - lo) - 15 * s) + abs(s) * 0.5 + abs(z * s + lo)
        assert np.all(np.abs(dec - x) <= slack * (1 + 1e-6) + 1e-30)


def test_matches_torch_quint4x2_given_the_same_scale_and_zero_point():
    diff = total = 0
    for bits in _groups(3):
        q, sb, z = O.int4_encode_group(bits)
        s = float(O.bf16_bits_to_f64(np.array([sb], dtype=np.uint16))[0])
        x = torch.from_numpy(_f32(bits))
        packed = torch.quantize_per_tensor(x, s, z, torch.quint4x2).int_repr().numpy()
        tq = np.stack([packed & 0xF, packed >> 4], axis=1).reshape(-1)  # element 2i in the low nibble
        # torch multiplies by a reciprocal, the oracle divides: they may differ only where
        # x / s sits within float rounding of a half-integer
        t = _f32(bits).astype(np.float64) / s
        near_tie = np.abs(np.abs(t - np.floor(t)) - 0.5) < 1e-5
        bad = (tq != q) & ~near_tie
        assert not bad.any()
        diff += int((tq != q).sum())
        total += len(q)
    assert diff <= total * 1e-3


def test_degenerate_groups():
    q, sb, z = O.int4_encode_group(np.zeros(32, dtype=np.uint16))
    assert sb == 0x3F80 and z == 0 and not q.any()
    pos = O.f32_to_bf16_bits(np.linspace(1, 4, 32).astype(np.float32))
    q, sb, z = O.int4_encode_group(pos)
    assert z == 0 and q.max() == 15
    neg = O.f32_to_bf16_bits(-np.linspace(1, 4, 32).astype(np.float32))
    q, sb, z = O.int4_encode_group(neg)
    assert z == 15 and q.min() == 0
    # a single nonzero value is reproduced exactly when the scale is exact (v / 15 a bf16)
    one = np.zeros(32, dtype=np.float32)
    one[7] = 15 * 0.25
    q, sb, z = O.int4_encode_group(O.f32_to_bf16_bits(one))
    dec = O.int4_decode_row(q, np.array([sb | (z << 16)], dtype=np.uint32))
    assert np.array_equal(dec, one.astype(np.float64))


def test_storage_cost_is_in_the_pages_range():
    # 32 codes of 4 bits + one 32-bit word (bf16 scale, zero point) per group
    per_elem = (32 * 0.5 + 4) / 32
    assert per_elem == 0.625 and 0.55 <= per_elem <= 0.65


def test_int4_paged_cache_gathers_the_decoded_rows_and_sinks():
    rng = np.random.default_rng(4)
    H, d = 2, 128
    cache = O.PagedKVCache(8, H, d, k_dtype="int4", v_dtype="int4", num_seqs=1, num_sink=2)
    row = np.array([5, 1, 3])
    x = O.f32_to_bf16_bits(rng.standard_normal((40, H, d)).astype(np.float32))
    y = O.f32_to_bf16_bits(rng.standard_normal((40, H, d)).astype(np.float32))
    for p in range(40):
        cache.append(0, row, p, x[p], y[p])
    K, V = cache.gather(0, row, 40)
    assert np.array_equal(K[:2], O.bf16_bits_to_f64(x[:2])) and np.array_equal(V[:2], O.bf16_bits_to_f64(y[:2]))
    for p in (2, 17, 39):
        for h in range(H):
            c, prm = O.int4_encode_row(x[p, h])
            assert np.array_equal(K[p, h], O.int4_decode_row(c, prm))
            c, prm = O.int4_encode_row(y[p, h])
            assert np.array_equal(V[p, h], O.int4_decode_row(c, prm))
    # copy-on-write carries the parameters with the codes
    cache.block_copy(1, 6)
    assert np.array_equal(cache.k_params[96:112], cache.k_params[16:32])
    assert np.array_equal(cache.v[96:112], cache.v[16:32])


def test_planted_int4_mistakes_are_caught():
    groups = _groups(5, 300)

    def unrounded_scale(bits):  # codes from the fp32 scale, the bf16 one stored
        x = _f32(bits)
        lo, hi = min(np.float32(0), x.min()), max(np.float32(0), x.max())
        s = np.float32(np.float32(hi - lo) / np.float32(15))
        z = int(np.clip(np.rint(np.float32(-lo) / s), 0, 15))
        return np.clip(np.rint(x / s) + z, 0, 15).astype(np.uint8)

    def range_without_zero(bits):
        x = _f32(bits)
        lo, hi = x.min(), x.max()
        s = np.float32(np.float32(hi - lo) / np.float32(15))
        s = np.float32(O.bf16_bits_to_f64(O.f32_to_bf16_bits(np.array([s], dtype=np.float32)))[0])
        return s * (np.clip(np.rint((x - lo) / s), 0, 15)) + lo

    def truncating(bits):
        q, sb, z = O.int4_encode_group(bits)
        x = _f32(bits)
        s = np.float32(O.bf16_bits_to_f64(np.array([sb], dtype=np.uint16))[0])
        return np.clip(np.trunc(x / s) + z, 0, 15).astype(np.uint8)

    assert any(not np.array_equal(unrounded_scale(b), O.int4_encode_group(b)[0]) for b in groups)
    assert any(np.any(range_without_zero(b)[_f32(b) == 0] != 0) for b in groups)
    assert any(not np.array_equal(truncating(b), O.int4_encode_group(b)[0]) for b in groups)


def test_batched_rows_encode_each_group_on_its_own():
    """The encoder takes rows with leading axes ([tokens][heads][d]) only as a batch of
    independent groups: every row equals its own one-group-at-a-time encoding, including rows
    whose groups differ wildly in range (a group's scale never depends on another group)."""
    gs = _groups(7, 240)
    rows = np.stack([np.concatenate(gs[i:i + 4]) for i in range(0, 240, 4)])  # 60 rows of d = 128
    batch = rows.reshape(6, 10, 128)
    codes, params = O.int4_encode_row(batch)
    assert codes.shape == (6, 10, 128) and params.shape == (6, 10, 4)
    for t in range(6):
        for h in range(10):
            row = batch[t, h]
            for g in range(4):
                q, sb, z = O.int4_encode_group(row[32 * g:32 * g + 32])
                assert np.array_equal(codes[t, h, 32 * g:32 * g + 32], q)
                assert int(params[t, h, g]) == sb | (z << 16)
