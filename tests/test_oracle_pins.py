"""Pins for the CPU oracle: values printed on the pages, closed forms, library routines,
brute force on tiny inputs.  None of these re-types the oracle's own formula; each is
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand, the wrong head grouping) fails at least one of them.  The last
section plants such slips in copies of the oracle and checks the pins catch them."""

import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            data, _, src = line.partition("|")
            yield data.split(), src.strip()


# ----------------------------------------------------------------------------------
# Byte formula (printed integers and sizes)
# ----------------------------------------------------------------------------------
def test_bytes_per_token_matches_printed_values():
    n = 0
    for (L, H, d, b, expected), src in _rows("kv_bytes_per_token.txt"):
        assert O.kv_bytes_per_token(int(L), int(H), int(d), int(b)) == int(expected), src
        n += 1
    assert n == 9


def test_total_bytes_match_printed_sizes():
    units = {"GiB": 2.0 ** 30, "GB": 1e9, "B": 1.0, "KiB-MB-GB": 1024.0 * 1024.0 * 1000.0}
    n = 0
    for line in open(os.path.join(GOLDEN, "kv_bytes_total.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        left, mid, src = [p.strip() for p in line.split("|")]
        L, H, d, b, S, B = map(int, left.split())
        unit, printed, decimals = mid.split()[:3]
        total = O.kv_bytes_total(L, H, d, b, S, B)
        assert round(total / units[unit], int(decimals)) == float(printed), (src, total)
        n += 1
    assert n == 17


def test_page_arithmetic_errors_are_not_reproduced():
    for line in open(os.path.join(GOLDEN, "kv_bytes_page_errors.txt"), encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        left, mid, src = [p.strip() for p in line.split("|")]
        L, H, d, b, S, B = map(int, left.split())
        printed_gb, exact = mid.split()
        total = O.kv_bytes_total(L, H, d, b, S, B)
        assert total == int(exact), src
        assert abs(total / 1e9 - float(printed_gb)) > 1.0, src


def test_gqa_divides_cache_by_group():
    # 显存账本 §二: GQA-8 cuts the cache to 1/8 of MHA with 64 query heads; MQA to 1/64.
    mha = O.kv_bytes_per_token(80, 64, 128, 2)
    assert O.kv_bytes_per_token(80, 8, 128, 2) * 8 == mha
    assert O.kv_bytes_per_token(80, 1, 128, 2) * 64 == mha
    # 显存账本 §七: GQA stacked with 8-bit KV gives 1/16 of MHA + FP16.
    assert O.kv_bytes_per_token(80, 8, 128, 1) * 16 == mha


# ----------------------------------------------------------------------------------
# locate() and fragmentation
# ----------------------------------------------------------------------------------
def test_locate_worked_example():
    table = [7, 3, 19, 42]
    n = 0
    for (pos, expected), _src in _rows("locate_example.txt"):
        pos, expected = int(pos), int(expected)
        if expected < 0:
            with pytest.raises(IndexError):
                O.locate(table, pos)
        else:
            assert O.locate(table, pos, 16) == expected
        n += 1
    assert n == 11


def test_locate_rejects_unassigned_and_negative():
    with pytest.raises(IndexError):
        O.locate([5, -1], 20)
    with pytest.raises(IndexError):
        O.locate([5], -1)


def test_locate_is_a_bijection_onto_the_assigned_blocks():
    rng = np.random.default_rng(1)
    table = rng.permutation(50)[:9]
    slots = O.slots_of_sequence(table, 9 * 16)
    assert len(set(slots.tolist())) == 9 * 16
    assert set((slots // 16).tolist()) == set(table.tolist())


@pytest.mark.parametrize("ctx", [1, 2, 15, 16, 17, 300, 4095, 4096, 4097])
def test_tail_waste_is_below_one_block(ctx):
    # 显存账本 §四: internal fragmentation never exceeds one block — worst case 15 tokens.
    waste = O.blocks_needed(ctx) * 16 - ctx
    assert 0 <= waste <= 15


def test_worst_case_tail_waste_is_fifteen_and_average_half_a_block():
    wastes = [O.blocks_needed(c) * 16 - c for c in range(1, 16 * 1000 + 1)]
    assert max(wastes) == 15
    assert abs(np.mean(wastes) - 7.5) < 1e-9  # ldpk §4.3: on average half a block


def test_naive_reservation_waste_example():
    # 显存账本 §三: 300 tokens used out of a 4096 reservation wastes 92%.
    assert math.floor(100 * (4096 - 300) / 4096) == 92
    # paged: the same request wastes at most one block
    assert O.blocks_needed(300) * 16 - 300 < 16


# ----------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------
def test_bf16_bits_roundtrip_and_rounding():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_f64(bits)
    finite = np.isfinite(vals)
    back = O.f32_to_bf16_bits(vals[finite].astype(np.float32))
    assert np.array_equal(back, bits[finite])
    # against torch's own fp32 -> bf16 (round to nearest even) on a dense sweep
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), ref)


def test_e4m3_decode_definition_values():
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert O.e4m3_decode(np.uint8(0xFE)) == -448.0
    assert O.e4m3_decode(np.uint8(0x38)) == 1.0
    assert O.e4m3_decode(np.uint8(0xB8)) == -1.0
    assert O.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6  # smallest normal
    assert O.e4m3_decode(np.uint8(0x07)) == 7 * 2.0 ** -9  # largest subnormal
    assert O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9  # smallest subnormal
    assert O.e4m3_decode(np.uint8(0x00)) == 0.0
    assert np.isnan(O.e4m3_decode(np.uint8(0x7F)))
    assert np.isnan(O.e4m3_decode(np.uint8(0xFF)))
    mags = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(mags) > 0)  # code order is value order


def test_e4m3_encode_roundtrips_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_e4m3_midpoints_tie_to_even_and_neighbours_round_to_nearest():
    mags = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        mid = (mags[c] + mags[c + 1]) / 2.0
        assert np.float32(mid) == mid  # exactly representable, so the tie is real
        even = c if c % 2 == 0 else c + 1
        assert O.e4m3_encode(np.float32(mid)) == even
        assert O.e4m3_encode(np.float32(-mid)) == even | 0x80
        below = np.nextafter(np.float32(mid), np.float32(0))
        above = np.nextafter(np.float32(mid), np.float32(1e9))
        assert O.e4m3_encode(below) == c
        assert O.e4m3_encode(above) == c + 1


def test_e4m3_saturates_and_handles_specials():
    assert O.e4m3_encode(np.float32(448.0)) == 0x7E
    assert O.e4m3_encode(np.float32(463.99)) == 0x7E
    assert O.e4m3_encode(np.float32(1e6)) == 0x7E
    assert O.e4m3_encode(np.float32(np.inf)) == 0x7E
    assert O.e4m3_encode(np.float32(-np.inf)) == 0xFE
    assert O.e4m3_encode(np.float32(2.0 ** -10)) == 0x00  # tie with 0 -> even (0)
    assert O.e4m3_encode(np.float32(-2.0 ** -11)) == 0x80  # negative underflow keeps sign
    assert O.e4m3_encode(np.float32(np.nan)) & 0x7F == 0x7F


def test_e4m3_encode_matches_bruteforce_nearest():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(3000) * np.exp2(rng.integers(-12, 10, 3000))).astype(np.float32)
    got = O.e4m3_encode(x)
    for xi, gi in zip(x, got):
        assert gi == O.e4m3_encode_bruteforce(float(xi))


def test_e4m3_encode_matches_torch_float8_in_range():
    # torch's float8_e4m3fn cast rounds to nearest even but does not saturate, so the
    # comparison covers the finite range only.
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(400000) * np.exp2(rng.integers(-14, 9, 400000))).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(x), ref)


def test_int8_encode_matches_rint_and_clamps():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(400000) * 60).astype(np.float32)
    x = np.concatenate([x, np.arange(-140, 140, 0.5, dtype=np.float32)])
    ref = np.clip(np.rint(x.astype(np.float64)), -127, 127).astype(np.int8)
    assert np.array_equal(O.int8_encode(x), ref)
    assert O.int8_encode(np.float32(0.5)) == 0
    assert O.int8_encode(np.float32(1.5)) == 2
    assert O.int8_encode(np.float32(2.5)) == 2
    assert O.int8_encode(np.float32(-2.5)) == -2
    assert O.int8_encode(np.float32(127.5)) == 127
    assert O.int8_encode(np.float32(-1000)) == -127
    assert O.int8_encode(np.float32(np.nan)) == 0


def test_quantize_row_divides_in_fp32_then_rounds():
    # decode(code) * scale is within half a code step of x (relative to scale)
    rng = np.random.default_rng(6)
    x = rng.standard_normal(4096).astype(np.float32)
    bits = O.f32_to_bf16_bits(x)
    xv = O.bf16_bits_to_f64(bits)
    s_k = np.float32(np.abs(xv).max() / 448.0)
    s_v = np.float32(np.abs(xv).max() / 127.0)
    kq = O.quantize_row(bits, s_k, "e4m3")
    vq = O.quantize_row(bits, s_v, "int8")
    k_back = O.e4m3_decode(kq) * float(s_k)
    v_back = O.int8_decode(vq.view(np.int8)) * float(s_v)
    assert np.all(np.abs(v_back - xv) <= 0.5 * float(s_v) * (1 + 1e-6))
    assert np.all(np.abs(k_back - xv) <= np.abs(xv) * 2.0 ** -4 + 2.0 ** -10 * float(s_k))
    # the largest |x| maps to the largest code
    i = np.argmax(np.abs(xv))
    assert kq[i] & 0x7F == 0x7E and abs(int(vq.view(np.int8)[i])) == 127


# ----------------------------------------------------------------------------------
# Attention
# ----------------------------------------------------------------------------------
def _sdpa_reference(q, K, V, scale):
    """torch's scaled_dot_product_attention in fp64 with KV heads expanded to query heads."""
    H_q, d = q.shape
    ctx, H_kv, _ = K.shape
    G = H_q // H_kv
    qt = torch.from_numpy(q).reshape(1, H_q, 1, d)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return out.reshape(H_q, d).numpy()


def _random_case(rng, H_q, H_kv, d, ctx):
    q = rng.standard_normal((H_q, d))
    K = rng.standard_normal((ctx, H_kv, d))
    V = rng.standard_normal((ctx, H_kv, d))
    return q, K, V


def _attention_pins_pass(fn) -> bool:
    """True iff ``fn`` (same signature as decode_attention) passes the library and
    closed-form pins.  Used on the oracle itself and on planted mutants."""
    rng = np.random.default_rng(7)
    for H_q, H_kv, d, ctx in [(4, 2, 8, 1), (8, 2, 16, 33), (6, 6, 8, 5), (4, 1, 8, 17), (8, 4, 4, 9)]:
        q, K, V = _random_case(rng, H_q, H_kv, d, ctx)
        scale = 1.0 / math.sqrt(d)
        if not np.allclose(fn(q, K, V, scale), _sdpa_reference(q, K, V, scale), rtol=0, atol=1e-12):
            return False
    # ctx = 1: the output is V_0 of the head's KV head, exactly
    q, K, V = _random_case(rng, 4, 2, 8, 1)
    out = fn(q, K, V, 0.3)
    if not np.array_equal(out, V[0, [0, 0, 1, 1], :]):
        return False
    # all keys equal: uniform weights, output = mean of V
    q, K, V = _random_case(rng, 4, 2, 8, 7)
    K[:] = K[0]
    if not np.allclose(fn(q, K, V, 0.5), V.mean(axis=0)[[0, 0, 1, 1]], atol=1e-14):
        return False
    # one key aligned with a huge score dominates
    q, K, V = _random_case(rng, 2, 1, 8, 9)
    K[4, 0] = np.sign(q[0]) * 1e3
    out = fn(q[:1], K, V, 1.0)
    if not np.allclose(out[0], V[4, 0], atol=1e-12):
        return False
    return True


def test_oracle_attention_passes_pins():
    assert _attention_pins_pass(O.decode_attention)


def test_empty_context_gives_zeros():
    q = np.ones((4, 8))
    K = np.zeros((0, 2, 8))
    assert np.array_equal(O.decode_attention(q, K, K, 1.0), np.zeros((4, 8)))


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(8)
    for n in [1, 2, 17, 4097]:
        w = O.softmax_weights(rng.standard_normal(n) * 30)
        assert abs(w.sum() - 1.0) < 1e-15 * max(1, n) ** 0.5 * 10
        assert np.all(w >= 0)


def test_mha_and_mqa_special_cases():
    rng = np.random.default_rng(9)
    # G = 1 reduces to plain multi-head attention per head
    q, K, V = _random_case(rng, 3, 3, 8, 12)
    out = O.decode_attention(q, K, V, 0.25)
    for h in range(3):
        s = 0.25 * K[:, h] @ q[h]
        w = np.exp(s - s.max())
        assert np.allclose(out[h], (w / w.sum()) @ V[:, h], atol=1e-14)
    # H_kv = 1 (MQA): every head reads the same K/V
    q, K, V = _random_case(rng, 5, 1, 8, 12)
    out = O.decode_attention(q, K, V, 0.25)
    single = [O.decode_attention(q[h:h + 1], K, V, 0.25)[0] for h in range(5)]
    assert np.array_equal(out, np.stack(single))


@pytest.mark.parametrize("part", [1, 2, 7, 16, 512, 100000])
def test_split_context_merge_equals_single_pass(part):
    rng = np.random.default_rng(10)
    q, K, V = _random_case(rng, 8, 2, 16, 1031)
    ref = O.decode_attention(q, K, V, 0.25)
    got = O.decode_attention_split(q, K, V, 0.25, part)
    assert np.allclose(got, ref, rtol=0, atol=1e-13)


def _fill_paged(rng, tables, ctxs, H, d, num_blocks):
    cache = O.PagedKVCache(num_blocks, H, d, num_seqs=len(ctxs))
    data = []
    for s, (row, n) in enumerate(zip(tables, ctxs)):
        kb = O.f32_to_bf16_bits(rng.standard_normal((n, H, d)).astype(np.float32))
        vb = O.f32_to_bf16_bits(rng.standard_normal((n, H, d)).astype(np.float32))
        for p in range(n):
            cache.append(s, row, p, kb[p], vb[p])
        data.append((kb, vb))
    return cache, data


def test_paged_equals_contiguous_and_is_permutation_invariant():
    rng = np.random.default_rng(11)
    H_q, H, d, nb = 8, 2, 16, 40
    ctxs = [1, 17, 100, 33]
    need = [O.blocks_needed(c) for c in ctxs]
    q = rng.standard_normal((len(ctxs), H_q, d))
    outs = []
    for perm_seed in (0, 1):
        perm = np.random.default_rng(100 + perm_seed).permutation(nb)
        tables, k = [], 0
        for n in need:
            row = np.full(8, -1)
            row[:n] = perm[k:k + n]
            k += n
            tables.append(row)
        cache, data = _fill_paged(np.random.default_rng(12), tables, ctxs, H, d, nb)
        dense = O.ContiguousKVCache(len(ctxs), H, 128, d)
        for s, (kb, vb) in enumerate(data):
            for p in range(ctxs[s]):
                dense.append(s, O.bf16_bits_to_f64(kb[p]), O.bf16_bits_to_f64(vb[p]))
        per_seq = []
        for s in range(len(ctxs)):
            K, V = cache.gather(s, tables[s], ctxs[s])
            Kd, Vd = dense.view(s)
            assert np.array_equal(K, Kd) and np.array_equal(V, Vd)
            per_seq.append(O.decode_attention(q[s], K, V, 0.25))
        outs.append(np.stack(per_seq))
    assert np.array_equal(outs[0], outs[1])


def test_shared_prefix_equals_duplicated_prefix_and_cow_keeps_source():
    rng = np.random.default_rng(13)
    H_q, H, d = 4, 2, 8
    prefix, suffix = 40, [5, 9]  # prefix ends inside block 2 (40 = 2*16 + 8)
    pool = O.BlockPool(32)
    cache = O.PagedKVCache(32, H, d, num_seqs=2)
    pk = O.f32_to_bf16_bits(rng.standard_normal((prefix, H, d)).astype(np.float32))
    pv = O.f32_to_bf16_bits(rng.standard_normal((prefix, H, d)).astype(np.float32))
    owner = np.full(8, -1)
    for p in range(prefix):
        pool.prepare_append(owner, p)
        cache.append(0, owner, p, pk[p], pv[p])
    rows = [pool.fork(owner, 3), pool.fork(owner, 3)]  # the prefix owner keeps its ref
    src_before = (cache.k[owner[2] * 16:(owner[2] + 1) * 16].copy(),
                  cache.v[owner[2] * 16:(owner[2] + 1) * 16].copy())
    sk = [O.f32_to_bf16_bits(rng.standard_normal((n, H, d)).astype(np.float32)) for n in suffix]
    sv = [O.f32_to_bf16_bits(rng.standard_normal((n, H, d)).astype(np.float32)) for n in suffix]
    for s in range(2):
        for i in range(suffix[s]):
            act = pool.prepare_append(rows[s], prefix + i)
            if act[0] == "copy":
                cache.block_copy(act[1], act[2])
            cache.append(s, rows[s], prefix + i, sk[s][i], sv[s][i])
    # the shared partial block was copied, never written
    assert np.array_equal(cache.k[owner[2] * 16:(owner[2] + 1) * 16], src_before[0])
    assert np.array_equal(cache.v[owner[2] * 16:(owner[2] + 1) * 16], src_before[1])
    assert rows[0][2] != owner[2] and rows[1][2] != owner[2] and rows[0][2] != rows[1][2]
    assert rows[0][0] == owner[0] and rows[1][1] == owner[1]
    assert pool.refcount[owner[0]] == 3 and pool.refcount[owner[2]] == 1
    # the same tokens laid out without sharing give bit-identical attention
    dup = O.PagedKVCache(32, H, d, num_seqs=2)
    q = rng.standard_normal((2, H_q, d))
    for s in range(2):
        row = np.arange(8) + 8 * s
        toks_k = np.concatenate([pk, sk[s]])
        toks_v = np.concatenate([pv, sv[s]])
        for p in range(prefix + suffix[s]):
            dup.append(s, row, p, toks_k[p], toks_v[p])
        K1, V1 = cache.gather(s, rows[s], prefix + suffix[s])
        K2, V2 = dup.gather(s, row, prefix + suffix[s])
        assert np.array_equal(K1, K2) and np.array_equal(V1, V2)
        assert np.array_equal(O.decode_attention(q[s], K1, V1, 0.3), O.decode_attention(q[s], K2, V2, 0.3))


def test_sinks_are_read_from_the_sink_buffer_and_paged_slot_untouched():
    rng = np.random.default_rng(14)
    H, d = 2, 128
    ks = np.float32([0.01, 0.02])
    vs = np.float32([0.03, 0.04])
    cache = O.PagedKVCache(4, H, d, k_dtype="e4m3", v_dtype="int8", k_scales=ks, v_scales=vs,
                           num_seqs=1, num_sink=4)
    row = np.array([2, 0])
    x = O.f32_to_bf16_bits(rng.standard_normal((20, H, d)).astype(np.float32))
    for p in range(20):
        cache.append(0, row, p, x[p], x[p])
    assert np.all(cache.k[32:36] == 0) and np.all(cache.v[32:36] == 0)  # slots of pos 0..3 untouched
    K, V = cache.gather(0, row, 20)
    assert np.array_equal(K[:4], O.bf16_bits_to_f64(x[:4]))
    assert np.array_equal(V[:4], O.bf16_bits_to_f64(x[:4]))
    # quantised positions decode to code * scale
    k_codes = np.stack([O.quantize_row(x[7][h], ks[h], "e4m3") for h in range(H)])
    assert np.array_equal(K[7], O.e4m3_decode(k_codes) * ks.astype(np.float64)[:, None])


# ----------------------------------------------------------------------------------
# Block pool
# ----------------------------------------------------------------------------------
def test_pool_allocates_lowest_free_first_and_recycles_at_zero():
    pool = O.BlockPool(6)
    assert [pool.alloc() for _ in range(3)] == [0, 1, 2]
    assert pool.incref(1) == 2
    assert pool.decref(1) == 1 and pool.num_free() == 3
    assert pool.decref(1) == 0 and pool.num_free() == 4
    assert pool.alloc() == 1
    assert pool.decref(5) == -1 and pool.incref(5) == -1  # not allocated
    assert pool.claim(4) and not pool.claim(4)
    assert [pool.alloc(), pool.alloc(), pool.alloc()] == [3, 5, -1]


def test_pool_refcounts_conserve_under_random_operations():
    rng = np.random.default_rng(15)
    pool = O.BlockPool(64)
    model = {}  # brute-force model: block -> refcount
    for _ in range(5000):
        op = rng.integers(3)
        if op == 0:
            b = pool.alloc()
            if b >= 0:
                assert b not in model
                assert b == min(set(range(64)) - set(model))
                model[b] = 1
        elif model:
            b = int(rng.choice(sorted(model)))
            if op == 1:
                pool.incref(b)
                model[b] += 1
            else:
                pool.decref(b)
                model[b] -= 1
                if model[b] == 0:
                    del model[b]
        assert pool.num_free() == 64 - len(model)
        assert all(pool.refcount[b] == c for b, c in model.items())


def test_fork_release_cycle_leaks_nothing():
    pool = O.BlockPool(100)
    base = np.full(12, -1)
    for p in range(150):
        pool.prepare_append(base, p)
    used = pool.num_free()
    for _ in range(20):
        rows = [pool.fork(base, O.blocks_needed(150)) for _ in range(4)]
        assert all(pool.refcount[b] == 5 for b in base[:10])
        for r in rows:
            act = pool.prepare_append(r, 150)
            assert act[0] == "copy"
            for p in range(151, 170):
                pool.prepare_append(r, p)
        for r in rows:
            pool.release(r, 12)
        assert pool.num_free() == used


def test_prefix_sharing_memory_ratio():
    # 显存账本 §四: 64 requests sharing a ~1200-token prompt hold it once (24 GB -> 0.4 GB).
    pool = O.BlockPool(64 * 80)
    owner = np.full(80, -1)
    for p in range(1200):
        pool.prepare_append(owner, p)
    rows = [pool.fork(owner, O.blocks_needed(1200)) for _ in range(64)]
    shared_blocks = 64 * 80 - pool.num_free()
    assert shared_blocks == O.blocks_needed(1200) == 75
    dup_blocks = 64 * O.blocks_needed(1200)
    assert dup_blocks / shared_blocks == 64
    assert all(pool.refcount[b] == 65 for b in owner[:75])
    del rows


# ----------------------------------------------------------------------------------
# Planted mistakes: copies of the oracle with one plausible slip each must fail a pin.
# ----------------------------------------------------------------------------------
def _mutant_wrong_grouping(q, K, V, scale):
    H_q, d = q.shape
    H_kv = K.shape[1]
    out = np.zeros((H_q, d))
    for h in range(H_q):
        kv = h % H_kv  # interleaved instead of contiguous grouping
        w = O.softmax_weights(scale * (K[:, kv] @ q[h]))
        out[h] = w @ V[:, kv]
    return out


def _mutant_dropped_scale(q, K, V, scale):
    return O.decode_attention(q, K, V, 1.0)


def _mutant_transposed_operand(q, K, V, scale):
    return O.decode_attention(q, V, K, scale)  # V used for scores, K for values


def _mutant_missing_last_token(q, K, V, scale):
    return O.decode_attention(q, K[:-1] if len(K) > 1 else K, V[:-1] if len(V) > 1 else V, scale)


def _mutant_unnormalised(q, K, V, scale):
    H_q, d = q.shape
    G = H_q // K.shape[1]
    out = np.zeros((H_q, d))
    for h in range(H_q):
        s = scale * (K[:, h // G] @ q[h])
        out[h] = np.exp(s - s.max()) @ V[:, h // G]
    return out


@pytest.mark.parametrize("mutant", [_mutant_wrong_grouping, _mutant_dropped_scale,
                                    _mutant_transposed_operand, _mutant_missing_last_token,
                                    _mutant_unnormalised])
def test_planted_attention_mistakes_are_caught(mutant):
    assert not _attention_pins_pass(mutant)


def test_planted_locate_mistake_is_caught():
    def bad_locate(row, pos, bs=16):
        return row[pos // bs] * bs + pos // bs  # offset taken from the wrong term
    table = [7, 3, 19, 42]
    mismatches = [(int(p), int(e)) for (p, e), _ in _rows("locate_example.txt")
                  if int(e) >= 0 and bad_locate(table, int(p)) != int(e)]
    assert mismatches


def test_planted_e4m3_rounding_mistake_is_caught():
    mags = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))

    def truncating(x):  # rounds toward zero instead of to nearest
        a = abs(float(x))
        return int(np.searchsorted(mags, a, side="right") - 1)
    x = np.float32(1.0 + 3 * 2.0 ** -5)  # between 1.0625 and 1.125, nearer the upper
    assert truncating(x) != int(O.e4m3_encode(x))
    assert int(O.e4m3_encode(x)) == O.e4m3_encode_bruteforce(float(x))


# ----------------------------------------------------------------------------------
# Chunked prefill (causal attention of several new tokens per sequence)
# ----------------------------------------------------------------------------------
def _sdpa_causal_rows(q_all, K, V, scale, rows):
    """torch SDPA with is_causal over a whole sequence (queries = every position), fp64."""
    n, H_q, d = q_all.shape
    H_kv = K.shape[1]
    G = H_q // H_kv
    qt = torch.from_numpy(q_all).permute(1, 0, 2).unsqueeze(0)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
    return out[0].permute(1, 0, 2).numpy()[rows]


@pytest.mark.parametrize("H_q,H_kv,ctx,first", [(4, 2, 40, 0), (8, 2, 37, 20), (6, 6, 19, 18), (8, 1, 50, 33)])
def test_prefill_matches_causal_sdpa(H_q, H_kv, ctx, first):
    rng = np.random.default_rng(20)
    d = 16
    q_all = rng.standard_normal((ctx, H_q, d))
    K = rng.standard_normal((ctx, H_kv, d))
    V = rng.standard_normal((ctx, H_kv, d))
    got = O.prefill_attention(q_all[first:], K, V, 0.25, first)
    ref = _sdpa_causal_rows(q_all, K, V, 0.25, slice(first, ctx))
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


def test_prefill_last_token_is_decode_and_chunks_compose():
    rng = np.random.default_rng(21)
    q_all = rng.standard_normal((30, 8, 16))
    K = rng.standard_normal((30, 2, 16))
    V = rng.standard_normal((30, 2, 16))
    one = O.prefill_attention(q_all[29:], K, V, 0.3, 29)[0]
    assert np.array_equal(one, O.decode_attention(q_all[29], K, V, 0.3))
    whole = O.prefill_attention(q_all, K, V, 0.3, 0)
    parts = np.concatenate([O.prefill_attention(q_all[a:b], K, V, 0.3, a) for a, b in [(0, 7), (7, 16), (16, 30)]])
    assert np.array_equal(whole, parts)
    # the first position sees only itself
    assert np.array_equal(whole[0], V[0, [0, 0, 0, 0, 1, 1, 1, 1]])


def test_planted_causal_mask_mistake_is_caught():
    rng = np.random.default_rng(22)
    q_all = rng.standard_normal((12, 4, 8))
    K = rng.standard_normal((12, 2, 8))
    V = rng.standard_normal((12, 2, 8))

    def off_by_one(q, K, V, scale, first):  # lets each query see the next key as well
        out = np.zeros(q.shape)
        for i in range(q.shape[0]):
            p = min(first + i + 1, K.shape[0] - 1)
            for h in range(q.shape[1]):
                s = scale * (K[:p + 1, h // 2] @ q[i, h])
                out[i, h] = O.softmax_weights(s) @ V[:p + 1, h // 2]
        return out
    ref = _sdpa_causal_rows(q_all, K, V, 0.5, slice(3, 12))
    assert np.allclose(O.prefill_attention(q_all[3:], K, V, 0.5, 3), ref, atol=1e-12)
    assert not np.allclose(off_by_one(q_all[3:], K, V, 0.5, 3), ref, atol=1e-6)
