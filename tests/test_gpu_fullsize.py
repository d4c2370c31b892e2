"""Full-size workloads in the launch configuration the benchmark times (partition_size 0):
the appended slots are compared bit for bit with the oracle's encoding, and sampled output
rows (sequence, query head) with the oracle computed row by row from the logical token
stream.  Properties that hold at any size are checked on every row."""

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300.workloads import bf16_bits, make_workload

from harness import ATOL_MAX, ATOL_MEAN, GpuState, logical_tokens, reference_row, to_f64, unpack_int4_pool

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _samples(w, n=10, seed=0):
    rng = np.random.default_rng(seed)
    ss = list(rng.integers(0, w.B, n))
    ss += [int(np.argmax(w.ctx_old)), int(np.argmin(w.ctx_old))]
    hs = list(rng.integers(0, w.H_q, n)) + [w.H_q - 1, 0]
    return list(zip(map(int, ss), map(int, hs)))


def _check_appended_slots(g, w, step=0):
    """Every appended token's slot holds the oracle's encoding of its K and V rows."""
    gk, gv, gks, gvs = g.pools()
    if w.k_dtype == "int4":
        n_slots = w.num_blocks * 16
        gk = unpack_int4_pool(gk, n_slots, w.H_kv, w.D, "k")
        gv = unpack_int4_pool(gv, n_slots, w.H_kv, w.D, "v")
    pos = w.positions(step)
    kb, vb = bf16_bits(w.k_new[step]), bf16_bits(w.v_new[step])
    for s in range(w.B):
        p = int(pos[s])
        if p < w.num_sink:
            assert np.array_equal(gks[s, p], kb[s]) and np.array_equal(gvs[s, p], vb[s])
            continue
        slot = O.locate(g.tables[s], p)
        if w.k_dtype == "bf16":
            assert np.array_equal(gk[slot], kb[s]) and np.array_equal(gv[slot], vb[s])
        elif w.k_dtype == "int4":
            for h in range(w.H_kv):
                for pool, bits in ((gk, kb), (gv, vb)):
                    codes, params = O.int4_encode_row(bits[s, h])
                    assert np.array_equal(pool[0][slot, h], codes) and np.array_equal(pool[1][slot, h], params)
        else:
            for h in range(w.H_kv):
                ks = np.float32(w.k_scales[h].item())
                vs = np.float32(w.v_scales[h].item())
                assert np.array_equal(gk[slot, h], O.quantize_row(kb[s, h], ks, "e4m3"))
                assert np.array_equal(gv[slot, h], O.quantize_row(vb[s, h], vs, "int8"))


def _check_rows(out, w, rows):
    errs = []
    for (s, h), ref in rows.items():
        errs.append(np.abs(out[s, h] - ref))
    errs = np.concatenate(errs)
    assert errs.max() <= ATOL_MAX, errs.max()
    assert errs.mean() <= ATOL_MEAN, errs.mean()
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("name", ["8b", "70b", "long_quant", "int4_8b", "swa"])
def test_full_size_step(name):
    w = make_workload(name, steps=1)
    g = GpuState(w)
    out, pairs = g.step(0, partition=0)
    out = to_f64(out)
    assert len(pairs) == 0
    assert g.err_bits() == 0
    _check_appended_slots(g, w)
    rows = {}
    cache = {}
    for s, h in _samples(w):
        if s not in cache:
            cache[s] = logical_tokens(w, s, 0)
        rows[(s, h)] = reference_row(w, s, h, 0, *cache[s])
    _check_rows(out, w, rows)
    # the same inputs through fixed 512-token partitions give the same rows
    out512 = to_f64(g.attend(w.q[0], w.context_lens(0), 512))
    _check_rows(out512, w, rows)
    assert np.abs(out512 - out).max() <= 2e-2


def test_full_size_prefix_fork_and_steady_step():
    w = make_workload("prefix_cow", steps=1)
    g = GpuState(w)
    fork_pos = w.positions(0)  # 1208 for every sequence
    pairs = g.prepare(fork_pos)
    assert len(pairs) == w.B  # every sequence copies the shared, partly filled block
    srcs = set(int(a) for a, _ in pairs)
    assert len(srcs) == 1
    g.append(w.k_new[0], w.v_new[0], fork_pos)
    out_fork = to_f64(g.attend(w.q[0], w.context_lens(0), 0))
    assert g.err_bits() == 0
    # the copies hold the prefix tokens 1200..1207 bit for bit, then the fork token
    gk, gv, _, _ = g.pools()
    pk, pv = bf16_bits(w.fill_k), bf16_bits(w.fill_v)
    for s in range(w.B):
        blk = int(g.tables[s, 75])
        assert np.array_equal(gk[blk * 16:blk * 16 + 8], pk[1200:1208])
        assert np.array_equal(gv[blk * 16:blk * 16 + 8], pv[1200:1208])
        assert np.array_equal(gk[blk * 16 + 8], bf16_bits(w.k_new[0, s]))
    # sampled fork rows: prefix + the fork token
    rows = {}
    for s, h in _samples(w, 6):
        kb = np.concatenate([pk, bf16_bits(w.k_new[0, s:s + 1])])
        vb = np.concatenate([pv, bf16_bits(w.v_new[0, s:s + 1])])
        rows[(s, h)] = reference_row(w, s, h, 0, kb, vb)
    _check_rows(out_fork, w, rows)

    # private suffixes (suffix token 0 was the fork token) and a steady-state step
    seqs, poss, idx = [], [], []
    off = 0
    for s in range(w.B):
        n = int(w.suffix_len[s])
        seqs += [s] * (n - 1)
        poss += range(w.prefix + 1, w.prefix + n)
        idx += range(off + 1, off + n)
        off += n
    for p in range(w.prefix + 1, w.prefix + int(w.suffix_len.max())):
        assert len(g.prepare(np.where(p < w.prefix + w.suffix_len, p, -1).astype(np.int32))) == 0
    idx_t = torch.tensor(idx, dtype=torch.long)
    g.bulk_append(w.suffix_k[idx_t], w.suffix_v[idx_t], np.array(seqs, np.int32), np.array(poss, np.int32))
    steady = (w.prefix + w.suffix_len).astype(np.int32)
    assert len(g.prepare(steady)) == 0
    g.append(w.k_new[0], w.v_new[0], steady)
    out = to_f64(g.attend(w.q[0], steady + 1, 0))
    assert g.err_bits() == 0
    rows = {}
    offs = np.concatenate([[0], np.cumsum(w.suffix_len)])
    for s, h in _samples(w, 8, seed=1):
        sk = bf16_bits(w.suffix_k[offs[s] + 1:offs[s + 1]])
        sv = bf16_bits(w.suffix_v[offs[s] + 1:offs[s + 1]])
        new_k = bf16_bits(w.k_new[0, s:s + 1])
        new_v = bf16_bits(w.v_new[0, s:s + 1])
        kb = np.concatenate([pk, new_k, sk, new_k])
        vb = np.concatenate([pv, new_v, sv, new_v])
        rows[(s, h)] = reference_row(w, s, h, 0, kb, vb)
    _check_rows(out, w, rows)
