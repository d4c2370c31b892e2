"""Full-size workloads in the launch configuration the benchmark times (partition_size 0), through
both entry points the benchmark and a caller use: pa_decode_step (the append and the attention in
one call, what the benchmark times) and the separate pa_kv_append + pa_decode_attention calls.

Every (sequence, query head) row of every workload is compared with the oracle, computed sequence
by sequence from the logical token stream (untitled KV-cache article at ldpk.cn/news/58971 §2.1:
the attention formula; "KV Cache 的显存账本：PagedAttention 与连续批处理" §四: the block table
only places the tokens, so the logical stream fixes the result).  At full size the balanced split
gives every CTA a range of (sequence, block) pairs that crosses sequence boundaries and the
32-entry table chunks of the producer, which the reduced cases never reach.  The appended slots
are compared bit for bit with the oracle's encoding.  Each case prints its max and mean error."""

import os

import numpy as np
import pytest
import torch

import oracle as O
from paged_kv_cache_table_gb300.workloads import bf16_bits, make_workload

from harness import (ATOL_MAX, ATOL_MEAN, GpuState, reference_all, reference_seq, to_f64, unpack_int4_pool,
                     unpack_tok_pool)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_appended_slots(g, w, step=0):
    """Every appended token's slot holds the oracle's encoding of its K and V rows."""
    gk, gv, gks, gvs = g.pools()
    if w.k_dtype == "int4":
        n_slots = w.num_blocks * 16
        gk = unpack_int4_pool(gk, n_slots, w.H_kv, w.D, "k")
        gv = unpack_int4_pool(gv, n_slots, w.H_kv, w.D, "v")
    elif w.k_dtype == "e4m3_tok":
        gk = unpack_tok_pool(gk, w.num_blocks * 16, w.H_kv, w.D)
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
            for pool, bits in ((gk, kb), (gv, vb)):
                codes, params = O.int4_encode_row(bits[s])
                assert np.array_equal(pool[0][slot], codes) and np.array_equal(pool[1][slot], params)
        elif w.k_dtype == "e4m3_tok":
            codes, sc = O.quantize_token_rows(kb[s])
            assert np.array_equal(gk[0][slot], codes) and np.array_equal(gk[1][slot], sc)
            for h in range(w.H_kv):
                vs = np.float32(w.v_scales[h].item())
                assert np.array_equal(gv[slot, h], O.quantize_row(vb[s, h], vs, "int8"))
        else:
            for h in range(w.H_kv):
                ks = np.float32(w.k_scales[h].item())
                vs = np.float32(w.v_scales[h].item())
                assert np.array_equal(gk[slot, h], O.quantize_row(kb[s, h], ks, "e4m3"))
                assert np.array_equal(gv[slot, h], O.quantize_row(vb[s, h], vs, "int8"))


def _check_all_rows(out, ref, what):
    """Every row within the attention tolerances; returns and prints (max, mean) abs error."""
    assert out.shape == ref.shape
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref)
    print(f"[full size] {what}: {out.shape[0] * out.shape[1]} rows, max abs err {err.max():.3e}, "
          f"mean abs err {err.mean():.3e}")
    assert err.max() <= ATOL_MAX, (what, err.max())
    assert err.mean() <= ATOL_MEAN, (what, err.mean())
    return float(err.max()), float(err.mean())


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.parametrize("name", ["8b", "70b", "long_quant", "long_quant_tok", "int4_8b", "swa"])
def test_full_size_every_row(name):
    w = make_workload(name, steps=1)
    # the longest contexts run the oracle's (sequence, KV head) pieces on all host cores; the pool
    # is spawned and closed before the first GPU call
    long_ctx = name.startswith("long_quant")
    ref = reference_all(w, 0, processes=min(32, os.cpu_count() or 1) if long_ctx else 0)
    g = GpuState(w)
    pos, ctx = w.positions(0), w.context_lens(0)
    assert len(g.prepare(pos)) == 0
    # the benchmark's entry point: append + attention in one call
    out_step = g.decode_step(w.k_new[0], w.v_new[0], w.q[0], pos, ctx, partition=0)
    assert g.err_bits() == 0
    _check_appended_slots(g, w)
    _check_all_rows(to_f64(out_step), ref, f"{name} pa_decode_step")
    # the separate calls (the append writes the same bits into the same slots again)
    g.append(w.k_new[0], w.v_new[0], pos)
    out_calls = g.attend(w.q[0], ctx, 0)
    assert g.err_bits() == 0
    assert np.array_equal(_bits(out_calls), _bits(out_step)), "step and separate calls differ"
    # fixed 512-token partitions (the pages' split) give the same rows within the tolerance
    out512 = g.attend(w.q[0], ctx, 512)
    _check_all_rows(to_f64(out512), ref, f"{name} partition 512")
    assert g.err_bits() == 0


def test_full_size_prefix_fork_and_steady_step():
    w = make_workload("prefix_cow", steps=1)
    g = GpuState(w)
    fork_pos = w.positions(0)  # 1208 for every sequence
    pairs = g.prepare(fork_pos)
    assert len(pairs) == w.B  # every sequence copies the shared, partly filled block
    srcs = set(int(a) for a, _ in pairs)
    assert len(srcs) == 1
    out_fork = to_f64(g.decode_step(w.k_new[0], w.v_new[0], w.q[0], fork_pos, w.context_lens(0), partition=0))
    assert g.err_bits() == 0
    # the copies hold the prefix tokens 1200..1207 bit for bit, then the fork token
    gk, gv, _, _ = g.pools()
    pk, pv = bf16_bits(w.fill_k), bf16_bits(w.fill_v)
    for s in range(w.B):
        blk = int(g.tables[s, 75])
        assert np.array_equal(gk[blk * 16:blk * 16 + 8], pk[1200:1208])
        assert np.array_equal(gv[blk * 16:blk * 16 + 8], pv[1200:1208])
        assert np.array_equal(gk[blk * 16 + 8], bf16_bits(w.k_new[0, s]))
    # every fork row: prefix + the fork token
    ref = np.zeros((w.B, w.H_q, w.D))
    for s in range(w.B):
        kb = np.concatenate([pk, bf16_bits(w.k_new[0, s:s + 1])])
        vb = np.concatenate([pv, bf16_bits(w.v_new[0, s:s + 1])])
        ref[s] = reference_seq(w, s, 0, kb, vb)
    _check_all_rows(out_fork, ref, "prefix_cow fork step")

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
    out = g.decode_step(w.k_new[0], w.v_new[0], w.q[0], steady, steady + 1, partition=0)
    assert g.err_bits() == 0
    g.append(w.k_new[0], w.v_new[0], steady)
    out_calls = g.attend(w.q[0], steady + 1, 0)
    assert np.array_equal(_bits(out_calls), _bits(out)), "step and separate calls differ"
    offs = np.concatenate([[0], np.cumsum(w.suffix_len)])
    for s in range(w.B):
        sk = bf16_bits(w.suffix_k[offs[s] + 1:offs[s + 1]])
        sv = bf16_bits(w.suffix_v[offs[s] + 1:offs[s + 1]])
        new_k = bf16_bits(w.k_new[0, s:s + 1])
        new_v = bf16_bits(w.v_new[0, s:s + 1])
        kb = np.concatenate([pk, new_k, sk, new_k])
        vb = np.concatenate([pv, new_v, sv, new_v])
        ref[s] = reference_seq(w, s, 0, kb, vb)
    _check_all_rows(to_f64(out), ref, "prefix_cow steady step")
    # the 75 whole prefix blocks attended once for all sequences (pa_decode_attention_shared)
    out_shared = g.attend_shared(w.q[0], steady + 1, list(range(w.B)), w.prefix - w.prefix % 16)
    assert g.err_bits() == 0
    _check_all_rows(to_f64(out_shared), ref, "prefix_cow shared prefix")

