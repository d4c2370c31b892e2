"""CPU-only checks of the C-ABI library: it builds and loads, exports every symbol the header
declares, rejects bad arguments on the host before touching a GPU, and its host block
manager makes the same decisions as the oracle's block pool."""

import ctypes
import os
import re
import threading

import numpy as np
import pytest

import oracle as O
from paged_kv_cache_table_gb300 import build as B
from paged_kv_cache_table_gb300 import native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    B.build()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "pa.h"), encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    declared = _header_functions()
    assert sorted(N.EXPORTED) == declared
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_header_is_plain_c(tmp_path):
    """include/pa.h is a C header: it compiles as strict C99 on its own (no C++, no CUDA types)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "pa.h"\nint main(void) { pa_cache_desc d; (void)d; return 0; }\n')
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings():
    assert N.status_string(0) == "PA_OK"
    assert N.status_string(3) == "PA_ERR_WORKSPACE_TOO_SMALL"
    assert N.status_string(99) == "PA_ERR_UNKNOWN"


def _desc(**kw):
    base = dict(num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=64, num_blocks=64, max_blocks_per_seq=17)
    base.update(kw)
    return N.make_desc(**base)


FAKE = 1 << 20  # never dereferenced: every call below returns before launching


def _no_gpu():
    try:
        import torch
        return not torch.cuda.is_available()
    except ImportError:
        return True


# Calls with fake device addresses are made only where no GPU is visible: should a host check
# ever go missing, such a call must not reach a device.
host_only = pytest.mark.skipif(not _no_gpu(), reason="fake device addresses: run without a GPU")


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), N.PA_ERR_UNSUPPORTED),
    (dict(block_size=32), N.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=9), N.PA_ERR_INVALID_ARG),
    (dict(num_q_heads=36, num_kv_heads=2), N.PA_ERR_UNSUPPORTED),  # G = 18 > 8
    (dict(num_blocks=0), N.PA_ERR_INVALID_ARG),
    (dict(k_dtype="e4m3", v_dtype="int8", head_dim=128), N.PA_ERR_INVALID_ARG),  # no scales
    (dict(k_dtype="e4m3", v_dtype="int8", head_dim=64, k_scales=FAKE, v_scales=FAKE), N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype="bf16", v_dtype="int8"), N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype=7), N.PA_ERR_INVALID_ARG),
    (dict(num_sink=4), N.PA_ERR_INVALID_ARG),  # sinks without buffers
    # INT4 needs head_dim 128 and an even number of KV heads
    (dict(k_dtype=N.PA_INT4, v_dtype=N.PA_INT4, num_q_heads=6, num_kv_heads=3, head_dim=128), N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype=N.PA_INT4, v_dtype=N.PA_INT4, head_dim=64), N.PA_ERR_UNSUPPORTED),
    # per-token K scales: head_dim 128, KV heads a multiple of 4, V scales required, V INT8 only
    (dict(k_dtype="e4m3_tok", v_dtype="int8", head_dim=128, num_kv_heads=4), N.PA_ERR_INVALID_ARG),
    (dict(k_dtype="e4m3_tok", v_dtype="int8", head_dim=64, v_scales=FAKE), N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype="e4m3_tok", v_dtype="int8", head_dim=128, num_q_heads=12, num_kv_heads=6, v_scales=FAKE),
     N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype="e4m3_tok", v_dtype="bf16", head_dim=128, v_scales=FAKE), N.PA_ERR_UNSUPPORTED),
    (dict(k_dtype="int8", v_dtype="e4m3_tok"), N.PA_ERR_UNSUPPORTED),
])
@host_only
def test_bad_descriptions_are_rejected_on_the_host(kw, status):
    d = _desc(**kw)
    with pytest.raises(N.PaError) as e:
        N.pa_kv_append(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0)
    assert e.value.status == status
    with pytest.raises(N.PaError) as e:
        N.pa_block_copy(d, FAKE, FAKE, FAKE, 1, None, 0)
    assert e.value.status == status
    assert N.pa_decode_workspace_size(d, 100, 32) == 0


@host_only
def test_null_and_misaligned_pointers_are_rejected():
    d = _desc()
    with pytest.raises(N.PaError) as e:
        N.pa_kv_append(d, 0, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0)
    assert e.value.status == N.PA_ERR_INVALID_ARG
    with pytest.raises(N.PaError) as e:
        N.pa_kv_append(d, FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0)
    assert e.value.status == N.PA_ERR_INVALID_ARG
    with pytest.raises(N.PaError) as e:
        N.pa_kv_append_tokens(d, FAKE, FAKE, FAKE, FAKE, 3, 0, FAKE, FAKE, None, 0)
    assert e.value.status == N.PA_ERR_INVALID_ARG
    with pytest.raises(N.PaError) as e:
        N.pa_block_copy(d, FAKE, FAKE, FAKE, -1, None, 0)
    assert e.value.status == N.PA_ERR_INVALID_ARG
    # zero rows / pairs: nothing to enqueue
    N.pa_kv_append_tokens(d, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE, None, 0)
    N.pa_block_copy(d, FAKE, FAKE, 0, 0, None, 0)


@host_only
def test_step_and_prefill_calls_reject_bad_arguments_on_the_host():
    """The combined calls check every argument (attention and append alike) before anything is
    enqueued; every call below returns from those checks (no device work, no CUDA call)."""
    nan = float("nan")
    pf = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128)
    # pa_prefill_step(desc, out, q, k, v, k_new, v_new, n, seq, pos, tables, q_start, ctx, max_q, scale)
    good = dict(out=FAKE, q=FAKE, k_new=FAKE, v_new=FAKE, n=5, seq=FAKE, pos=FAKE, max_q=16, scale=0.1)
    bad = [
        (dict(scale=nan), N.PA_ERR_INVALID_ARG),
        (dict(max_q=-1), N.PA_ERR_INVALID_ARG),
        (dict(out=0), N.PA_ERR_INVALID_ARG),
        (dict(q=FAKE + 8), N.PA_ERR_INVALID_ARG),
        (dict(k_new=0), N.PA_ERR_INVALID_ARG),      # an append argument
        (dict(seq=0), N.PA_ERR_INVALID_ARG),
        (dict(n=-1), N.PA_ERR_INVALID_ARG),
    ]
    for kw, status in bad:
        a = dict(good, **kw)
        with pytest.raises(N.PaError) as e:
            N.pa_prefill_step(pf, a["out"], a["q"], FAKE, FAKE, a["k_new"], a["v_new"], a["n"], a["seq"], a["pos"],
                              FAKE, FAKE, FAKE, a["max_q"], a["scale"], None, 0)
        assert e.value.status == status, kw
    # quantised and sink-holding caches take the same argument checks (every cache kind is served)
    quant = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, k_dtype="e4m3", v_dtype="int8",
                  k_scales=FAKE, v_scales=FAKE)
    int4 = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, k_dtype="int4", v_dtype="int4")
    sinks = _desc(num_sink=4, k_sink=FAKE, v_sink=FAKE)
    for d in (quant, int4, sinks):
        for call in (lambda d: N.pa_prefill_step(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 5, FAKE, FAKE, FAKE, FAKE,
                                                 FAKE, 16, nan, None, 0),
                     lambda d: N.pa_prefill_attention(d, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, nan, None, 0),
                     lambda d: N.pa_prefill_attention(d, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 0.1, None, 0)):
            with pytest.raises(N.PaError) as e:
                call(d)
            assert e.value.status == N.PA_ERR_INVALID_ARG
    # pa_decode_step with fixed partitions (its plan needs no device query)
    dd = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_seqs=4)
    ws = N.pa_decode_workspace_size(dd, 1000, 512)
    assert ws > 0
    ws_ptr = 1 << 24  # 256-byte aligned
    # pa_decode_step(desc, out, q, k, v, k_new, v_new, tables, positions, ctx, max_ctx, scale, part, ws, bytes)
    good = dict(q=FAKE, pos=FAKE, scale=0.1, part=512, ws=ws_ptr, nbytes=ws, k_new=FAKE)
    bad = [
        (dict(scale=nan), N.PA_ERR_INVALID_ARG),
        (dict(pos=0), N.PA_ERR_INVALID_ARG),
        (dict(q=FAKE + 8), N.PA_ERR_INVALID_ARG),
        (dict(part=100), N.PA_ERR_INVALID_ARG),     # not a multiple of 16
        (dict(ws=ws_ptr + 16), N.PA_ERR_INVALID_ARG),
        (dict(nbytes=ws - 1), N.PA_ERR_WORKSPACE_TOO_SMALL),
        (dict(k_new=0), N.PA_ERR_INVALID_ARG),      # an append argument
    ]
    for kw, status in bad:
        a = dict(good, **kw)
        with pytest.raises(N.PaError) as e:
            N.pa_decode_step(dd, FAKE, a["q"], FAKE, FAKE, a["k_new"], FAKE, FAKE, a["pos"], FAKE, 1000, a["scale"],
                             a["part"], a["ws"], a["nbytes"], None, 0)
        assert e.value.status == status, kw


def test_workspace_size_fixed_partitions():
    d = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_seqs=64)
    a = N.pa_decode_workspace_size(d, 4096, 512)
    b = N.pa_decode_workspace_size(d, 4096, 256)
    c = N.pa_decode_workspace_size(d, 8192, 512)
    assert 0 < a < b and c == 2 * a - 256  # partials scale with the partition count; 256-byte header
    assert N.pa_decode_workspace_size(d, 4096, 24) == 0  # not a multiple of 16
    assert N.pa_decode_workspace_size(d, -1, 512) == 0


# ----------------------------------------------------------------------------------
# host block manager vs the oracle's pool
# ----------------------------------------------------------------------------------
def test_block_manager_matches_oracle_pool_on_random_operations():
    rng = np.random.default_rng(0)
    bm = N.BlockManager(48)
    pool = O.BlockPool(48)
    live = []
    for _ in range(4000):
        op = rng.integers(5)
        if op == 0:
            a, b = bm.alloc(), pool.alloc()
            assert a == b
            if a >= 0:
                live.append(a)
        elif op == 1 and live:
            x = int(rng.choice(live))
            assert bm.incref(x) == pool.incref(x)
        elif op == 2 and live:
            x = int(rng.choice(live))
            r = bm.decref(x)
            assert r == pool.decref(x)
            if r == 0:
                live.remove(x)
        elif op == 3:
            x = int(rng.integers(-2, 50))
            assert bm.claim(x) == pool.claim(x)
            if 0 <= x < 48 and x not in live and pool.refcount[x] == 1:
                live.append(x)
        else:
            x = int(rng.integers(-2, 50))
            assert bm.refcount(x) == (int(pool.refcount[x]) if 0 <= x < 48 else -1)
        assert bm.num_free() == pool.num_free()


def test_prepare_step_matches_oracle_prepare_append():
    rng = np.random.default_rng(1)
    B_, M = 6, 12
    bm = N.BlockManager(80)
    pool = O.BlockPool(80)
    tabs = np.full((B_, M), -1, dtype=np.int32)
    otabs = np.full((B_, M), -1, dtype=np.int64)
    lens = np.zeros(B_, dtype=np.int64)
    for step in range(120):
        pos = np.where(rng.random(B_) < 0.8, lens, -1).astype(np.int32)
        pairs, changed = bm.prepare_step(tabs, pos)
        opairs = []
        n_changed = 0
        for s in range(B_):
            if pos[s] >= 0:
                act = pool.prepare_append(otabs[s], int(pos[s]))
                if act[0] == "copy":
                    opairs.append((act[1], act[2]))
                if act[0] != "ok":
                    n_changed += 1
        assert [tuple(p) for p in pairs.tolist()] == opairs
        assert changed == n_changed
        assert np.array_equal(tabs, otabs)
        lens += pos >= 0
        if step % 30 == 29:  # fork sequence 0 into 1 and 2 (prefix sharing), then diverge
            for dst in (1, 2):
                bm.release(tabs[dst], M)
                pool.release(otabs[dst], M)
                n = -(-int(lens[0]) // 16)
                tabs[dst] = bm.fork(tabs[0], n)
                otabs[dst] = pool.fork(otabs[0], n)
                lens[dst] = lens[0]
        assert bm.num_free() == pool.num_free()


@pytest.mark.parametrize("window", [1, 16, 37, 100])
def test_slide_window_matches_oracle_pool(window):
    """Sequences that decode, fork (shared prefixes) and slide their window: the library's
    release decisions, tables, refcounts and free list follow the oracle's slide_window."""
    rng = np.random.default_rng(window)
    B_, M = 5, 40
    bm = N.BlockManager(200)
    pool = O.BlockPool(200)
    tabs = np.full((B_, M), -1, dtype=np.int32)
    otabs = np.full((B_, M), -1, dtype=np.int64)
    lens = np.zeros(B_, dtype=np.int64)
    for step in range(500):
        pos = np.where(rng.random(B_) < 0.9, lens, -1).astype(np.int32)
        bm.prepare_step(tabs, pos)
        for s in range(B_):
            if pos[s] >= 0:
                pool.prepare_append(otabs[s], int(pos[s]))
        lens += pos >= 0
        released, freed = bm.slide_window(tabs, lens.astype(np.int32), window)
        o_before = int((otabs >= 0).sum())
        o_freed = sum(pool.slide_window(otabs[s], int(lens[s]), window) for s in range(B_))
        assert released == o_before - int((otabs >= 0).sum())
        assert freed == o_freed
        assert np.array_equal(tabs, otabs)
        assert bm.num_free() == pool.num_free()
        if step == 250:  # sequences 1 and 2 fork sequence 0's live blocks (shared, refcount 3)
            for dst in (1, 2):
                bm.release(tabs[dst], M)
                pool.release(otabs[dst], M)
                n = -(-int(lens[0]) // 16)
                live = np.nonzero(otabs[0][:n] >= 0)[0]
                for lb in live:
                    tabs[dst][lb] = tabs[0][lb]
                    bm.incref(int(tabs[0][lb]))
                    otabs[dst][lb] = otabs[0][lb]
                    pool.incref(int(otabs[0][lb]))
                lens[dst] = lens[0]
            assert np.array_equal(tabs, otabs)
    for b in range(200):
        assert bm.refcount(b) == pool.refcount[b]
    assert bm.slide_window(tabs, lens.astype(np.int32), 0) == (0, 0)


def test_slide_window_rejects_bad_arguments_and_foreign_blocks():
    bm = N.BlockManager(8)
    tabs = np.full((1, 4), -1, dtype=np.int32)
    with pytest.raises(N.PaError):
        bm.slide_window(tabs, np.array([40], dtype=np.int32), -1)
    tabs[0, 0] = 3  # the pool never handed out block 3
    with pytest.raises(N.PaError):
        bm.slide_window(tabs, np.array([40], dtype=np.int32), 8)


def test_prepare_step_out_of_blocks_and_bad_position():
    bm = N.BlockManager(2)
    tabs = np.full((3, 4), -1, dtype=np.int32)
    with pytest.raises(N.PaError) as e:
        bm.prepare_step(tabs, np.array([0, 0, 0], dtype=np.int32))
    assert e.value.status == N.PA_ERR_OUT_OF_BLOCKS
    assert list(tabs[:, 0]) == [0, 1, -1]  # rows before the failure keep their blocks
    with pytest.raises(N.PaError) as e:
        bm.prepare_step(tabs, np.array([64, -1, -1], dtype=np.int32))
    assert e.value.status == N.PA_ERR_INVALID_ARG


def test_block_manager_is_thread_safe():
    bm = N.BlockManager(4096)
    base = [bm.alloc() for _ in range(64)]
    errors = []

    def worker(seed):
        rng = np.random.default_rng(seed)
        mine = []
        try:
            for _ in range(3000):
                if rng.random() < 0.5 or not mine:
                    b = int(base[rng.integers(len(base))])
                    bm.incref(b)
                    mine.append(b)
                else:
                    bm.decref(mine.pop())
            for b in mine:
                bm.decref(b)
        except Exception as ex:  # pragma: no cover
            errors.append(ex)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors
    assert all(bm.refcount(b) == 1 for b in base)
    assert bm.num_free() == 4096 - 64


def test_release_frees_only_unshared_blocks_and_nothing_leaks():
    bm = N.BlockManager(32)
    row = np.full(8, -1, dtype=np.int32)
    for p in range(100):
        bm.prepare_step(row[None, :], np.array([p], dtype=np.int32))
    assert bm.num_free() == 32 - 7
    fork = bm.fork(row, 7)
    assert bm.release(row, 8) == 0  # still held by the fork
    assert bm.release(fork, 8) == 7
    assert bm.num_free() == 32


def test_prefill_workspace_size():
    """The decoded bf16 copy of pa_prefill_attention_ws: a dense table of num_seqs x ceil(max_ctx/16)
    int32 entries (rounded up to 256 bytes), then K and V pools of that many 16-slot bf16 blocks;
    none for caches and shapes that keep the plain path."""
    quant = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, k_dtype="e4m3", v_dtype="int8", k_scales=FAKE,
                 v_scales=FAKE, max_blocks_per_seq=100)
    mb = (1000 + 15) // 16
    table = (4 * mb * 4 + 255) // 256 * 256
    pool = 4 * mb * 16 * 8 * 128 * 2
    assert N.pa_prefill_workspace_size(_desc(**quant), 1000) == table + 2 * pool
    assert N.pa_prefill_workspace_size(_desc(**quant), 0) == 256 + 2 * 4 * 16 * 8 * 128 * 2  # one block each
    int4 = dict(quant, k_dtype="int4", v_dtype="int4", k_scales=None, v_scales=None)
    tok = dict(quant, k_dtype="e4m3_tok", k_scales=None)
    sinks = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, num_sink=4, k_sink=FAKE, v_sink=FAKE,
                 max_blocks_per_seq=100)
    for kw in (int4, tok, sinks):
        assert N.pa_prefill_workspace_size(_desc(**kw), 1000) == table + 2 * pool
    # the plain path: bf16 without sinks, head_dim 64, G not a power of two
    assert N.pa_prefill_workspace_size(_desc(num_q_heads=32, num_kv_heads=8, head_dim=128), 1000) == 0
    assert N.pa_prefill_workspace_size(_desc(num_sink=4, k_sink=FAKE, v_sink=FAKE), 200) == 0
    assert N.pa_prefill_workspace_size(_desc(**dict(quant, num_q_heads=24)), 1000) == 0
    # invalid: max_context_len beyond the table, negative, or a bad description
    assert N.pa_prefill_workspace_size(_desc(**quant), 100 * 16 + 1) == 0
    assert N.pa_prefill_workspace_size(_desc(**quant), -1) == 0
    assert N.pa_prefill_workspace_size(_desc(**dict(quant, k_scales=None)), 1000) == 0


@host_only
def test_prefill_ws_rejects_bad_arguments_on_the_host():
    quant = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, k_dtype="e4m3", v_dtype="int8", k_scales=FAKE,
                  v_scales=FAKE, max_blocks_per_seq=100)
    need = N.pa_prefill_workspace_size(quant, 1000)
    ws = 1 << 24  # 256-byte aligned
    # pa_prefill_attention_ws(desc, out, q, k, v, tables, q_start, ctx, max_q, max_ctx, scale, ws, bytes)
    good = dict(out=FAKE, max_q=16, max_ctx=1000, scale=0.1, ws=ws, nbytes=need)
    bad = [
        (dict(scale=float("nan")), N.PA_ERR_INVALID_ARG),
        (dict(out=0), N.PA_ERR_INVALID_ARG),
        (dict(max_ctx=-1), N.PA_ERR_INVALID_ARG),
        (dict(max_ctx=100 * 16 + 1), N.PA_ERR_INVALID_ARG),
        (dict(ws=0), N.PA_ERR_INVALID_ARG),
        (dict(ws=ws + 128), N.PA_ERR_INVALID_ARG),
        (dict(nbytes=need - 1), N.PA_ERR_WORKSPACE_TOO_SMALL),
    ]
    for kw, status in bad:
        a = dict(good, **kw)
        with pytest.raises(N.PaError) as e:
            N.pa_prefill_attention_ws(quant, a["out"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["max_q"], a["max_ctx"],
                                      a["scale"], a["ws"], a["nbytes"], None, 0)
        assert e.value.status == status, kw
    # nothing to do (no query rows): checked, then nothing enqueued
    N.pa_prefill_attention_ws(quant, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 1000, 0.1, ws, need, None, 0)


@host_only
def test_prefill_step_ws_checks_every_argument_first():
    """The step form checks the attention's workspace and bounds and the append's arguments
    before it enqueues the append."""
    quant = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, k_dtype="e4m3", v_dtype="int8", k_scales=FAKE,
                  v_scales=FAKE, max_blocks_per_seq=100)
    need = N.pa_prefill_workspace_size(quant, 1000)
    ws = 1 << 24
    # pa_prefill_step_ws(desc, out, q, k, v, k_new, v_new, n, seq, pos, tables, q_start, ctx, max_q, max_ctx,
    #                    scale, ws, bytes)
    good = dict(k_new=FAKE, n=5, max_ctx=1000, ws=ws, nbytes=need, scale=0.1)
    bad = [
        (dict(max_ctx=100 * 16 + 1), N.PA_ERR_INVALID_ARG),
        (dict(ws=ws + 64), N.PA_ERR_INVALID_ARG),
        (dict(nbytes=need - 1), N.PA_ERR_WORKSPACE_TOO_SMALL),
        (dict(k_new=0), N.PA_ERR_INVALID_ARG),      # an append argument
        (dict(n=-1), N.PA_ERR_INVALID_ARG),
        (dict(scale=float("nan")), N.PA_ERR_INVALID_ARG),
    ]
    for kw, status in bad:
        a = dict(good, **kw)
        with pytest.raises(N.PaError) as e:
            N.pa_prefill_step_ws(quant, FAKE, FAKE, FAKE, FAKE, a["k_new"], FAKE, a["n"], FAKE, FAKE, FAKE, FAKE,
                                 FAKE, 16, a["max_ctx"], a["scale"], a["ws"], a["nbytes"], None, 0)
        assert e.value.status == status, kw


def test_shared_decode_workspace_size():
    """The decode workspace, then one int32 flag per sequence, then the prefix's partial rows:
    num_seqs x ceil(shared_len / 128) x num_q_heads rows of head_dim + 4 floats, each part
    256-byte aligned."""
    d = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_seqs=64, max_blocks_per_seq=300)
    for part in (512, 256):
        dec = N.pa_decode_workspace_size(d, 4096, part)
        flags = (64 * 4 + 255) // 256 * 256
        up = (dec + 255) // 256 * 256
        for shared_len, chunks in ((0, 0), (16, 1), (128, 1), (1200, 10), (4096, 32)):
            rows = 64 * chunks * 32 * (128 + 4) * 4
            assert N.pa_decode_shared_workspace_size(d, 4096, part, shared_len) == up + flags + rows
    # shared_len not a multiple of 16, negative, or beyond max_context_len; a bad partition
    for bad in (24, -16, 4096 + 16):
        assert N.pa_decode_shared_workspace_size(d, 4096, 512, bad) == 0
    assert N.pa_decode_shared_workspace_size(d, 4096, 24, 1200) == 0


@host_only
def test_shared_decode_rejects_bad_arguments_on_the_host():
    d = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_seqs=8, max_blocks_per_seq=100)
    need = N.pa_decode_shared_workspace_size(d, 1000, 512, 512)
    ws = 1 << 24
    # pa_decode_attention_shared(desc, out, q, k, v, tables, ctx, max_ctx, scale, partition, seqs, n_shared,
    #                            shared_len, ws, bytes)
    good = dict(out=FAKE, max_ctx=1000, scale=0.1, seqs=FAKE, n=4, L=512, ws=ws, nbytes=need)
    bad = [
        (dict(scale=float("nan")), N.PA_ERR_INVALID_ARG),
        (dict(out=0), N.PA_ERR_INVALID_ARG),
        (dict(L=520), N.PA_ERR_INVALID_ARG),       # not a multiple of 16
        (dict(L=1008), N.PA_ERR_INVALID_ARG),      # beyond max_context_len
        (dict(L=-16), N.PA_ERR_INVALID_ARG),
        (dict(n=9), N.PA_ERR_INVALID_ARG),         # more than num_seqs
        (dict(n=-1), N.PA_ERR_INVALID_ARG),
        (dict(seqs=0), N.PA_ERR_INVALID_ARG),      # a list is needed when n_shared > 0
        (dict(ws=ws + 128), N.PA_ERR_INVALID_ARG),
        (dict(nbytes=need - 1), N.PA_ERR_WORKSPACE_TOO_SMALL),
    ]
    for kw, status in bad:
        a = dict(good, **kw)
        with pytest.raises(N.PaError) as e:
            N.pa_decode_attention_shared(d, a["out"], FAKE, FAKE, FAKE, FAKE, FAKE, a["max_ctx"], a["scale"], 512,
                                         a["seqs"], a["n"], a["L"], a["ws"], a["nbytes"], None, 0)
        assert e.value.status == status, kw
    # caches the shared path does not serve
    quant = _desc(num_q_heads=32, num_kv_heads=8, head_dim=128, num_seqs=8, max_blocks_per_seq=100,
                  k_dtype="e4m3", v_dtype="int8", k_scales=FAKE, v_scales=FAKE)
    sinks = _desc(num_seqs=8, max_blocks_per_seq=100, num_sink=4, k_sink=FAKE, v_sink=FAKE)
    window = _desc(num_seqs=8, max_blocks_per_seq=100, sliding_window=256)
    for dd in (quant, sinks, window):
        with pytest.raises(N.PaError) as e:
            N.pa_decode_attention_shared(dd, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1000, 0.1, 512, FAKE, 4, 512, ws,
                                         1 << 30, None, 0)
        assert e.value.status == N.PA_ERR_UNSUPPORTED
