"""CPU tests of the C ABI: the library loads, exports every entry point that
include/kvarn.h declares, validates arguments on the host, and keeps the cache
bookkeeping right (region rules of anbeeld.com "KVarN KV Cache: Implementation and
Benchmarks", 2.1). No kernel is launched: caches here use KVARN_FLAG_HOST_ONLY."""
import os
import re

import pytest

from quantized_kv_cache_seal_gb300 import kvarn as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 1 << 30  # a device address that is never dereferenced in host-only mode


def header_functions():
    text = open(os.path.join(ROOT, "include", "kvarn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvarn_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    L = K.load()
    names = header_functions()
    assert len(names) >= 15
    missing = [n for n in names if not hasattr(L, n)]
    assert missing == []
    assert sorted(K.EXPORTS) == names


def host_cache(**kw):
    args = dict(num_layers=2, max_seqs=4, num_q_heads=8, num_kv_heads=2, max_seq_len=2048,
                flags=K.KVARN_FLAG_HOST_ONLY)
    args.update(kw)
    cfg = K.make_config(**args)
    n = K.kvarn_cache_required_bytes(cfg)
    return K.kvarn_cache_create(cfg, FAKE, n), cfg


def test_status_strings_and_record_sizes():
    assert K.kvarn_status_string(0) == "ok"
    assert K.kvarn_status_string(3) == "capacity exceeded"
    for b in (2, 3, 4, 5, 6, 8):
        assert K.kvarn_record_bytes(b) == 528 + 2048 * b
    for b in (0, 1, 7, 9, 16):
        assert K.kvarn_record_bytes(b) == 0


@pytest.mark.parametrize("kb,vb,ok", [(3, 3, True), (5, 5, True), (6, 6, True), (2, 8, True), (8, 4, True),
                                      (6, 5, True), (5, 4, True), (3, 2, True),
                                      (2, 3, False), (5, 6, False), (4, 6, False), (7, 7, False), (3, 4, False)])
def test_width_pairs(kb, vb, ok):
    """K/V widths: 2, 4 and 8 in any pair; 3, 5 and 6 symmetric; the presets K6/V5,
    K5/V4 and K3/V2 (anbeeld.com section 6)."""
    cfg = K.make_config(k_bits=kb, v_bits=vb, flags=K.KVARN_FLAG_HOST_ONLY)
    if ok:
        assert K.kvarn_cache_required_bytes(cfg) > 0
    else:
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_cache_required_bytes(cfg)
        assert e.value.status == 1


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("group_size", 64), ("sink_tokens", 0),
                                         ("k_bits", 7), ("v_bits", 1), ("num_q_heads", 24),
                                         ("sinkhorn_iters", -1), ("max_seq_len", 0)])
def test_bad_config_rejected(field, value):
    cfg = K.make_config(flags=K.KVARN_FLAG_HOST_ONLY)
    setattr(cfg, field, value)
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_cache_required_bytes(cfg)
    assert e.value.status == 1


def test_create_checks_size_and_alignment():
    cfg = K.make_config(max_seqs=2, max_seq_len=1024, flags=K.KVARN_FLAG_HOST_ONLY)
    n = K.kvarn_cache_required_bytes(cfg)
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_cache_create(cfg, FAKE, n - 1)
    assert e.value.status == 2
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_cache_create(cfg, FAKE + 16, n)
    assert e.value.status == 1


def test_seal_timing_and_regions_streaming():
    """A group seals exactly when its 128th token arrives; tail grows 0..127."""
    h, cfg = host_cache()
    for n in range(1, 600):
        K.kvarn_decode_step(h, 0, [1], FAKE, FAKE, FAKE, FAKE, 0.1)
        assert K.kvarn_seq_length(h, 0, 1) == n
        s = K.kvarn_cache_stats(h)
        sealed = max(n - 128, 0) // 128
        assert s.pool_slots_used == sealed
        assert s.sealed_tokens == 128 * sealed
        assert s.exact_tokens == n - 128 * sealed
        for g in range(sealed):
            K.kvarn_group_record(h, 0, 1, g, 0, 0)
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_group_record(h, 0, 1, sealed, 0, 0)
        assert e.value.status == 5
    assert K.kvarn_seq_length(h, 1, 1) == 0  # other layer untouched


@pytest.mark.parametrize("floor", [1, 3])
def test_tail_floor_seal_timing_streaming_and_bulk(floor):
    """With a tail floor of F groups (anbeeld.com 2.1, BeeLlama's F = 1) group g seals
    when group g + F fills: decode steps and a bulk append agree, and once the body has
    started at least 128 F recent tokens stay exact."""
    h, cfg = host_cache(tail_floor=floor)
    for n in range(1, 128 + 128 * (floor + 2) + 3):
        K.kvarn_decode_step(h, 0, [1], FAKE, FAKE, FAKE, FAKE, 0.1)
        s = K.kvarn_cache_stats(h)
        sealed = max(max(n - 128, 0) // 128 - floor, 0)
        assert s.pool_slots_used == sealed
        assert s.sealed_tokens == 128 * sealed
        assert s.exact_tokens == n - 128 * sealed
        if n >= 128 + 128 * floor:
            assert s.exact_tokens - 128 >= 128 * floor
        for g in range(sealed):
            K.kvarn_group_record(h, 0, 1, g, 0, 0)
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_group_record(h, 0, 1, sealed, 0, 0)
        assert e.value.status == 5
    K.kvarn_append(h, 0, [2], [n], FAKE, FAKE)
    assert K.kvarn_cache_stats(h).pool_slots_used == 2 * sealed


def test_tail_floor_config_and_ring_size():
    for bad in (-1, 4):
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_cache_required_bytes(K.make_config(flags=K.KVARN_FLAG_HOST_ONLY, tail_floor=bad))
        assert e.value.status == 1
    base = K.make_config(max_seqs=2, max_seq_len=4096, pool_groups=8, flags=K.KVARN_FLAG_HOST_ONLY)
    one = K.make_config(max_seqs=2, max_seq_len=4096, pool_groups=8, flags=K.KVARN_FLAG_HOST_ONLY, tail_floor=1)
    # one more 128-row group of fp16 K and V per (sequence, KV head): 2 * 8 * 128 * 128 * 2 * 2 bytes
    grow = K.kvarn_cache_required_bytes(one) - K.kvarn_cache_required_bytes(base)
    assert 2 * 8 * 128 * 128 * 2 * 2 <= grow <= 2 * 8 * 128 * 128 * 2 * 2 + 2 * 256


def test_bulk_append_equals_streaming_bookkeeping():
    h, _ = host_cache()
    K.kvarn_append(h, 0, [0, 2], [700, 129], FAKE, FAKE)
    assert K.kvarn_seq_length(h, 0, 0) == 700 and K.kvarn_seq_length(h, 0, 2) == 129
    s = K.kvarn_cache_stats(h)
    assert s.pool_slots_used == (700 - 128) // 128 + (129 - 128) // 128
    K.kvarn_seq_release(h, 0)
    assert K.kvarn_seq_length(h, 0, 0) == 0
    assert K.kvarn_cache_stats(h).pool_slots_used == 0


def test_capacity_errors_leave_state_unchanged():
    h, _ = host_cache(pool_groups=3, max_seq_len=1024)
    K.kvarn_append(h, 0, [0], [128 + 2 * 128], FAKE, FAKE)
    before = (K.kvarn_seq_length(h, 0, 0), K.kvarn_cache_stats(h).pool_slots_used)
    with pytest.raises(K.KVarNError) as e:       # needs 2 more slots, 1 left
        K.kvarn_append(h, 0, [0], [256], FAKE, FAKE)
    assert e.value.status == 3
    with pytest.raises(K.KVarNError) as e:       # longer than max_seq_len
        K.kvarn_append(h, 0, [1], [1025], FAKE, FAKE)
    assert e.value.status == 3
    assert (K.kvarn_seq_length(h, 0, 0), K.kvarn_cache_stats(h).pool_slots_used) == before
    # a decode step that would need a slot when none is left
    K.kvarn_append(h, 0, [1], [128 + 127], FAKE, FAKE)      # takes the last slot? no: 0 sealed
    K.kvarn_append(h, 1, [1], [128 + 128], FAKE, FAKE)      # takes the third slot
    assert K.kvarn_cache_stats(h).pool_slots_used == 3
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_decode_step(h, 0, [1], FAKE, FAKE, FAKE, FAKE, 0.1)
    assert e.value.status == 3
    assert K.kvarn_seq_length(h, 0, 1) == 255


def test_argument_validation():
    h, _ = host_cache()
    for args in ([h, 2, [0], [1], FAKE, FAKE], [h, 0, [4], [1], FAKE, FAKE], [h, 0, [0, 0], [1, 1], FAKE, FAKE],
                 [h, 0, [0], [-1], FAKE, FAKE], [h, 0, [0], [5], 0, FAKE]):
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_append(*args)
        assert e.value.status == 1
    with pytest.raises(K.KVarNError):
        K.kvarn_decode_attention(h, 0, [0], FAKE, FAKE, float("nan"))
    with pytest.raises(K.KVarNError):
        K.kvarn_seq_length(h, 0, 9)


def test_prefill_argument_checks_and_fused_bookkeeping():
    """kvarn_prefill_attention: q_lens within 0..length, pointers present when any query
    row exists, finite scale; nothing changes on a rejected call. kvarn_prefill appends
    first (sealing the groups the chunk completes) and checks q_lens against the
    extended length; a rejected fused call appends nothing."""
    h, _ = host_cache()
    K.kvarn_append(h, 0, [0], [300], FAKE, FAKE)
    K.kvarn_prefill_attention(h, 0, [0], [300], FAKE, FAKE, 0.1)   # every token's query
    K.kvarn_prefill_attention(h, 0, [0], [0], 0, 0, 0.1)           # no rows: no pointers needed
    K.kvarn_prefill_attention(h, 0, [0, 1], [1, 0], FAKE, FAKE, 0.1)
    for args in ([h, 0, [0], [301], FAKE, FAKE, 0.1], [h, 0, [0], [-1], FAKE, FAKE, 0.1],
                 [h, 0, [0], [5], 0, FAKE, 0.1], [h, 0, [0], [5], FAKE, 0, 0.1],
                 [h, 0, [0], [5], FAKE, FAKE, float("inf")], [h, 0, [0, 0], [1, 1], FAKE, FAKE, 0.1],
                 [h, 0, [1], [1], FAKE, FAKE, 0.1]):
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_prefill_attention(*args)
        assert e.value.status == 1
    K.kvarn_prefill(h, 0, [1], [128 + 256 + 5], FAKE, FAKE, FAKE, FAKE, 0.1)
    assert K.kvarn_seq_length(h, 0, 1) == 128 + 256 + 5
    assert K.kvarn_cache_stats(h).pool_slots_used == 1 + 2  # seq 0: group 0; seq 1: groups 0, 1
    with pytest.raises(K.KVarNError):
        K.kvarn_prefill(h, 0, [2], [10], FAKE, FAKE, FAKE, FAKE, float("nan"))
    with pytest.raises(K.KVarNError):
        K.kvarn_prefill(h, 0, [2], [10], FAKE, FAKE, 0, FAKE, 0.1)
    assert K.kvarn_seq_length(h, 0, 2) == 0


def test_prefill_batch_limit():
    """Up to 256 sequences per prefill call (the kernel parameter table); one more is a
    capacity error, not a launch."""
    h, _ = host_cache(max_seqs=300, num_layers=1, max_seq_len=256, pool_groups=8)
    ids = list(range(256))
    K.kvarn_append(h, 0, ids, [3] * 256, FAKE, FAKE)
    K.kvarn_prefill_attention(h, 0, ids, [3] * 256, FAKE, FAKE, 0.1)
    K.kvarn_append(h, 0, [256], [2], FAKE, FAKE)
    with pytest.raises(K.KVarNError) as e:
        K.kvarn_prefill_attention(h, 0, ids + [256], [1] * 257, FAKE, FAKE, 0.1)
    assert e.value.status == 3


def _snapshot(h):
    import numpy as np
    n = K.kvarn_snapshot_bytes(h)
    buf = np.zeros(n, np.uint8)
    K.kvarn_snapshot_save(h, buf, n)
    return buf


def _state(h, cfg):
    """Lengths, slots used and the record pointer offsets of every sealed group."""
    lens = [[K.kvarn_seq_length(h, l, s) for s in range(cfg.max_seqs)] for l in range(cfg.num_layers)]
    recs = []
    for l in range(cfg.num_layers):
        for s in range(cfg.max_seqs):
            for g in range(max(lens[l][s] - 128, 0) // 128 - cfg.tail_floor):
                recs.append(K.kvarn_group_record(h, l, s, g, 1, 1)[0] - FAKE)
    return lens, K.kvarn_cache_stats(h).pool_slots_used, recs


@pytest.mark.parametrize("floor", [0, 1])
def test_snapshot_round_trip_of_the_bookkeeping(floor):
    """A snapshot restored into a fresh cache of the same configuration reproduces the
    lengths, the slots in use and every group's record address; later appends then seal
    into the lowest free slots."""
    h, cfg = host_cache(tail_floor=floor, pool_groups=64)
    K.kvarn_append(h, 0, [0, 2], [700, 300], FAKE, FAKE)
    K.kvarn_append(h, 1, [1], [1000], FAKE, FAKE)
    for _ in range(130):
        K.kvarn_decode_step(h, 0, [0, 2], FAKE, FAKE, FAKE, FAKE, 0.1)
    K.kvarn_seq_release(h, 2)  # leaves holes in the pool
    img = _snapshot(h)
    assert img.size == K.kvarn_snapshot_bytes(h) and bytes(img[:8]) == b"KVARNSN1"
    h2, _ = host_cache(tail_floor=floor, pool_groups=64)
    K.kvarn_append(h2, 0, [3], [500], FAKE, FAKE)  # state that the load replaces
    K.kvarn_snapshot_load(h2, img, img.size)
    assert _state(h2, cfg) == _state(h, cfg)
    used = K.kvarn_cache_stats(h2).pool_slots_used
    taken = {K.kvarn_group_record(h2, l, s, g, 0, 0)[0] for l in range(2) for s in range(4)
             for g in range(max(K.kvarn_seq_length(h2, l, s) - 128, 0) // 128 - floor)}
    K.kvarn_append(h2, 1, [3], [128 + 128 * (floor + 1)], FAKE, FAKE)  # seals one group
    new = K.kvarn_group_record(h2, 1, 3, 0, 0, 0)[0]
    assert new not in taken and K.kvarn_cache_stats(h2).pool_slots_used == used + 1
    assert _snapshot(h2).size == K.kvarn_snapshot_bytes(h2)


def test_snapshot_rejects_bad_images_and_leaves_the_cache_unchanged():
    import numpy as np
    h, cfg = host_cache(pool_groups=32)
    K.kvarn_append(h, 0, [0], [600], FAKE, FAKE)
    img = _snapshot(h)
    h2, _ = host_cache(pool_groups=32)
    K.kvarn_append(h2, 0, [1], [300], FAKE, FAKE)
    before = _state(h2, cfg)
    bad = []
    b = img.copy(); b[0] = ord("X"); bad.append(b)                       # magic
    b = img.copy(); b[8] = 9; bad.append(b)                              # version
    bad.append(img[:-1].copy())                                          # truncated
    hdr = 16 + 4 * 14 + 8 + 5 * 8                                        # header bytes
    lens = np.frombuffer(img[hdr:hdr + 8 * 8].tobytes(), np.int64).copy()
    b = img.copy(); l2 = lens.copy(); l2[0] = 5000; b[hdr:hdr + 64] = np.frombuffer(l2.tobytes(), np.uint8); bad.append(b)
    tab = hdr + 8 * 8
    b = img.copy(); b[tab:tab + 4] = np.frombuffer(np.int32(99).tobytes(), np.uint8); bad.append(b)   # slot out of range
    b = img.copy(); b[tab + 4:tab + 8] = b[tab:tab + 4]; bad.append(b)   # a slot used twice
    for b in bad:
        with pytest.raises(K.KVarNError) as e:
            K.kvarn_snapshot_load(h2, b, b.size)
        assert e.value.status == 1
    assert _state(h2, cfg) == before
    other, _ = host_cache(pool_groups=32, k_bits=4)                     # another configuration
    with pytest.raises(K.KVarNError):
        K.kvarn_snapshot_load(other, img, img.size)
    K.kvarn_snapshot_load(h2, img, img.size)
    assert _state(h2, cfg) == _state(h, cfg)


def test_bits_per_element_formula():
    """Body bits/element = b + 528*8/16384 per side (fig1.dev: about 2.3 at two bits)."""
    for kb, vb in [(2, 2), (4, 2), (4, 4), (8, 8)]:
        h, _ = host_cache(k_bits=kb, v_bits=vb)
        s = K.kvarn_cache_stats(h)
        assert abs(s.body_bits_per_element - ((kb + vb) / 2 + 528 * 8 / 16384)) < 1e-12
        K.kvarn_append(h, 0, [0], [128 + 128 * 10], FAKE, FAKE)
        s = K.kvarn_cache_stats(h)
        elems = (128 + 1280) * 2 * 128 * 2
        expect = (10 * 2 * (K.kvarn_record_bytes(kb) + K.kvarn_record_bytes(vb)) + 128 * 2 * 128 * 2 * 2) * 8 / elems
        assert abs(s.all_in_bits_per_element - expect) < 1e-9


@pytest.mark.parametrize("floor", [0, 1])
def test_bench_step_bytes_matches_the_cache_accounting(floor, monkeypatch):
    """The roofline numerator of bench.py (algorithmic bytes of one decode step) equals
    an independent count from the library's own accounting after the step: every sealed
    record and exact fp16 token read, q read and out written, the new token written, and
    for a sealing sequence its 127 older group tokens read and the new records written."""
    import sys
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setattr(bench, "FLOOR", floor)
    lengths = [300, 383, 511, 1000, 127, 128, 255, 4096 + 127]
    h, _ = host_cache(max_seqs=len(lengths), num_layers=1, num_q_heads=bench.HQ, num_kv_heads=bench.HKV,
                      k_bits=bench.KB, v_bits=bench.VB, max_seq_len=8192, pool_groups=256, tail_floor=floor)
    ids = list(range(len(lengths)))
    K.kvarn_append(h, 0, ids, lengths, FAKE, FAKE)
    used = K.kvarn_cache_stats(h).pool_slots_used
    K.kvarn_decode_step(h, 0, ids, FAKE, FAKE, FAKE, FAKE, 0.1)
    st = K.kvarn_cache_stats(h)
    sealing = st.pool_slots_used - used  # groups sealed by the step
    assert sealing == (4 if floor == 0 else 3)
    pair = st.record_bytes_k + st.record_bytes_v
    # a sealing step reads the group's tokens from the tail: 127 and the new one without a
    # floor, all 128 with one
    tail_read = 127 if floor == 0 else 128
    expected = (st.sealed_bytes + st.exact_bytes + len(lengths) * (bench.HQ * 512 + bench.HKV * 512)
                + sealing * bench.HKV * (tail_read * 512 + pair))
    assert bench.step_bytes(lengths) == expected


def test_every_entry_point_rejects_a_null_cache_handle():
    import ctypes
    L = K.load()
    I = ctypes.c_int32
    ids, cnt = (I * 1)(0), (I * 1)(1)
    ptr, size, n64 = ctypes.c_void_p(), ctypes.c_size_t(), ctypes.c_int64()
    calls = {
        "kvarn_append": lambda: L.kvarn_append(None, 0, 1, ids, cnt, FAKE, FAKE, None),
        "kvarn_decode_attention": lambda: L.kvarn_decode_attention(None, 0, 1, ids, FAKE, FAKE, 0.1, None),
        "kvarn_decode_attention_noalloc": lambda: L.kvarn_decode_attention_noalloc(None, 0, 1, ids, FAKE, FAKE, 0.1,
                                                                                   None),
        "kvarn_decode_step": lambda: L.kvarn_decode_step(None, 0, 1, ids, FAKE, FAKE, FAKE, FAKE, 0.1, None),
        "kvarn_prefill_attention": lambda: L.kvarn_prefill_attention(None, 0, 1, ids, cnt, FAKE, FAKE, 0.1, None),
        "kvarn_prefill": lambda: L.kvarn_prefill(None, 0, 1, ids, cnt, FAKE, FAKE, FAKE, FAKE, 0.1, None),
        "kvarn_dequant_group": lambda: L.kvarn_dequant_group(None, 0, 0, 0, 0, 0, 0, 1, FAKE, None),
        "kvarn_seq_release": lambda: L.kvarn_seq_release(None, 0),
        "kvarn_seq_length": lambda: L.kvarn_seq_length(None, 0, 0, ctypes.byref(n64)),
        "kvarn_group_record": lambda: L.kvarn_group_record(None, 0, 0, 0, 0, 0, ctypes.byref(ptr), ctypes.byref(size)),
        "kvarn_exact_regions": lambda: L.kvarn_exact_regions(None, 0, 0, *[ctypes.byref(ptr)] * 4),
        "kvarn_cache_stats": lambda: L.kvarn_cache_stats(None, ctypes.byref(K.kvarn_stats())),
        "kvarn_check_device_error": lambda: L.kvarn_check_device_error(None, None),
        "kvarn_snapshot_bytes": lambda: L.kvarn_snapshot_bytes(None, ctypes.byref(size)),
        "kvarn_snapshot_save": lambda: L.kvarn_snapshot_save(None, FAKE, 1000, None),
        "kvarn_snapshot_load": lambda: L.kvarn_snapshot_load(None, FAKE, 1000, None),
    }
    for name, call in calls.items():
        assert call() == 1, name
