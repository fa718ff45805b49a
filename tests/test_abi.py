"""CPU tests of the C ABI: the library loads, exports every symbol the
header declares, validates arguments, and its host-side logic (native
packing, the pool's LRU policy in dry-run mode, checkpoint/resume, fault
injection) matches the oracle."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import moe_synth as S
import oracle
import routed_expert_ffn_histogram_gb300 as M
from routed_expert_ffn_histogram_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 20
    L = M.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_python_names_exist():
    assert all(hasattr(M, n) for n in M.__all__), [n for n in M.__all__ if not hasattr(M, n)]


def test_status_strings_and_no_device_count():
    for s in [0, -1, -2, -3, -4, -5, -6]:
        assert M.status_str(s)
    assert M.lib().moe_device_count() >= 0


def test_expert_bytes():
    for H, I in [(2880, 2880), (2048, 768), (256, 512)]:
        eb = M.moe_expert_bytes(H, I)
        canon = 3 * (H * I // 2 + H * I // 32)
        # row-major matrices (rows padded to 32 bytes) plus the column-blocked
        # copy of down: 16 columns x H rows, 8 code bytes + 1 scale byte per row
        dt = (I // 16) * (-(-(H * 9) // 128) * 128)
        assert eb % 1024 == 0 and canon + dt <= eb <= (canon + dt) * (1.01 if H >= 2048 else 1.15)
    with pytest.raises(M.MoeError):
        M.moe_expert_bytes(100, 64)


def test_pack_native_layout():
    """Gate/up rows interleave in chunks of 32; every row is codes then scales."""
    wl = S.WORKLOADS[0]
    H, I = wl.hidden, wl.inter
    w = S.expert_weights(wl, 0, 1)
    eb = M.moe_expert_bytes(H, I)
    buf = np.zeros(eb, np.uint8)
    M.moe_pack_expert(w, H, I, buf)
    rs_gu = -(-(H // 2 + ((H // 32 + 15) // 16) * 16) // 32) * 32
    rs_d = -(-(I // 2 + ((I // 32 + 15) // 16) * 16) // 32) * 32
    for r in [0, 1, 31, 32, 63, 64, 200, I - 1]:
        g = (r // 32) * 64 + r % 32
        row = buf[g * rs_gu:(g + 1) * rs_gu]
        assert np.array_equal(row[:H // 2], w["gate_codes"][r])
        assert np.array_equal(row[H // 2:H // 2 + H // 32], w["gate_scales"][r])
        assert not row[H // 2 + H // 32:].any()
        row = buf[(g + 32) * rs_gu:(g + 33) * rs_gu]
        assert np.array_equal(row[:H // 2], w["up_codes"][r])
        assert np.array_equal(row[H // 2:H // 2 + H // 32], w["up_scales"][r])
    d_off = 2 * I * rs_gu
    for r in [0, 7, H - 1]:
        row = buf[d_off + r * rs_d:d_off + (r + 1) * rs_d]
        assert np.array_equal(row[:I // 2], w["down_codes"][r])
        assert np.array_equal(row[I // 2:I // 2 + I // 32], w["down_scales"][r])
    # column-blocked copy of down: block c = elements 16c..16c+15 of every row
    # (8 code bytes per row, rows in order), then every row's scale of block c//2
    dt_off = -(-(d_off + H * rs_d) // 128) * 128
    dt_stride = -(-(H * 9) // 128) * 128
    for c in [0, 1, 2, I // 16 - 1]:
        blk = buf[dt_off + c * dt_stride:dt_off + (c + 1) * dt_stride]
        codes = blk[:H * 8].reshape(H, 8)
        assert np.array_equal(codes, w["down_codes"][:, 8 * c:8 * c + 8])
        assert np.array_equal(blk[H * 8:H * 9], w["down_scales"][:, c // 2])
        assert not blk[H * 9:].any()


def test_invalid_arguments_rejected_before_launch():
    L = M.lib()
    sz = C.c_size_t()
    assert L.moe_route_workspace_bytes(10, 300, 2, C.byref(sz)) == M.MOE_ERR_INVALID
    assert L.moe_route_workspace_bytes(10, 8, 9, C.byref(sz)) == M.MOE_ERR_INVALID
    assert L.moe_route_plan(None, 4, 8, 2, None, None, None, None, None, None, None, None, 0, None) == \
        M.MOE_ERR_INVALID
    assert L.moe_combine(None, None, None, 2, 0, 8, None, None) == M.MOE_ERR_INVALID
    assert L.moe_quant_mxfp8(None, 33, None, 1, 1, None, None, 2, None) == M.MOE_ERR_INVALID
    assert L.moe_ffn_workspace_bytes(4, 2, 250, 512, 0, C.byref(sz)) == M.MOE_ERR_INVALID
    # the accumulate flag is the only bit allowed beside the path; it does not change the size
    assert L.moe_ffn_workspace_bytes(4, 2, 256, 512, 0x400, C.byref(sz)) == M.MOE_ERR_INVALID
    assert L.moe_ffn_workspace_bytes(4, 2, 256, 512, M.MOE_PATH_DECODE, C.byref(sz)) == M.MOE_OK
    plain = sz.value
    assert L.moe_ffn_workspace_bytes(4, 2, 256, 512, M.MOE_PATH_DECODE | M.MOE_FFN_ACCUMULATE, C.byref(sz)) == M.MOE_OK
    assert sz.value == plain
    assert L.moe_expert_ffn(None, 0, None, 1, 1, None, None, None, None, None, None, 0, None, 0, None, None) == \
        M.MOE_ERR_INVALID
    assert L.moe_decode_layer_acc(None, 0, None, None, 1, 1, None, None, None, None, None, None, None, None, 0,
                                  None, None) == M.MOE_ERR_INVALID
    assert L.moe_pool_prefetch(None, 0, 1, None, None, None) == M.MOE_ERR_INVALID
    bits = C.c_uint32(7)
    assert L.moe_ffn_status(None, M.MOE_PATH_DECODE, None, C.byref(bits)) == M.MOE_ERR_INVALID
    assert L.moe_ffn_status(None, 9, None, C.byref(bits)) == M.MOE_ERR_INVALID
    assert L.moe_debug_stall_next_decode(-1) == M.MOE_ERR_INVALID
    assert L.moe_debug_stall_next_decode(0) == M.MOE_OK
    d = _lib.MoePoolDesc(1, 8, 9, 256, 512, None, None, 0, 1)
    h = C.c_void_p()
    assert L.moe_pool_create(C.byref(d), C.byref(h)) == M.MOE_ERR_INVALID  # S > E
    d = _lib.MoePoolDesc(1, 8, 4, 256, 512, None, None, 0, 0)
    assert L.moe_pool_create(C.byref(d), C.byref(h)) == M.MOE_ERR_INVALID  # buffers required


def _stream_counts(wl, layer, step):
    ids, _ = oracle.route(S.logits(wl, layer, step), wl.top_k)
    return np.bincount(ids.reshape(-1), minlength=wl.experts).astype(np.int32)


def test_dry_run_pool_matches_oracle_lru():
    """The library's pool policy equals the oracle's LRU event by event
    (slot maps, load lists and counters bit-exact) on the skewed GPT-OSS
    offload routing, 24 layers x 40 steps."""
    wl = S.WORKLOADS[2]
    pool = M.Pool(wl.layers, wl.experts, wl.slots, wl.hidden, wl.inter, dry_run=True)
    ref = [oracle.LRUPool(wl.slots, wl.experts) for _ in range(wl.layers)]
    for step in range(40):
        for l in range(wl.layers):
            c = _stream_counts(wl, l, step)
            loads = ref[l].step(c)
            assert pool.stage(l, c) == M.MOE_OK
            assert pool.last_loads(l) == loads
            assert np.array_equal(pool.slot_map(l), ref[l].slot_map())
    for l in range(wl.layers):
        got = pool.counters(l)
        exp = ref[l].counters()
        assert (got["hits"], got["misses"], got["evictions"]) == (exp["hits"], exp["misses"], exp["evictions"])
        assert got["h2d_bytes"] == exp["misses"] * M.moe_expert_bytes(wl.hidden, wl.inter)


def test_dry_run_capacity_and_preload():
    pool = M.Pool(1, 8, 2, 256, 512, dry_run=True, preload=True)
    assert np.array_equal(pool.slot_map(0), [0, 1, -1, -1, -1, -1, -1, -1])
    assert pool.stage(0, np.array([1, 1, 1, 0, 0, 0, 0, 0], np.int32)) == M.MOE_ERR_CAPACITY
    assert np.array_equal(pool.slot_map(0), [0, 1, -1, -1, -1, -1, -1, -1])
    assert pool.stage(0, np.array([0, 3, 0, 0, 0, 0, 0, 2], np.int32)) == M.MOE_OK
    assert pool.last_loads(0) == [(7, 0)]  # preloaded stamps tie -> lowest slot evicted


def test_checkpoint_resume_roundtrip():
    wl = S.WORKLOADS[2]
    a = M.Pool(wl.layers, wl.experts, wl.slots, wl.hidden, wl.inter, dry_run=True)
    for step in range(10):
        for l in range(wl.layers):
            a.stage(l, _stream_counts(wl, l, step))
    state = a.save()
    b = M.Pool(wl.layers, wl.experts, wl.slots, wl.hidden, wl.inter, dry_run=True)
    assert b.load(state) == M.MOE_OK
    for step in range(10, 20):
        for l in range(wl.layers):
            c = _stream_counts(wl, l, step)
            a.stage(l, c)
            b.stage(l, c)
            assert a.last_loads(l) == b.last_loads(l)
    assert a.counters() == b.counters()
    other = M.Pool(wl.layers, wl.experts, 4, wl.hidden, wl.inter, dry_run=True)
    assert other.load(state) == M.MOE_ERR_STATE
    bad = bytearray(state)
    bad[24:28] = (99).to_bytes(4, "little", signed=True)  # corrupt a slot entry
    assert b.load(bytes(bad)) == M.MOE_ERR_STATE


def test_injected_copy_failure_rolls_back():
    """A failed copy leaves the event unapplied; the retry is a clean event."""
    pool = M.Pool(1, 8, 2, 256, 512, dry_run=True)
    ref = oracle.LRUPool(2, 8)
    c1 = np.array([1, 0, 0, 1, 0, 0, 0, 0], np.int32)
    assert pool.stage(0, c1) == M.MOE_OK
    ref.step(c1)
    before = (pool.slot_map(0).copy(), pool.counters(0))
    pool.inject_copy_failures(1)
    c2 = np.array([0, 0, 1, 1, 0, 0, 0, 0], np.int32)
    with pytest.raises(M.MoeError) as ei:
        pool.stage(0, c2)
    assert ei.value.status == M.MOE_ERR_CUDA
    assert np.array_equal(pool.slot_map(0), before[0])
    after = pool.counters(0)
    assert after["errors"] == 1 and after["misses"] == before[1]["misses"] and after["hits"] == before[1]["hits"]
    assert pool.stage(0, c2) == M.MOE_OK
    assert pool.last_loads(0) == ref.step(c2)
    assert np.array_equal(pool.slot_map(0), ref.slot_map())


def test_device_planned_staging_arguments_checked_on_the_host():
    """The device-planned staging calls validate on the host before any CUDA
    call: a dry-run pool cannot attach, an unattached pool cannot stage on
    the device, join or detach, bad pointers and layers are refused, and the
    state size is one record per layer (16-byte multiples)."""
    import ctypes as C

    import routed_expert_ffn_histogram_gb300 as M

    L = M._lib.lib()
    pool = M.Pool(3, 32, 8, 2880, 2880, dry_run=True)
    n = pool.device_state_bytes()
    assert n > 0 and n % (3 * 16) == 0
    buf = C.create_string_buffer(n + 16)
    aligned = (C.addressof(buf) + 15) & ~15
    assert L.moe_pool_device_attach(pool.handle, aligned, n, None, 100) == M.MOE_ERR_STATE
    assert L.moe_pool_device_attach(pool.handle, None, n, None, 100) == M.MOE_ERR_INVALID
    assert L.moe_pool_device_attach(pool.handle, aligned + 4, n, None, 100) == M.MOE_ERR_INVALID
    assert L.moe_pool_device_attach(pool.handle, aligned, n - 16, None, 100) == M.MOE_ERR_INVALID
    assert L.moe_pool_device_attach(None, aligned, n, None, 100) == M.MOE_ERR_INVALID
    counts = (C.c_int32 * 32)()
    slots = (C.c_int32 * 32)()
    assert L.moe_pool_stage_device(pool.handle, 0, counts, slots, None, None, None) == M.MOE_ERR_STATE
    assert L.moe_pool_stage_device(pool.handle, 3, counts, slots, None, None, None) == M.MOE_ERR_INVALID
    assert L.moe_pool_stage_device(pool.handle, 0, None, slots, None, None, None) == M.MOE_ERR_INVALID
    assert L.moe_pool_stage_device(pool.handle, 0, counts, None, None, None, None) == M.MOE_ERR_INVALID
    # routing + planning in one launch: the same checks, plus the routing's
    # (logits and outputs present, 1 <= k <= E, T >= 1, T * k <= 32)
    lg = (C.c_float * 64)()
    o32 = [(C.c_int32 * 64)() for _ in range(5)]
    wt = (C.c_float * 64)()

    def rsd(layer, logits, T, k, slot_map):
        return L.moe_pool_route_stage_device(pool.handle, layer, logits, T, k, o32[0], wt, o32[1], o32[2], o32[3],
                                             o32[4], slot_map, None, None, None)

    assert rsd(0, lg, 1, 4, slots) == M.MOE_ERR_STATE
    assert rsd(3, lg, 1, 4, slots) == M.MOE_ERR_INVALID
    assert rsd(0, None, 1, 4, slots) == M.MOE_ERR_INVALID
    assert rsd(0, lg, 1, 4, None) == M.MOE_ERR_INVALID
    assert rsd(0, lg, 0, 4, slots) == M.MOE_ERR_INVALID
    assert rsd(0, lg, 1, 0, slots) == M.MOE_ERR_INVALID
    assert rsd(0, lg, 1, 33, slots) == M.MOE_ERR_INVALID
    assert rsd(0, lg, 9, 4, slots) == M.MOE_ERR_UNSUPPORTED
    assert L.moe_pool_route_stage_device(None, 0, lg, 1, 4, o32[0], wt, o32[1], o32[2], o32[3], o32[4], slots,
                                         None, None, None) == M.MOE_ERR_INVALID
    assert L.moe_pool_device_join(pool.handle, 0, None) == M.MOE_ERR_STATE
    assert L.moe_pool_device_join(pool.handle, -1, None) == M.MOE_ERR_INVALID
    assert L.moe_pool_device_detach(pool.handle, None, 100) == M.MOE_ERR_STATE
    assert L.moe_pool_device_detach(None, None, 100) == M.MOE_ERR_INVALID
    # the host-side calls still work on the (never attached) pool
    assert pool.counters()["events"] == 0
    pool.close()
