"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function declared in include/attn.h, rejects bad
arguments before touching a device, and its integer schedules equal the
oracle's plain-Python restatement element by element."""
import ctypes as C
import os
import re
import shutil

import numpy as np
import pytest

import oracle
from io_aware_exact_attn_gb300 import _ffi, api, build as B, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_ffi.LIB_PATH) or B._stale():
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc unavailable and library not built")
        B.build()
    return _ffi.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 12, names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_ffi.SIGNATURES), set(names) ^ set(_ffi.SIGNATURES)
    assert lib.attn_version() >= 1


def test_status_strings(lib):
    for code in list(_ffi.STATUS):
        assert lib.attn_status_string(code)


def _ptr(x):
    return C.c_void_p(x)


def test_argument_validation_without_gpu(lib):
    m = None
    good = 4096
    # NULL / misaligned pointers and bad sizes are rejected before any device call
    assert lib.attn_fwd(None, _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, 0.125, m, None) == -1
    assert lib.attn_fwd(_ptr(good + 2), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, 0.125, m,
                        None) == -3
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 3, 2, 128, 64, 0.125, m,
                        None) == -1
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 96, 0.125, m,
                        None) == -2
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 0, 64, 0.125, m,
                        None) == -1
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, -1.0, m,
                        None) == -1
    bad = _ffi.attn_mask_t(7, 0, None, 0)
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, 0.125,
                        C.byref(bad), None) == -1
    sparse_no_mask = _ffi.attn_mask_t(2, 0, None, 0)
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, 0.125,
                        C.byref(sparse_no_mask), None) == -1
    assert "multiple" in lib.attn_last_error_message().decode() or lib.attn_last_error_message()
    # debug records: the setter checks its arguments and touches no device
    assert lib.attn_debug_set_tile_counts(_ptr(good + 2), 64) == -3
    assert lib.attn_debug_set_tile_counts(_ptr(good), -1) == -1
    assert lib.attn_debug_set_tile_counts(None, -1) == 0   # off; the capacity is ignored
    # merge: part count limits
    arr = (C.c_void_p * 1)(good)
    assert lib.attn_merge_lse(arr, arr, 0, _ptr(good), 0, None, 1, 1, 4, 64, 0, None) == -1
    assert lib.attn_merge_lse(arr, arr, 65, _ptr(good), 0, None, 1, 1, 4, 64, 0, None) == -1
    # bwd workspace size and check
    need = lib.attn_bwd_workspace_bytes(2, 4, 2, 100, 64)
    rows = 2 * 4 * 128   # padded query rows: D and LSE*log2 e (float32), then 32 bytes each
    assert need == 2 * ((rows * 4 + 255) // 256) * 256 + rows * 32
    # ragged: (B+1) ints, then the same statistics for Hq * (total + 127 B) rows, the
    # 32-byte rows in whole 128-row blocks
    vrows = 4 * (1000 + 127 * 3)
    vneed = ((4 * 4 + 255) // 256) * 256 + 2 * ((vrows * 4 + 255) // 256) * 256 + \
        (((vrows + 127) // 128) * 4096 + 255) // 256 * 256
    assert lib.attn_varlen_bwd_workspace_bytes(3, 1000, 4) == vneed
    p = [_ptr(good)] * 10
    assert lib.attn_bwd(*p, need - 256, 2, 4, 2, 100, 64, 0.125, None, None) == -6
    # chunked backward: workspace, pointer, offset and size checks come before any device call
    ws = lib.attn_bwd_workspace_bytes(1, 4, 4, 300, 128)
    assert lib.attn_bwd_preprocess(_ptr(good), _ptr(good), _ptr(good), 1, 4, 300, 128, 0, _ptr(good), ws - 1,
                                   None) == -6
    assert lib.attn_bwd_preprocess(_ptr(good), _ptr(good), _ptr(good), 1, 4, 300, 128, 299, _ptr(good), ws,
                                   None) == -1                                           # head stride < Nq
    assert lib.attn_bwd_preprocess(_ptr(good), _ptr(good), _ptr(good + 2), 1, 4, 300, 128, 0, _ptr(good), ws,
                                   None) == -3
    pb = [_ptr(good)] * 4
    out = [_ptr(good)] * 3
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws - 1, *out, 1, 4, 2, 300, 200, 128, 0.088, None, 0, 0, 0, 0, 1,
                                None) == -6
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws, _ptr(good), None, _ptr(good), 1, 4, 2, 300, 200, 128, 0.088,
                                None, 0, 0, 0, 0, 1, None) == -1                         # dk missing
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws, *out, 1, 4, 2, 300, 200, 128, 0.088, None, 1 << 31, 0, 0, 0,
                                1, None) == -1                                           # offsets too far apart
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws, *out, 1, 4, 2, 300, 200, 128, 0.088, None, -1, 0, 0, 0, 1,
                                None) == -1                                              # negative position
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws, *out, 1, 4, 2, 300, 200, 128, 0.088, None, 0, 0, 299, 0, 1,
                                None) == -1                                              # q head stride < Nq
    assert lib.attn_partial_bwd(*pb, _ptr(good), ws, *out, 1, 4, 3, 300, 200, 128, 0.088, None, 0, 0, 0, 0, 1,
                                None) == -1                                              # Hq % Hkv
    # sliding window needs a width of at least one
    no_width = _ffi.attn_mask_t(3, 0, None, 0)
    assert lib.attn_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), None, 1, 2, 2, 128, 64, 0.125,
                        C.byref(no_width), None) == -1
    # decode: workspace size, split count, row and length limits
    assert lib.attn_decode_splits(8, 8, 32768) == 14           # ceil(6 * 148 / 64) splits
    assert lib.attn_decode_splits(1, 1, 100) == 1              # never more splits than key tiles
    assert lib.attn_decode_splits(1, 1, 1 << 20) == 64
    wsb = lib.attn_decode_workspace_bytes(2, 8, 2, 3, 1000, 64, 4)
    rows = 2 * 8 * 3
    per = ((rows * 64 * 4 + 255) // 256) * 256 + ((rows * 4 + 255) // 256) * 256
    assert wsb == 2 * 4 * per          # 4 * 3 rows per kv head fit one tile: two partials per split
    assert lib.attn_decode_workspace_bytes(2, 8, 2, 3, 1000, 64, 40) == 40 * per    # 80 partials would not merge
    assert lib.attn_decode_workspace_bytes(2, 64, 1, 3, 1000, 64, 4) == 4 * 2 * 64 * 3 * (64 * 4 + 4)  # 192 rows
    q = [_ptr(good)] * 3
    assert lib.attn_decode_fwd(*q, None, _ptr(good), None, 2, 8, 2, 3, 1000, 64, 0.125, 1, 4, _ptr(good),
                               wsb - 1, None) == -6
    assert lib.attn_decode_fwd(*q, None, _ptr(good), None, 2, 64, 1, 8, 1000, 64, 0.125, 1, 4, _ptr(good),
                               1 << 30, None) == -1                                       # 64 * 8 rows > 256
    assert lib.attn_decode_fwd(*q, None, _ptr(good), None, 2, 8, 2, 3, 2, 64, 0.125, 1, 4, _ptr(good),
                               1 << 30, None) == -1                                       # Nq > Nk
    assert lib.attn_decode_fwd(*q, None, _ptr(good), None, 2, 8, 2, 3, 1000, 64, 0.125, 1, 65, _ptr(good),
                               1 << 30, None) == -1                                       # too many splits
    # e4m3 forward: d = 128 only, positive finite scale factors, workspace for V^T
    assert lib.attn_fwd_fp8_workspace_bytes(2, 4, 300, 128) == 2 * 4 * 128 * 384
    f8 = [_ptr(good)] * 3
    fws = lib.attn_fwd_fp8_workspace_bytes(1, 2, 128, 128)
    assert lib.attn_fwd_fp8(*f8, 1.0, 1.0, 1.0, _ptr(good), None, 1, 2, 2, 128, 64, 0.125, None, _ptr(good),
                            1 << 30, None) == -2
    assert lib.attn_fwd_fp8(*f8, 1.0, 0.0, 1.0, _ptr(good), None, 1, 2, 2, 128, 128, 0.125, None, _ptr(good),
                            1 << 30, None) == -1
    assert lib.attn_fwd_fp8(*f8, 1.0, 1.0, float("inf"), _ptr(good), None, 1, 2, 2, 128, 128, 0.125, None,
                            _ptr(good), 1 << 30, None) == -1
    assert lib.attn_fwd_fp8(*f8, 1.0, 1.0, 1.0, _ptr(good), None, 1, 2, 2, 128, 128, 0.125, None, _ptr(good),
                            fws - 1, None) == -6
    assert lib.attn_fwd_fp8(*f8, 1.0, 1.0, 1.0, _ptr(good), None, 1, 2, 2, 128, 128, 0.125, None, None,
                            fws, None) == -1
    # partial fwd: head stride smaller than the rows is rejected
    assert lib.attn_partial_fwd(_ptr(good), _ptr(good), _ptr(good), _ptr(good), _ptr(good), 1, 2, 2, 256, 256,
                                64, 0.125, None, 0, 0, 100, 0, None) == -1


def test_status_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("has a GPU")
    assert lib.attn_get_status(None) == -7


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8, 13])
@pytest.mark.parametrize("lanes", [0, 1, 3, 8])
def test_chunk_schedule_matches_oracle(lib, n, lanes):
    got = api.build_chunk_schedule(n, lanes)
    want = oracle.chunk_pair_schedule(n, lanes)
    assert got == want
    assert sorted(got) == sorted((q, k) for q in range(n) for k in range(q + 1))


def test_chunk_schedule_balance():
    """Costs add up to n^2 half-tiles, and each lane's load is within one pair
    (cost 2) of the mean load."""
    for n in (3, 4, 8, 16, 32):
        for lanes in (n, 3, 8):
            per = oracle.chunk_pair_lanes(n, lanes)
            pairs = oracle.chunk_pair_schedule(n, lanes)
            total = sum(1 if q == k else 2 for q, k in pairs)
            assert total == n * n
            assert len(pairs) == n * (n + 1) // 2
            assert sorted(p for lane in per for p in lane) == sorted(pairs)
            loads = [sum(1 if q == k else 2 for q, k in lane) for lane in per]
            mean = n * n / lanes
            assert all(abs(x - mean) <= 2 for x in loads), (n, lanes, loads)


CASES = [
    (0, 1, 2, 2, 600, 600, 0, 0, 64), (1, 1, 2, 2, 600, 600, 0, 0, 128), (1, 2, 3, 3, 1000, 1000, 0, 0, 64),
    (1, 1, 4, 4, 4096, 4096, 4096, 0, 128), (1, 1, 4, 2, 4096, 4096, 4096, 8192, 128),
    (1, 1, 2, 1, 300, 700, 128, 0, 64), (0, 2, 3, 1, 129, 1, 0, 0, 128), (1, 1, 1, 1, 1, 1, 0, 0, 64),
    (1, 1, 2, 2, 512, 512, 0, 300, 128),
    # head grouping kicks in: K+V of a head is 4 MiB (16 heads per group) / 16 MiB with GQA 4
    (1, 2, 32, 32, 8192, 8192, 0, 0, 128), (1, 1, 32, 8, 32768, 32768, 0, 0, 128),
    (0, 3, 7, 7, 65536, 65536, 0, 0, 64),
]


@pytest.mark.parametrize("case", CASES)
def test_fwd_schedule_matches_oracle(lib, case):
    kind, B_, H, Hkv, nq, nk, qo, ko, d = case
    got = api.build_schedule(kind, B_, H, nq, nk, qo, ko, Hkv=Hkv, d=d)
    want = np.array(oracle.fwd_work_units(["none", "causal"][kind], B_, H, nq, nk, qo, ko, Hkv=Hkv, d=d),
                    dtype=np.int32)
    np.testing.assert_array_equal(got, want.reshape(-1, 3))


def test_head_groups():
    assert oracle.schedule.head_group(2, 32, 32, 8192, 128) == 16
    assert oracle.schedule.head_group(1, 32, 8, 32768, 128) == 16
    assert oracle.schedule.head_group(8, 16, 16, 512, 64) == 128
    assert oracle.schedule.head_group(1, 4, 4, 1 << 20, 128) == 1


@pytest.mark.parametrize("cib", [False, True])
def test_fwd_schedule_block_sparse_matches_oracle(lib, cib):
    n = 1000
    nb = -(-n // 128)
    bm = inputs.block_sparse_mask(nb, nb, 0.25, seed=5)
    got = api.build_schedule(2, 2, 3, n, n, 0, 0, host_block_mask=bm, causal_in_blocks=cib, d=64)
    want = oracle.fwd_work_units("block_sparse", 2, 3, n, n, 0, 0, bm, cib, d=64)
    np.testing.assert_array_equal(got, np.array(want, dtype=np.int32).reshape(-1, 3))


WINDOW_CASES = [
    # (B, Hq, Hkv, Nq, Nk, q_offset, kv_offset, d, window)
    (1, 2, 2, 1000, 1000, 0, 0, 128, 1), (1, 2, 2, 1000, 1000, 0, 0, 128, 100),
    (2, 3, 1, 700, 700, 0, 0, 64, 128), (1, 2, 2, 1000, 1000, 0, 0, 128, 129),
    (1, 1, 1, 1500, 1500, 0, 0, 64, 300), (1, 2, 1, 600, 900, 256, 0, 128, 333),
    (1, 2, 2, 512, 512, 1024, 512, 128, 700), (1, 2, 2, 2048, 2048, 0, 0, 128, 100000),
    (1, 4, 4, 8192, 8192, 0, 0, 128, 4096),
]


@pytest.mark.parametrize("case", WINDOW_CASES)
def test_fwd_schedule_sliding_window_matches_oracle(lib, case):
    B_, H, Hkv, nq, nk, qo, ko, d, w = case
    got = api.build_schedule(3, B_, H, nq, nk, qo, ko, Hkv=Hkv, d=d, window=w)
    want = oracle.fwd_work_units("sliding_window", B_, H, nq, nk, qo, ko, Hkv=Hkv, d=d, window=w)
    np.testing.assert_array_equal(got, np.array(want, dtype=np.int32).reshape(-1, 3))


def test_schedule_rejects_bad_window(lib):
    with pytest.raises(RuntimeError):
        api.build_schedule(3, 1, 1, 256, 256, window=0)


def test_schedule_covers_every_visible_tile_pair_once():
    """Coverage from the visibility matrix itself: each work unit visits exactly
    the key tiles that hold at least one key visible to one of its rows."""
    for kind, qo, ko in (("causal", 0, 0), ("causal", 256, 0), ("none", 0, 0)):
        nq, nk = 700, 900
        units = oracle.fwd_work_units(kind, 1, 1, nq, nk, qo, ko)
        vis = oracle.visible(np.arange(nq), nk, oracle.MaskSpec(kind), qo, ko)
        seen = set()
        for bh, qc, cnt in units:
            rows = slice(qc * 256, min(nq, qc * 256 + 256))
            tiles = {j // 128 for j in np.flatnonzero(vis[rows].any(axis=0))}
            assert cnt == len(tiles)
            assert qc not in seen
            seen.add(qc)
        assert seen == set(range(-(-nq // 256)))


def test_workload_inputs_are_seeded():
    q1, k1, v1, d1 = inputs.make_qkvdo(1, 2, 1, 64, 64, 64)
    q2, k2, v2, d2 = inputs.make_qkvdo(1, 2, 1, 64, 64, 64)
    assert all(bool((a == b).all()) for a, b in ((q1, q2), (k1, k2), (v1, v2), (d1, d2)))
    m = inputs.block_sparse_mask(128, 128)
    assert m.sum() == 128 + round((128 * 128 - 128) / 8) == 2160
    assert m[np.arange(128), np.arange(128)].all()
