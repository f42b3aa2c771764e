"""The C-ABI library builds, loads and exports every entry point declared in
include/*.h; argument checks that return before any CUDA call behave as the
header documents.  CPU only: no compute call is made here."""

import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def zr():
    from gradient_synchronisation_gb300 import _build

    _build.build()
    import gradient_synchronisation_gb300 as zr

    return zr


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"^\s*(?:zr_status|size_t|const char\s*\*)\s*(zr_\w+)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_four_operations():
    names = declared_symbols()
    for op in ("zr_ring_allreduce", "zr_skipreduce", "zr_sparse_aggregate", "zr_partition"):
        assert op in names


def test_library_exports_every_declared_symbol(zr):
    lib = ctypes.CDLL(zr.LIB_PATH)
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(declared_symbols()) <= set(zr.EXPORTS)


def test_binding_has_no_cpu_path():
    src = open(os.path.join(ROOT, "gradient_synchronisation_gb300", "__init__.py")).read()
    assert "oracle" not in src
    for f in glob.glob(os.path.join(ROOT, "gradient_synchronisation_gb300", "**", "*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            assert "import oracle" not in open(f).read() and "from oracle" not in open(f).read(), f


def test_status_strings_and_version(zr):
    assert zr.status_string(zr.ZR_OK) == "ok"
    for code in range(9):
        assert zr.status_string(code)
    assert "sm_103a" in zr.version()


def test_workspace_sizes(zr):
    assert zr.zr_sparse_workspace_size(0, 100, 4) == 0
    assert zr.zr_sparse_workspace_size(8, 0, 4) == 0
    assert zr.zr_sparse_workspace_size(8, 100, -1) == 0
    assert zr.zr_sparse_workspace_size(8, 100, zr.ZR_MAX_PARTS + 1) == 0
    a = zr.zr_sparse_workspace_size(8, 1 << 25, 8)
    b = zr.zr_sparse_workspace_size(8, 1 << 25, 16)
    assert 0 < a < b and a % 256 == 0
    # the push-side partition's workspace: one count per (partition, CTA),
    # independent of the entry count
    assert zr.zr_partition_workspace_size(1000, 0) == 0
    assert zr.zr_partition_workspace_size(1000, 8) > 0
    assert zr.zr_partition_workspace_size(0, 8) == zr.zr_partition_workspace_size((1 << 31) - 1, 8)


def test_static_scratch_holds_every_valid_partition_request(zr):
    """The no-allocation entry's fixed scratch covers the workspace of every
    valid request; the size is read from the header so the binding's copy
    cannot drift from it."""
    import re

    hdr = open(os.path.join(ROOT, "include", "zr.h")).read()
    m = re.search(r"#define ZR_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m, "ZR_STATIC_SCRATCH_BYTES not found in zr.h"
    assert zr.ZR_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    for parts in (1, 8, 16, 33, 255, zr.ZR_MAX_PARTS):
        for nnz in (0, 1, 1 << 20, (1 << 31) - 1):
            assert 0 < zr.zr_partition_workspace_size(nnz, parts) <= zr.ZR_STATIC_SCRATCH_BYTES


def test_dense_argument_errors_before_launch(zr):
    fake = [1 << 40, (1 << 40) + (1 << 30)]
    assert zr.zr_ring_allreduce(fake, 0, 16, zr.ZR_F32, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce(fake, 65, 16, zr.ZR_F32, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce(fake, 2, -1, zr.ZR_F32, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce(fake, 2, 16, 7, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce(fake, 2, 16, zr.ZR_F32, 2, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce([fake[0] + 4, fake[1]], 2, 16, zr.ZR_F32, 1, None) == zr.ZR_ERR_ALIGNMENT
    assert zr.zr_ring_allreduce([fake[0], fake[0] + 32], 2, 16, zr.ZR_F32, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_ring_allreduce([fake[0], 0], 2, 16, zr.ZR_F32, 1, None) == zr.ZR_ERR_INVALID_ARG
    # m == 0 is a valid no-op (nothing to launch)
    assert zr.zr_ring_allreduce(fake, 2, 0, zr.ZR_F32, 1, None) == zr.ZR_OK
    for k in (-1, 2):
        cfg = zr.SkipCfg(zr.ZR_SKIP_STATIC, k, 0, 0, zr.ZR_DIV_N, 0)
        assert zr.zr_skipreduce(fake, 2, 16, zr.ZR_F32, cfg, None) == zr.ZR_ERR_INVALID_ARG
    for bad in (zr.SkipCfg(5, 1, 0, 0, zr.ZR_DIV_N, 0), zr.SkipCfg(0, 1, 0, 0, 9, 0),
                zr.SkipCfg(0, 1, 0, 0, zr.ZR_DIV_N, 2)):
        assert zr.zr_skipreduce(fake, 2, 16, zr.ZR_F32, bad, None) == zr.ZR_ERR_INVALID_ARG


def test_bucket_and_dropout_argument_errors_before_launch(zr):
    # Made-up pointers on a machine without a GPU: every call below must be
    # refused on the host, before anything could be launched.
    a = [1 << 40, (1 << 40) + (1 << 30)]
    b = [(1 << 40) + (2 << 30), (1 << 40) + (3 << 30)]
    ok = zr.SkipCfg(zr.ZR_SKIP_RANDOM, 1, 0, 0, zr.ZR_DIV_N, 0)
    bad_flags = zr.SkipCfg(zr.ZR_SKIP_RANDOM, 1, 0, 0, zr.ZR_DIV_N, 4)
    bad_k = zr.SkipCfg(zr.ZR_SKIP_RANDOM, 2, 0, 0, zr.ZR_DIV_N, 0)
    f32 = zr.ZR_F32
    assert zr.zr_skipreduce_buckets([], 2, f32, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_skipreduce_buckets([(a, 16, ok)], 0, f32, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_skipreduce_buckets([(a, 16, ok)] * 129, 2, f32, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_skipreduce_buckets([(a, 16, bad_flags)], 2, f32, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_skipreduce_buckets([(a, 16, ok), (b, 16, bad_k)], 2, f32, None) == zr.ZR_ERR_INVALID_ARG
    # buffers of two buckets overlapping each other
    assert zr.zr_skipreduce_buckets([(a, 16, ok), ([a[0] + 32, b[0]], 16, ok)], 2, f32,
                                    None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_skipreduce_buckets([(a, 16, ok), ([b[0] + 8, b[1]], 16, ok)], 2, f32,
                                    None) == zr.ZR_ERR_ALIGNMENT
    # every bucket empty: a valid no-op
    assert zr.zr_skipreduce_buckets([(a, 0, ok), (b, 0, ok)], 2, f32, None) == zr.ZR_OK
    # 32 buckets of 64 ranks fill the 2048-pointer table; one more bucket does not fit
    many = [[(1 << 40) + ((j * 64 + r) << 20) for r in range(64)] for j in range(33)]
    cfg0 = zr.SkipCfg(zr.ZR_SKIP_STATIC, 0, 0, 0, zr.ZR_DIV_N, 0)
    assert zr.zr_skipreduce_buckets([(p, 0, cfg0) for p in many[:32]], 64, f32, None) == zr.ZR_OK
    assert zr.zr_skipreduce_buckets([(p, 0, cfg0) for p in many], 64, f32,
                                    None) == zr.ZR_ERR_INVALID_ARG
    dr = zr.zr_allreduce_dropout
    assert dr(a, 2, 16, f32, (1 << 32) + 1, 0, 0, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert dr(a, 2, 16, f32, 0, 0, 0, 2, None) == zr.ZR_ERR_INVALID_ARG
    assert dr(a, 0, 16, f32, 0, 0, 0, 1, None) == zr.ZR_ERR_INVALID_ARG
    assert dr([a[0] + 4, a[1]], 2, 16, f32, 0, 0, 0, 1, None) == zr.ZR_ERR_ALIGNMENT
    assert dr(a, 2, 0, f32, 1 << 32, 0, 0, 1, None) == zr.ZR_OK


def test_dropout_threshold_wrapper_matches_oracle():
    import gradient_synchronisation_gb300 as g
    from oracle import ring

    for p in (0.0, 1.0, 0.5, 0.1, 1e-9, 0.999999, 2.0 ** -32):
        assert g.dropout_threshold(p) == ring.dropout_threshold(p)


def test_sparse_argument_errors_before_launch(zr):
    p = 1 << 40
    ws = zr.zr_sparse_workspace_size(2, 1000, 4)
    call = lambda **kw: zr.zr_sparse_aggregate(  # noqa: E731
        kw.get("idx", [p, p]), kw.get("val", [p, p]), kw.get("nnz", [3, 4]), kw.get("n", 2),
        kw.get("m", 1000), kw.get("parts", 4), 0, kw.get("avg", 0), p, p, kw.get("cap", 7), p, p,
        kw.get("ws", p), kw.get("ws_bytes", ws), None)
    assert call(n=0) == zr.ZR_ERR_INVALID_ARG
    assert call(m=0) == zr.ZR_ERR_INVALID_ARG
    assert call(m=1 << 31) == zr.ZR_ERR_INVALID_ARG
    assert call(parts=zr.ZR_MAX_PARTS + 1) == zr.ZR_ERR_INVALID_ARG
    assert call(avg=3) == zr.ZR_ERR_INVALID_ARG
    assert call(nnz=[3, -1]) == zr.ZR_ERR_INVALID_ARG
    assert call(idx=[p, 0]) == zr.ZR_ERR_INVALID_ARG
    assert call(cap=6) == zr.ZR_ERR_CAPACITY
    assert call(ws_bytes=ws - 1) == zr.ZR_ERR_CAPACITY
    assert call(ws=p + 8) == zr.ZR_ERR_ALIGNMENT
    assert call(ws=0) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_partition(p, p, 10, 0, 0, p, p, p, p, 1 << 20, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_partition(p, p, -1, 4, 0, p, p, p, p, 1 << 20, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_partition(p, p, 10, 4, 0, p, p, p, p, 1, None) == zr.ZR_ERR_CAPACITY


def test_skip_fraction_to_k(zr):
    assert zr.skip_fraction_to_k(0.5, 8) == 4
    assert zr.skip_fraction_to_k(0.25, 8) == 2
    assert zr.skip_fraction_to_k(0.0, 8) == 0
    with pytest.raises(ValueError):
        zr.skip_fraction_to_k(0.3, 8)
    with pytest.raises(ValueError):
        zr.skip_fraction_to_k(1.0, 8)


def test_choose_scheme_host_call_matches_oracle(zr):
    # zr_choose_scheme is plain host arithmetic: it runs here, without a GPU.
    from oracle import stats

    rng = np.random.default_rng(8)
    for n in (2, 4, 8, 16, 32, 64):
        logn = n.bit_length() - 1
        for trial in range(50):
            nnz_total = int(rng.integers(1, 10**7))
            counts = [nnz_total]
            for level in range(1, logn + 1):
                counts.append(int(rng.integers(max(1, counts[-1] // 2), counts[-1] + 1)))
            choice, g, bp, hc = zr.zr_choose_scheme(counts, n)
            want_g = stats.gammas_from_counts(counts, nnz_total, n)
            want_choice, want_bp, want_hc = stats.choose_scheme(want_g, n)
            assert choice == want_choice
            assert g == pytest.approx(want_g, rel=1e-12)
            assert bp == pytest.approx(want_bp, rel=1e-12) and hc == pytest.approx(want_hc, rel=1e-12)
    assert zr.zr_choose_scheme([10, 5], 3)[0] == -1     # not a power of two
    assert zr.zr_choose_scheme([0, 0], 2)[0] == -1      # no entries
    assert zr.zr_choose_scheme([10, -1], 2)[0] == -1


def test_densification_argument_errors_before_launch(zr):
    p = 1 << 40
    ws = zr.zr_densification_workspace_size(4, 1000)
    assert ws > 0
    assert zr.zr_densification_workspace_size(3, 1000) == 0
    call = lambda **kw: zr.zr_densification(  # noqa: E731
        [p] * kw.get("n", 4), kw.get("nnz", [3, 4, 5, 6]), kw.get("n", 4), kw.get("m", 1000), p,
        kw.get("ws", p), kw.get("ws_bytes", ws), None)
    assert call(n=3, nnz=[1, 2, 3]) == zr.ZR_ERR_INVALID_ARG
    assert call(m=0) == zr.ZR_ERR_INVALID_ARG
    assert call(nnz=[3, -1, 5, 6]) == zr.ZR_ERR_INVALID_ARG
    assert call(nnz=[3, 4, 5, 2000]) == zr.ZR_ERR_INVALID_ARG
    assert call(ws=p + 8) == zr.ZR_ERR_ALIGNMENT
    assert call(ws_bytes=ws - 1) == zr.ZR_ERR_CAPACITY


def test_hash_bitmap_sizes_and_argument_errors_before_launch(zr):
    hdr = open(os.path.join(ROOT, "include", "zr.h")).read()
    m = re.search(r"#define ZR_HASH_RANGE (\d+)", hdr)
    assert m and zr.ZR_HASH_RANGE == int(m.group(1))
    rng = zr.ZR_HASH_RANGE
    for dense, parts in ((1, 1), (rng, 8), (rng + 1, 8), ((1 << 25), 16), ((1 << 31) - 1, 256)):
        ranges = -(-dense // rng)
        stride = (ranges + 1 + 3) // 4 * 4
        nb = max(0, (parts - 1).bit_length())
        counts = -(-(parts * stride * 4) // 256) * 256
        assert zr.zr_hash_directory_size(dense, parts) == 256 + counts + ranges * nb * 32 * 8
        assert zr.zr_hash_bitmap_workspace_size(dense, parts) > 0
    for bad in ((0, 8), ((1 << 31), 8), (100, 0), (100, zr.ZR_MAX_PARTS + 1)):
        assert zr.zr_hash_directory_size(*bad) == 0
        assert zr.zr_hash_bitmap_workspace_size(*bad) == 0
    p = 1 << 40
    dsz = zr.zr_hash_directory_size(1000, 4)
    assert zr.zr_hash_directory(1000, 4, 0, None, dsz, None) == zr.ZR_ERR_INVALID_ARG
    assert zr.zr_hash_directory(1000, 4, 0, p + 4, dsz, None) == zr.ZR_ERR_ALIGNMENT
    assert zr.zr_hash_directory(1000, 4, 0, p, dsz - 1, None) == zr.ZR_ERR_CAPACITY
    ws = zr.zr_hash_bitmap_workspace_size(1000, 4)
    cap = (1000 + 31) // 32 + 4
    enc = lambda **kw: zr.zr_hash_bitmap_encode(  # noqa: E731
        kw.get("dir", p), 1000, 4, 0, kw.get("keys", p), kw.get("n_keys", 10), p,
        kw.get("cap", cap), p, kw.get("ws", p), kw.get("ws_bytes", ws), None)
    assert enc(dir=None) == zr.ZR_ERR_INVALID_ARG
    assert enc(keys=None) == zr.ZR_ERR_INVALID_ARG
    assert enc(n_keys=-1) == zr.ZR_ERR_INVALID_ARG
    assert enc(cap=cap - 1) == zr.ZR_ERR_CAPACITY
    assert enc(ws=p + 8) == zr.ZR_ERR_ALIGNMENT
    assert enc(ws_bytes=ws - 1) == zr.ZR_ERR_CAPACITY
    dec = lambda **kw: zr.zr_hash_bitmap_decode(  # noqa: E731
        kw.get("dir", p), 1000, 4, 0, p, kw.get("out", p), kw.get("cap", 10), p, p,
        kw.get("ws_bytes", ws), None)
    assert dec(dir=None) == zr.ZR_ERR_INVALID_ARG
    assert dec(out=None) == zr.ZR_ERR_INVALID_ARG
    assert dec(cap=-1) == zr.ZR_ERR_INVALID_ARG
    assert dec(ws_bytes=ws - 1) == zr.ZR_ERR_CAPACITY
