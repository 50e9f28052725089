"""C ABI checks that need no GPU: the library loads, exports every entry
point the header declares, validates arguments before touching CUDA, and its
host LPT matches the oracle's bit for bit."""

import os
import re

import numpy as np
import pytest

from oracle import lpt as olpt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mos():
    import matrix_optimizer_step_gb300 as m
    from matrix_optimizer_step_gb300 import build

    build.build()
    m.load_library()
    return m


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"DMUON_API\s+[\w\s\*]+?\b(dmuon_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(mos):
    lib = mos.load_library()
    names = _declared_symbols()
    assert "dmuon_muon_step" in names and "dmuon_lpt_assign" in names and "dmuon_adamw_step" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(mos.capi.EXPORTED) == names


def test_status_strings(mos):
    for s in range(0, 9):
        assert mos.dmuon_status_string(s)
    assert mos.dmuon_status_string(99) == "unknown status"


def test_lpt_bit_exact_vs_oracle(mos):
    r = np.random.default_rng(0)
    for trial in range(200):
        n = int(r.integers(0, 300))
        R = int(r.integers(1, 160))
        hi = int(r.choice([2, 10, 1000, 10 ** 12]))
        sizes = [int(x) for x in r.integers(0, hi, n)]
        got = mos.dmuon_lpt_assign(sizes, R)
        want = olpt.lpt_assign(sizes, R)
        assert got[0] == want[0] and got[1] == want[1], (trial, n, R)


def test_lpt_large_tile_list_vs_oracle(mos):
    # The size of a real tile list: ~30k tiles of a few distinct costs on 148 slots.
    r = np.random.default_rng(1)
    sizes = [int(x) for x in r.choice([18, 66, 226], 30000)]
    got = mos.dmuon_lpt_assign(sizes, 148)
    want = olpt.lpt_assign(sizes, 148)
    assert got == (want[0], want[1])


def test_lpt_graham_tight_instance(mos):
    for R in (2, 4, 8):
        sizes = []
        for k in range(2 * R - 1, R, -1):
            sizes += [k, k]
        sizes += [R, R, R]
        _, loads = mos.dmuon_lpt_assign(sizes, R)
        assert max(loads) == 4 * R - 1


def test_lpt_errors(mos):
    with pytest.raises(mos.DmuonError) as e:
        mos.dmuon_lpt_assign([1, 2], 0)
    assert e.value.status == 1
    with pytest.raises(mos.DmuonError):
        mos.dmuon_lpt_assign([1, -1], 2)
    with pytest.raises(mos.DmuonError):
        mos.dmuon_lpt_assign([2 ** 62, 2 ** 62], 1)
    assert mos.dmuon_lpt_assign([], 3) == ([], [0, 0, 0])


def test_muon_step_host_validation_without_gpu(mos):
    # Host-side validation runs before any CUDA call, so it works here.
    capi = mos.capi
    ctx = mos.dmuon_context_create(0)
    try:
        d = capi.DmuonMatrix()
        d.rank = 1
        d.shape[0] = 128
        d.master, d.momentum, d.grad = 1 << 20, 2 << 20, 3 << 20  # fake, never dereferenced
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step(ctx, [d], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        assert e.value.status == capi.DMUON_ERR_RANK_LT2
        d.rank = 2
        d.shape[0], d.shape[1] = 8, 0
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step(ctx, [d], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        assert e.value.status == capi.DMUON_ERR_SHAPE
        d.shape[1] = 16
        d.grad_dtype = 7
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step(ctx, [d], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        assert e.value.status == capi.DMUON_ERR_DTYPE
        d.grad_dtype = capi.DMUON_DTYPE_BF16
        d.grad = None
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step(ctx, [d], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step(ctx, [], float("nan"), 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        with pytest.raises(mos.DmuonError):
            mos.dmuon_muon_step(ctx, [], 0.02, 0.95, 0.01, 101, 3.4445, -4.775, 2.0315, stream=0)
        mos.dmuon_muon_step(ctx, [], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
        with pytest.raises(mos.DmuonError):
            mos.dmuon_adamw_step(ctx, [], 1e-3, 0.9, 0.95, 1e-8, 0.0, 0, stream=0)
        with pytest.raises(mos.DmuonError):
            mos.dmuon_adamw_step(ctx, [], 1e-3, 1.0, 0.95, 1e-8, 0.0, 1, stream=0)
    finally:
        mos.dmuon_context_destroy(ctx)


def test_overlapping_written_memory_rejected_without_gpu(mos):
    """Memory a step writes (master, momentum, bf16 param; AdamW master and
    moments) may not overlap other written memory or a gradient, within a
    tensor or across tensors; gradients may share memory.  Checked on the
    host before any CUDA call (fake pointers, never dereferenced)."""
    capi = mos.capi
    MiB = 1 << 20

    def mat(master, momentum, grad, param=None, shape=(8, 16)):
        d = capi.DmuonMatrix()
        d.rank = len(shape)
        for i, s in enumerate(shape):
            d.shape[i] = s
        d.master, d.momentum, d.grad = master, momentum, grad
        d.param_bf16 = param
        d.grad_dtype = capi.DMUON_DTYPE_BF16
        return d

    def vec(master, m, v, grad, numel=100, param=None):
        t = capi.DmuonVector()
        t.numel = numel
        t.master, t.exp_avg, t.exp_avg_sq, t.grad = master, m, v, grad
        t.param_bf16 = param
        t.grad_dtype = capi.DMUON_DTYPE_F32
        return t

    def muon_status(mats):
        try:
            mos.dmuon_muon_step(ctx, mats, 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
            return 0, ""
        except mos.DmuonError as e:
            return e.status, str(e)

    ctx = mos.dmuon_context_create(0)
    try:
        # 8 x 16 fp32 = 512 bytes per buffer.
        bad = [
            [mat(1 * MiB, 1 * MiB + 256, 3 * MiB)],                    # master / momentum, same tensor
            [mat(1 * MiB, 2 * MiB, 1 * MiB + 500)],                    # grad inside master
            [mat(1 * MiB, 2 * MiB, 3 * MiB, param=2 * MiB + 510)],     # param inside momentum
            [mat(1 * MiB, 2 * MiB, 3 * MiB), mat(4 * MiB, 1 * MiB + 4, 5 * MiB)],  # across tensors
            [mat(1 * MiB, 2 * MiB, 3 * MiB), mat(4 * MiB, 5 * MiB, 2 * MiB)],      # grad = other's momentum
        ]
        for mats in bad:
            status, msg = muon_status(mats)
            assert status == capi.DMUON_ERR_INVALID_ARG and "overlaps" in msg, (status, msg)
        good = [
            [mat(1 * MiB, 1 * MiB + 512, 3 * MiB, param=1 * MiB + 1024)],  # adjacent, not overlapping
            [mat(1 * MiB, 2 * MiB, 3 * MiB), mat(4 * MiB, 5 * MiB, 3 * MiB)],  # shared gradient
        ]
        for mats in good:
            status, msg = muon_status(mats)
            assert "overlaps" not in msg, msg  # fails later only for want of a device here
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_adamw_step(ctx, [vec(1 * MiB, 2 * MiB, 3 * MiB, 4 * MiB),
                                       vec(5 * MiB, 2 * MiB + 396, 6 * MiB, 7 * MiB)],
                                 1e-3, 0.9, 0.95, 1e-8, 0.0, 1, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG and "overlaps" in str(e.value)
        # Across the two routes of one host-buffer step.
        hp = capi.muon_hparams(0.02, 0.95, 0.01)
        ap = capi.adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.0, 1)
        with pytest.raises(mos.DmuonError) as e:
            capi.dmuon_step_host(ctx, [mat(1 * MiB, 2 * MiB, 3 * MiB)], [capi.DmuonHostIO(512, None)], hp,
                                 vecs=[vec(1 * MiB + 64, 5 * MiB, 6 * MiB, 7 * MiB)],
                                 vec_io=[capi.DmuonHostIO(512, None)], adamw=ap, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG and "overlaps" in str(e.value)
    finally:
        mos.dmuon_context_destroy(ctx)


def test_golden_last_two_dims_accepted_ranks(mos):
    """The pages' table: [128] is rejected (rank 1); [8,16] and [4,8,16] pass
    host validation (they only fail later for lack of a device here)."""
    import json

    capi = mos.capi
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "last_two_dims.json")))
    ctx = mos.dmuon_context_create(0)
    try:
        for case in gold["cases"]:
            d = capi.DmuonMatrix()
            d.rank = len(case["shape"])
            for i, s in enumerate(case["shape"]):
                d.shape[i] = s
            d.master, d.momentum, d.grad = 1 << 20, 2 << 20, 3 << 20  # fake, never dereferenced
            d.grad_dtype = capi.DMUON_DTYPE_BF16
            try:
                mos.dmuon_muon_step(ctx, [d], 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, stream=0)
                status = 0
            except mos.DmuonError as e:
                status = e.status
            if case["accepted"]:
                assert status in (0, capi.DMUON_ERR_UNSUPPORTED, capi.DMUON_ERR_CUDA), case
            else:
                assert status == capi.DMUON_ERR_RANK_LT2, case
    finally:
        mos.dmuon_context_destroy(ctx)



def test_layered_lpt_bit_exact_vs_oracle(mos):
    r = np.random.default_rng(2)
    for trial in range(150):
        n = int(r.integers(0, 200))
        R = int(r.integers(1, 40))
        n_layers = int(r.integers(1, 30))
        sizes = [int(x) for x in (10 ** r.uniform(3, 8, n)).astype(np.int64)]
        layers = [int(x) for x in r.integers(-1, n_layers, n)]
        thr = int(r.choice([0, 5_000_000, 10 ** 7]))
        got = mos.dmuon_lpt_assign_layered(sizes, layers, R, thr)
        want = olpt.lpt_assign_layered(sizes, layers, R, thr)
        assert got[0] == want[0] and got[1] == want[1], trial


def test_layered_lpt_llama_owner_partition(mos):
    from matrix_optimizer_step_gb300 import workloads

    wl = workloads.workload("llama3_8b")
    numels = [s.numel for s in wl.matrices]
    layers = [int(s.name.split(".")[1]) for s in wl.matrices]
    got = mos.owner_partition(numels, 8, layers=layers)
    want = olpt.lpt_assign_layered(numels, layers, 8)
    assert list(got[0]) == want[0] and list(got[1]) == want[1]
    with pytest.raises(mos.DmuonError):
        mos.dmuon_lpt_assign_layered([1, -2], [0, 0], 2)


def test_step_host_host_validation_without_gpu(mos):
    capi = mos.capi
    hp = capi.muon_hparams(0.02, 0.95, 0.01)
    ctx = mos.dmuon_context_create(0)
    try:
        d = capi.DmuonMatrix()
        d.rank = 2
        d.shape[0], d.shape[1] = 8, 16
        d.master, d.momentum, d.grad = 1 << 20, 2 << 20, 3 << 20  # fake, never dereferenced
        d.grad_dtype = capi.DMUON_DTYPE_BF16
        io = capi.DmuonHostIO(512, None)
        for groups in (0, 65):
            with pytest.raises(mos.DmuonError) as e:
                capi.dmuon_step_host(ctx, [d], [io], hp, n_groups=groups, stream=0)
            assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        with pytest.raises(mos.DmuonError) as e:  # hyper-parameters missing
            capi.dmuon_step_host(ctx, [d], [io], None, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        with pytest.raises(mos.DmuonError) as e:  # no host gradient
            capi.dmuon_step_host(ctx, [d], [capi.DmuonHostIO(None, None)], hp, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        with pytest.raises(mos.DmuonError) as e:  # host parameter but no device parameter
            capi.dmuon_step_host(ctx, [d], [capi.DmuonHostIO(512, 1024)], hp, stream=0)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        d.rank = 1
        with pytest.raises(mos.DmuonError) as e:
            capi.dmuon_step_host(ctx, [d], [io], hp, stream=0)
        assert e.value.status == capi.DMUON_ERR_RANK_LT2
        capi.dmuon_step_host(ctx, [], [], None, stream=0)  # nothing to do
    finally:
        mos.dmuon_context_destroy(ctx)


def test_set_tuning_rejects_unknown_keys_and_bad_values(mos):
    capi = mos.capi
    for key, value in ((0, 1), (1, 0), (1, 1), (5, 0), (13, 1), (12, -1), (-3, 0), (8, -1), (9, 0), (9, 17), (10, 0), (10, 70000), (11, 0), (11, 1 << 21)):
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_set_tuning(key, value)
        assert e.value.status == capi.DMUON_ERR_INVALID_ARG, (key, value)
    # Valid settings are accepted and put back to the defaults.
    for key, value, default in ((8, 0, 32), (9, 4, 1), (10, 1, 1024), (11, 1, 32768), (7, 0, 1), (12, 0, 128)):
        mos.dmuon_set_tuning(key, value)
        mos.dmuon_set_tuning(key, default)


def test_noalloc_validation_without_gpu(mos):
    """The allocation-free entry point applies dmuon_muon_step's shape checks
    and its own size limit on the host, before any CUDA call, and without
    overflowing its size sums (fake pointers: never dereferenced)."""
    capi = mos.capi

    def desc(shape, dtype=capi.DMUON_DTYPE_BF16):
        d = capi.DmuonMatrix()
        d.rank = len(shape)
        for i, s in enumerate(shape[:4]):
            d.shape[i] = s
        d.grad_dtype = dtype
        d.master, d.momentum, d.grad = 1 << 40, 2 << 40, 3 << 40
        return d

    def status(d, flags=capi.DMUON_FLAG_NESTEROV):
        with pytest.raises(mos.DmuonError) as e:
            mos.dmuon_muon_step_noalloc(d, 0.02, 0.95, 0.01, 5, 3.4445, -4.775, 2.0315, flags=flags, stream=0)
        return e.value.status, str(e.value)

    # Products that would wrap 2^64 in a naive size sum, and a slice of 2^62 elements.
    assert status(desc((1 << 31, 1 << 31, 8, 8)))[0] == capi.DMUON_ERR_SHAPE
    assert status(desc((1 << 31, 1 << 31)))[0] == capi.DMUON_ERR_SHAPE
    assert status(desc((1 << 20, 1 << 20, 2)))[0] == capi.DMUON_ERR_SHAPE
    assert status(desc((65536 * 128 + 1, 1)))[0] == capi.DMUON_ERR_SHAPE
    # Over the static limit: message names it.
    st, msg = status(desc((4096, 4096)))
    assert st == capi.DMUON_ERR_SHAPE and "static limit" in msg
    st, msg = status(desc((2048, 2048)), flags=capi.DMUON_FLAG_FP32_NS)  # fp32 path: 8 B per element per X
    assert st == capi.DMUON_ERR_SHAPE and "static limit" in msg
    st, msg = status(desc((40000, 8, 8)))  # small scratch, tables over 1 MiB
    assert st == capi.DMUON_ERR_SHAPE and "static limit" in msg
    # Other checks of the main entry point.
    assert status(desc((5,)))[0] == capi.DMUON_ERR_RANK_LT2
    assert status(desc((2, 2, 2, 2, 2)))[0] == capi.DMUON_ERR_SHAPE
    assert status(desc((0, 8)))[0] == capi.DMUON_ERR_SHAPE
    assert status(desc((8, 8), dtype=7))[0] == capi.DMUON_ERR_DTYPE
    assert status(desc((8, 8)), flags=4)[0] == capi.DMUON_ERR_INVALID_ARG
    d = desc((8, 8))
    d.momentum = d.master  # written memory shared
    assert status(d)[0] == capi.DMUON_ERR_INVALID_ARG


def test_context_tuning_is_per_context_without_gpu(mos):
    """A context copies the process-wide defaults when created; changing the
    defaults later or another context's copy leaves it alone (no GPU: the
    setters are host-only)."""
    capi = mos.capi
    a = mos.dmuon_context_create(0)
    try:
        mos.dmuon_set_tuning(12, 7)  # default for contexts created from now on
        b = mos.dmuon_context_create(0)
        try:
            mos.dmuon_context_set_tuning(a, 8, 0)
            mos.dmuon_context_set_tuning(b, 8, 1000)
            for key, value in ((1, 0), (13, 1), (8, -1), (9, 0)):
                with pytest.raises(mos.DmuonError) as e:
                    mos.dmuon_context_set_tuning(a, key, value)
                assert e.value.status == capi.DMUON_ERR_INVALID_ARG
            with pytest.raises(mos.DmuonError) as e:
                mos.dmuon_context_set_tuning(None, 8, 0)
            assert e.value.status == capi.DMUON_ERR_INVALID_ARG
        finally:
            mos.dmuon_context_destroy(b)
    finally:
        mos.dmuon_set_tuning(12, 128)
        mos.dmuon_context_destroy(a)
