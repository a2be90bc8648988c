"""C-ABI host side, no GPU: the library loads, exports every declared symbol,
and its plan (pure host logic) equals the oracle's plan integer for integer."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from hsdp_sharded_parameter_gb300 import capi as C
from hsdp_sharded_parameter_gb300 import workloads as WL


def test_library_exports_every_declared_symbol():
    names = C.header_symbols()
    assert len(names) >= 20
    lib = C.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []


PLANS = [(4, 1, [7, 16, 5, 3], [8, 8, 1, 4]),
         (3, 2, [0, 1, 2, 10, 11, 40], [5, 1, 17, 3, 1, 2]),
         (1, 8, [9, 4], [3, 1]),
         (8, 2, [1, 2, 3, 4, 5, 6, 7, 8, 9], [1] * 9),
         (5, 3, list(range(30)), [1 + i % 7 for i in range(30)])]


def same_plan(cp, op):
    assert (cp.W, cp.S, cp.D, cp.P, cp.sum_padded) == (op.W, op.S, op.D, op.P, op.sum_padded)
    assert np.array_equal(cp.offsets(), op.o)
    for p in range(op.P):
        assert cp.padded_sharded_param_size(p) == op.dss[p]
        for s in range(op.S):
            assert cp.sharded_size(p, s) == (op.off[p, s], op.len[p, s])
    for dt in ["f32", "bf16"]:
        assert cp.slice_numel(dt) == op.slice(dt)
    for w in range(op.W):
        a, b = cp.group_ranks(w), op.group_ranks(w)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert cp.comm_calls() == op.comm_calls()


@pytest.mark.parametrize("S,D,d0,inner", PLANS)
def test_plan_equals_oracle(S, D, d0, inner):
    same_plan(C.Plan(d0, inner, S * D, S), O.Layout(d0, inner, S * D, S))


@pytest.mark.parametrize("key", WL.ORDER)
def test_workload_plans_equal_oracle(key):
    wl = WL.WORKLOADS[key]
    same_plan(C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size),
              O.Layout(wl.d0, wl.inner, wl.rank_size, wl.shard_size))


def test_enable_param_shard_off_forces_shard_size_one():
    cp = C.Plan([8, 3], [4, 1], 8, 4, enable_param_shard=0)
    assert (cp.S, cp.D) == (1, 8)
    assert cp.comm_calls() == (0, 8)


def test_errors_are_reported_not_crashed():
    with pytest.raises(C.FsdpError) as e:
        C.Plan([7], [8], 4, 4, shard_dim=1)
    assert e.value.code == C.FSDP_ERR_NOT_IMPLEMENTED and "shard_dim" in str(e.value)
    with pytest.raises(C.FsdpError) as e:
        C.Plan([7], [8], 6, 4)
    assert e.value.code == C.FSDP_ERR_INVALID_ARG
    with pytest.raises(C.FsdpError) as e:
        C.Plan([7], [0], 4, 4)
    assert e.value.code == C.FSDP_ERR_INVALID_ARG
    cp = C.Plan([7], [8], 4, 4)
    with pytest.raises(C.FsdpError):
        cp.sharded_size(1, 0)
    with pytest.raises(C.FsdpError):
        cp.sharded_size(0, 4)
    lib = C.lib()
    assert lib.fsdp_plan_destroy(None) == 0
    h = ctypes.c_void_p()
    # a data call on a plan that was never uploaded is refused on the host
    rc = lib.fsdp_rs_ar_reduce(cp.handle, None, None, None)
    assert rc == C.FSDP_ERR_INVALID_ARG and b"not uploaded" in lib.fsdp_last_error()
    rc = lib.fsdp_bind(cp.handle, 0, 0, None, None, ctypes.byref(h))
    assert rc == C.FSDP_ERR_INVALID_ARG


def test_wait_limit_and_status_calls_check_their_arguments():
    # the failure-detection calls of the capped sync: settable on a host-only
    # plan; reading the status word needs the uploaded plan (it lives in the
    # plan's device memory) and refuses a NULL output
    cp = C.Plan([7], [8], 4, 4)
    assert cp.set_wait_limit(5_000_000) is cp
    assert cp.set_wait_limit(0) is cp  # 0 restores the default
    assert cp.inject_stall(True) is cp and cp.inject_stall(False) is cp
    lib = C.lib()
    st = ctypes.c_int(-1)
    rc = lib.fsdp_plan_status(cp.handle, None, ctypes.byref(st))
    assert rc == C.FSDP_ERR_INVALID_ARG and b"not uploaded" in lib.fsdp_last_error()
    assert st.value == -1
    for fn, arg in [(lib.fsdp_plan_set_wait_limit, 1), (lib.fsdp_plan_inject_stall, 1)]:
        assert fn(None, arg) == C.FSDP_ERR_INVALID_ARG
    assert lib.fsdp_plan_status(None, None, ctypes.byref(st)) == C.FSDP_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_upload_without_gpu_fails_cleanly():
    cp = C.Plan([7], [8], 4, 4)
    with pytest.raises(C.FsdpError) as e:
        cp.upload()
    assert e.value.code in (C.FSDP_ERR_CUDA, C.FSDP_ERR_NOMEM)


@pytest.mark.parametrize("seed", range(6))
def test_bucketed_plans_equal_oracle(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.integers(1, 25))
    S, D = int(rng.integers(1, 9)), int(rng.integers(1, 4))
    d0 = [int(x) for x in rng.integers(0, 500, P)]
    inner = [int(x) for x in rng.choice([1, 2, 5, 64, 128], P)]
    bucket = sorted(int(x) for x in rng.integers(0, 5, P))
    same_plan(C.Plan(d0, inner, S * D, S, bucket=bucket), O.Layout(d0, inner, S * D, S, bucket=bucket))


def test_bucket_order_is_checked():
    with pytest.raises(C.FsdpError) as e:
        C.Plan([4, 4], [1, 1], 4, 4, bucket=[1, 0])
    assert e.value.code == C.FSDP_ERR_INVALID_ARG and "bucket" in str(e.value)


# Host-side sanitizer of the work tables (compute-sanitizer is not used):
# every run of every kernel's table reads and writes inside the buffers at
# the sizes the bindings require, every destination is covered exactly once,
# and the tile prefix the kernels search matches the runs.
@pytest.mark.parametrize("key", WL.ORDER)
def test_workload_tables_stay_in_bounds(key):
    wl = WL.WORKLOADS[key]
    C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size).check_tables()


def test_random_plan_tables_stay_in_bounds():
    rng = np.random.default_rng(2024)
    for _ in range(300):
        P = int(rng.integers(1, 12))
        S, D = int(rng.integers(1, 17)), int(rng.integers(1, 5))
        d0 = [int(x) for x in rng.integers(0, 3000, P)]
        d0[int(rng.integers(0, P))] = int(rng.integers(0, S + 1))  # short params: empty shards
        inner = [int(x) for x in rng.choice([1, 2, 3, 7, 64, 127, 4096], P)]
        bucket = sorted(int(x) for x in rng.integers(0, 4, P)) if rng.integers(0, 2) else None
        C.Plan(d0, inner, S * D, S, bucket=bucket).check_tables()


def test_tables_of_a_very_long_parameter_list_stay_in_bounds():
    rng = np.random.default_rng(5)
    P = 100_000
    d0 = [int(x) for x in rng.integers(0, 20, P)]
    inner = [int(x) for x in rng.choice([1, 2, 5, 64], P)]
    C.Plan(d0, inner, 16, 8).check_tables()


def test_error_messages_are_per_thread():
    # fsdp_last_error() is thread-local: threads that fail differently at the
    # same time each read back their own message, while other threads build
    # and check plans concurrently
    import threading

    lib = C.lib()
    results, errors = {}, []
    barrier = threading.Barrier(8)

    def failing(i):
        barrier.wait()
        for _ in range(200):
            d0 = (ctypes.c_int64 * 1)(7)
            inner = (ctypes.c_int64 * 1)(8)
            h = ctypes.c_void_p()
            if i % 2:
                rc = lib.fsdp_plan_create(1, d0, inner, 6, 4, 1, 0, ctypes.byref(h))  # 6 % 4 != 0
            else:
                rc = lib.fsdp_plan_create(1, d0, inner, 4, 4, 1, 1, ctypes.byref(h))  # shard_dim 1
            msg = lib.fsdp_last_error().decode()
            if (i % 2 and (rc != C.FSDP_ERR_INVALID_ARG or "shard_dim" in msg)) or \
               (not i % 2 and (rc != C.FSDP_ERR_NOT_IMPLEMENTED or "shard_dim" not in msg)):
                errors.append((i, rc, msg))
        results[i] = True

    def building(i):
        barrier.wait()
        for k in range(50):
            C.Plan([7 + k, 16, 5], [8, 1, 3], 8, 4).check_tables()
        results[i] = True

    threads = [threading.Thread(target=failing if i < 6 else building, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert errors == [] and len(results) == 8


def test_pointer_lists_are_checked_before_the_library_reads_them():
    # the library reads W*P (or W) pointers from the arrays it is given; the
    # binding refuses a list of another length, and for the allocation-free
    # call also tensors of the wrong dtype or not on a GPU, before any call
    import torch

    plan = C.Plan([7, 16], [8, 1], 4, 2)  # host-only: no GPU needed
    g = torch.zeros(8, dtype=torch.bfloat16)
    f = torch.zeros(plan.slice_numel("f32"), dtype=torch.float32)
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.fsdp_rs_ar_reduce_noalloc(plan, "bf16", [g] * 7, [f] * 4)
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.fsdp_rs_ar_reduce_noalloc(plan, "bf16", [g] * 8, [f] * 3)
    with pytest.raises(C.FsdpError, match="expected contiguous"):  # CPU tensors
        C.fsdp_rs_ar_reduce_noalloc(plan, "bf16", [g] * 8, [f] * 4)
    with pytest.raises(C.FsdpError, match="expected contiguous"):  # wrong dtype
        C.fsdp_rs_ar_reduce_noalloc(plan, "bf16", [g.float()] * 8, [f] * 4)
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.Binding(plan, "grads", "bf16", [g] * 3)
    with pytest.raises(C.FsdpError, match="tensors given"):
        C.Binding(plan, "fused", "f32", [f] * 5, check_sizes=False)
