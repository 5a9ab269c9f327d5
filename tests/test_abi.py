"""CPU checks of the C ABI: the library builds and loads without a GPU, exports every
function include/zopt.h declares, validates arguments before any launch, and its host-only
layout (deg/zero.py, ZeroMaster) equals the oracle's bit for bit."""
import ctypes

import numpy as np
import pytest

import workloads
from oracle import layout as OL
from zero_sharded_optimizer_flat_gb300 import build_lib

build_lib.build()
import zero_sharded_optimizer_flat_gb300 as Z  # noqa: E402


def test_exports_every_declared_symbol():
    names = Z.declared_functions()
    assert "zopt_adamw_step" in names and "zopt_grad_norm_clip" in names and "zopt_shard_layout" in names
    L = ctypes.CDLL(Z.LIB_PATH)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert Z.lib().zopt_version().startswith(b"zopt")


def _check_layout(numel, decay, bucket, world):
    for rank in range(world):
        lay = Z.ShardLayout(numel, decay, bucket, world, rank)
        assert lay.numel == sum(numel)
        assert lay.shard_len == OL.shard_len(numel, bucket, world)
        assert [(s, e, p) for s, e, p, _ in lay.buckets()] == OL.buckets(numel, bucket, world)
        segs = [tuple(int(x) for x in r) for r in lay.segments()]
        assert segs == OL.segments(numel, bucket, world, rank)
        mask = OL.decay_mask_of_shard(list(decay), numel, bucket, world, rank)
        ref_nd = np.zeros(lay.shard_len, bool)
        ref_nd[mask == 0] = True
        got_nd = np.zeros(lay.shard_len, bool)
        runs = lay.nodecay_runs()
        for b, e in runs:
            assert b < e
            got_nd[b:e] = True
        assert np.array_equal(got_nd, ref_nd)
        # sorted, disjoint and not adjacent
        assert np.all(runs[1:, 0] > runs[:-1, 1])


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_layout_matches_oracle_random(world):
    rng = np.random.default_rng(world)
    for trial in range(25):
        k = int(rng.integers(1, 12))
        numel = [int(x) for x in rng.integers(0, 40, size=k)]
        if sum(numel) == 0:
            numel[0] = 1
        decay = [bool(x) for x in rng.integers(0, 2, size=k)]
        bucket = int(rng.integers(1, 50))
        _check_layout(numel, decay, bucket, world)


def test_layout_matches_oracle_workloads():
    for name in ("c1", "c2", "c3"):
        w = workloads.get(name)
        numel = [p.numel for p in w.adamw]
        decay = [p.decay for p in w.adamw]
        lay = Z.ShardLayout(numel, decay, w.bucket, w.world, w.rank)
        assert lay.shard_len == OL.shard_len(numel, w.bucket, w.world)
        assert [tuple(int(x) for x in r) for r in lay.segments()] == OL.segments(numel, w.bucket, w.world, w.rank)
    w = workloads.get("c4")
    lay = Z.ShardLayout([p.numel for p in w.adamw], [p.decay for p in w.adamw], w.bucket, 8, 0)
    assert lay.shard_len == 250_000_000 and len(lay.buckets()) == 60


@pytest.mark.parametrize("args,frag", [
    (([], None, 16, 1, 0), "needs trainable parameters"),
    (([0, 0], None, 16, 1, 0), "empty"),
    (([4], None, 16, 0, 0), "world"),
    (([4], None, 16, 2, 2), "rank"),
    (([4], None, 0, 1, 0), "bucket"),
    (([-1, 4], None, 16, 1, 0), "negative"),
])
def test_layout_rejects_bad_arguments(args, frag):
    with pytest.raises(Z.ZoptError) as e:
        Z.ShardLayout(*args)
    assert e.value.status == 1 and frag in str(e.value)


def test_device_calls_validate_before_launch():
    """Every call below fails validation, so none reaches a launch (the pointers are fake)."""
    L = Z.lib()
    stats = ctypes.c_void_p(256)
    # n < 1, NULL grad, misaligned grad, short workspace: all rejected without touching CUDA
    assert L.zopt_grad_norm_clip(None, 0, 0, 1.0, None, 0, stats, None) == 1
    assert L.zopt_grad_norm_clip(None, 0, 8, 1.0, None, 0, stats, None) == 1
    assert L.zopt_grad_norm_clip(ctypes.c_void_p(4), 0, 8, 1.0, ctypes.c_void_p(256), 4096, stats, None) == 1
    assert b"aligned" in L.zopt_last_error()
    assert L.zopt_grad_norm_clip(ctypes.c_void_p(256), 0, 8, 1.0, ctypes.c_void_p(256), 8, stats, None) == 1
    assert b"workspace" in L.zopt_last_error()
    assert L.zopt_grad_norm_clip(ctypes.c_void_p(256), 7, 8, 1.0, ctypes.c_void_p(256), 4096, stats, None) == 2
    assert L.zopt_grad_norm_clip(ctypes.c_void_p(256), 0, 8, -1.0, ctypes.c_void_p(256), 4096, stats, None) == 1
    lay = Z.ShardLayout([100, 3], [1, 0], 64, 1, 0)
    hp = Z._Hparams(1e-3, 0.9, 0.95, 1e-8, 0.1, 1, 0)
    p = ctypes.c_void_p(1 << 20)
    tab = ctypes.c_void_p(4096)
    bad = Z._Hparams(1e-3, 1.0, 0.95, 1e-8, 0.1, 1, 0)
    assert L.zopt_adamw_step(lay.handle, tab, p, p, p, p, 1, None, ctypes.byref(bad), None, p, None) == 1
    assert b"betas" in L.zopt_last_error()
    nan_lr = Z._Hparams(float("nan"), 0.9, 0.95, 1e-8, 0.1, 1, 0)
    assert L.zopt_adamw_step(lay.handle, tab, p, p, p, p, 1, None, ctypes.byref(nan_lr), None, p, None) == 1
    assert L.zopt_adamw_step(lay.handle, tab, p, p, p, p, 5, None, ctypes.byref(hp), None, p, None) == 2
    assert L.zopt_adamw_step(lay.handle, None, p, p, p, p, 1, None, ctypes.byref(hp), None, p, None) == 1
    assert L.zopt_adamw_step(lay.handle, tab, ctypes.c_void_p(8), p, p, p, 1, None, ctypes.byref(hp), None, p,
                             None) == 1


def test_ns_workspace_many_is_the_sum_of_rounded_single_workspaces():
    shapes = [(768, 2304, 12), (768, 768, 12), (3072, 768, 12), (130, 70, 1), (4096, 4096, 3)]
    want = sum(-(-Z.ns_workspace(r, c, b) // 1024) * 1024 for r, c, b in shapes)
    assert Z.ns_workspace_many(shapes) == want
    assert Z.ns_workspace_many([(0, 5, 1)]) == 0
    assert Z.ns_workspace_many([(5, 5, 65536)]) == 0
    assert Z.lib().zopt_ns_workspace_many(None, 0) == 0


def test_ns_orthogonalize_many_validates_before_launch():
    """Each call fails validation before any CUDA work (the pointers are fake)."""
    L = Z.lib()
    coef = (ctypes.c_float * 3)(*Z.DEFAULT_ABC)
    ws = ctypes.c_void_p(1 << 20)
    job = Z._NsJob(ctypes.c_void_p(1 << 16), ctypes.c_void_p(1 << 18), 64, 128, 128, 128, 0, 0, 1, Z.BF16)
    arr = (Z._NsJob * 1)(job)
    big = 1 << 40
    assert L.zopt_ns_orthogonalize_many(arr, 0, 5, coef, 1e-7, ws, big, None) == 1
    assert L.zopt_ns_orthogonalize_many(None, 1, 5, coef, 1e-7, ws, big, None) == 1
    assert L.zopt_ns_orthogonalize_many(arr, 1, 0, coef, 1e-7, ws, big, None) == 1
    assert L.zopt_ns_orthogonalize_many(arr, 1, 5, coef, 1e-7, ctypes.c_void_p((1 << 20) + 8), big, None) == 1
    assert b"aligned" in L.zopt_last_error()
    assert L.zopt_ns_orthogonalize_many(arr, 1, 5, coef, 1e-7, ws, 1024, None) == 1
    assert b"workspace" in L.zopt_last_error()
    bad = (Z._NsJob * 2)(job, Z._NsJob(ctypes.c_void_p(1 << 16), ctypes.c_void_p(1 << 18), 64, 128, 100, 128, 0, 0,
                                       1, Z.BF16))
    assert L.zopt_ns_orthogonalize_many(bad, 2, 5, coef, 1e-7, ws, big, None) == 1
    assert b"leading dimension" in L.zopt_last_error()
    f16 = (Z._NsJob * 1)(Z._NsJob(ctypes.c_void_p(1 << 16), ctypes.c_void_p(1 << 18), 64, 128, 128, 128, 0, 0, 1, 9))
    assert L.zopt_ns_orthogonalize_many(f16, 1, 5, coef, 1e-7, ws, big, None) == 2
    nan = (ctypes.c_float * 3)(float("nan"), 1.0, 1.0)
    assert L.zopt_ns_orthogonalize_many(arr, 1, 5, nan, 1e-7, ws, big, None) == 1


def test_muon_step_many_validates_before_launch():
    L = Z.lib()
    shapes = [(768, 2304, 12), (768, 768, 12)]
    assert Z.muon_workspace_many(shapes) > Z.muon_workspace_many(shapes[:1]) > 0
    assert Z.muon_workspace_many([(0, 4, 1)]) == 0
    hp = Z._muon_hparams(1e-3, 0.95, 0.1, True, True, 5, Z.DEFAULT_ABC, 1e-7, 1000.0)
    p = ctypes.c_void_p(1 << 20)
    job = Z._MuonJob(p, p, p, None, ctypes.c_void_p(1 << 16), 64, 128, 1, Z.BF16)
    arr = (Z._MuonJob * 1)(job)
    big = 1 << 40
    assert L.zopt_muon_step_many(arr, 0, ctypes.byref(hp), p, big, None) == 1
    assert L.zopt_muon_step_many(arr, 1, None, p, big, None) == 1
    assert L.zopt_muon_step_many(arr, 1, ctypes.byref(hp), p, 64, None) == 1
    assert b"workspace" in L.zopt_last_error()
    mis = (Z._MuonJob * 1)(Z._MuonJob(ctypes.c_void_p((1 << 20) + 4), p, p, None, ctypes.c_void_p(1 << 16), 64, 128,
                                      1, Z.BF16))
    assert L.zopt_muon_step_many(mis, 1, ctypes.byref(hp), p, big, None) == 1
    assert b"misaligned" in L.zopt_last_error()
    bad = Z._muon_hparams(1e-3, 1.5, 0.1, True, True, 5, Z.DEFAULT_ABC, 1e-7, 1000.0)
    assert L.zopt_muon_step_many(arr, 1, ctypes.byref(bad), p, big, None) == 1


def test_size_limits_validate_before_launch():
    """Shapes beyond ZOPT_NS_MAX_DIM (2^30), ZOPT_NS_MAX_ELEMS (2^36 elements), ZOPT_NS_MAX_LD
    (2^32) or ZOPT_NS_MAX_SPAN (2^56 elements per batch), and a Muon batch above 2^46 elements,
    are refused before any launch: the kernels keep tile coordinates in 32 bits."""
    L = Z.lib()
    assert Z.ns_workspace(1, 1 << 31) == 0
    assert Z.ns_workspace((1 << 30) + 1, 8) == 0
    assert Z.ns_workspace(1 << 30, 64) > 0          # 2^36 elements: at the limit
    assert Z.ns_workspace(1 << 30, 65) == 0         # one column more
    assert Z.ns_workspace_many([(1, 1 << 31, 1)]) == 0
    assert L.zopt_muon_workspace(1, 1 << 31, 1) == 0
    coef = (ctypes.c_float * 3)(*Z.DEFAULT_ABC)
    ws, big = ctypes.c_void_p(1 << 20), 1 << 40
    G, X = ctypes.c_void_p(1 << 16), ctypes.c_void_p(1 << 18)
    wide = (Z._NsJob * 1)(Z._NsJob(G, X, 1, 1 << 31, 1 << 31, 1 << 31, 0, 0, 1, Z.BF16))
    assert L.zopt_ns_orthogonalize_many(wide, 1, 5, coef, 1e-7, ws, big, None) == 1
    assert b"2^30" in L.zopt_last_error()
    assert L.zopt_ns_orthogonalize(G, X, Z.BF16, 1, 1 << 31, 1 << 31, 1 << 31, 0, 0, 1, Z.BF16, 5, coef, 1e-7, ws,
                                   big, None) == 1
    assert b"2^30" in L.zopt_last_error()
    ld = (Z._NsJob * 1)(Z._NsJob(G, X, 64, 128, 1 << 33, 128, 0, 0, 1, Z.BF16))
    assert L.zopt_ns_orthogonalize_many(ld, 1, 5, coef, 1e-7, ws, big, None) == 1
    assert b"leading dimension above" in L.zopt_last_error()
    span = (Z._NsJob * 1)(Z._NsJob(G, X, 64, 128, 128, 128, 1 << 56, 64 * 128, 3, Z.BF16))
    assert L.zopt_ns_orthogonalize_many(span, 1, 5, coef, 1e-7, ws, big, None) == 1
    assert b"spans" in L.zopt_last_error()
    hp = Z._muon_hparams(1e-3, 0.95, 0.1, True, True, 5, Z.DEFAULT_ABC, 1e-7, 1000.0)
    p = ctypes.c_void_p(1 << 20)
    huge = (Z._MuonJob * 1)(Z._MuonJob(p, p, p, None, ctypes.c_void_p(1 << 16), 1 << 20, 1 << 20, 1, Z.BF16))
    assert L.zopt_muon_step_many(huge, 1, ctypes.byref(hp), p, big, None) == 1
    assert b"2^36" in L.zopt_last_error()
    assert L.zopt_muon_step(p, p, p, Z.BF16, None, 1 << 15, 1 << 15, 1 << 17, ctypes.byref(hp),
                            ctypes.c_void_p(1 << 16), p, big, None) == 1
    assert b"2^46" in L.zopt_last_error()


def test_state_bytes_is_the_sharded_memory_plan():
    """zopt_layout_state_bytes against deg/zero.py's memory plan (sharded_static_bytes: fp32
    master + AdamW moments + fp32 gradient per shard, 16 B per parameter over W ranks): each rank
    holds 16 B per shard slot (14 with a bf16 gradient); over the ranks that is 16 B per padded
    bucket slot, between 16 N and 16 (N + buckets (W - 1))."""
    c4 = workloads.get("c4")
    numel = [p.numel for p in c4.adamw]
    lay = Z.ShardLayout(numel, None, c4.bucket, 8, 0)
    assert lay.state_bytes() == 16 * 250_000_000 and lay.state_bytes(Z.BF16) == 14 * 250_000_000
    for numel, bucket, world in [([100, 3, 77], 64, 3), ([5000, 1, 1234], 1000, 8), (numel, c4.bucket, 8)]:
        total = sum(Z.ShardLayout(numel, None, bucket, world, r).state_bytes() for r in range(world))
        padded = sum(L for _, _, L in OL.buckets(numel, bucket, world))
        assert total == 16 * padded
        N, nb = sum(numel), len(OL.buckets(numel, bucket, world))
        assert 16 * N <= total <= 16 * (N + nb * (world - 1))
    assert Z.lib().zopt_layout_state_bytes(None, 0) == -1
    assert Z.lib().zopt_layout_state_bytes(lay.handle, 7) == -1


def test_accumulate2_validates_before_launch():
    L = Z.lib()
    acc, g = ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 21)
    assert L.zopt_grad_accumulate2(acc, g, None, Z.BF16, 64, 1, 1.0, None, 0, None, None) == 1
    assert L.zopt_grad_accumulate2(acc, g, ctypes.c_void_p((1 << 22) + 8), Z.BF16, 64, 1, 1.0, None, 0, None,
                                   None) == 1
    assert b"aligned" in L.zopt_last_error()
    assert L.zopt_grad_accumulate2(acc, g, g, Z.BF16, 0, 1, 1.0, None, 0, None, None) == 1
    assert L.zopt_grad_accumulate2(acc, g, g, 9, 64, 1, 1.0, None, 0, None, None) == 2


def test_adamw_clip_step_validates_before_launch():
    """zopt_adamw_clip_step takes zopt_adamw_step's checks (shared code) and its own: d_clip and
    d_ws required and aligned, a workspace of zopt_adamw_clip_workspace(S) bytes, max_norm not
    negative or NaN. Every call below fails before any CUDA call (the pointers are fake)."""
    L = Z.lib()
    lay = Z.ShardLayout([100, 3], [1, 0], 64, 1, 0)  # S = 103 (one partial): 256 + 8 bytes
    S = lay.shard_len
    assert L.zopt_adamw_clip_workspace(S) == 256 + 8
    assert L.zopt_adamw_clip_workspace(0) == 0
    assert L.zopt_adamw_clip_workspace(2048 * 5000) == 256 + 8 * 4096  # at most 4096 blocks
    hp = Z._Hparams(1e-3, 0.9, 0.95, 1e-8, 0.1, 1, 0)
    bad = Z._Hparams(1e-3, 1.0, 0.95, 1e-8, 0.1, 1, 0)
    p, tab, clip, ws = ctypes.c_void_p(1 << 20), ctypes.c_void_p(4096), ctypes.c_void_p(512), ctypes.c_void_p(1 << 12)
    need = L.zopt_adamw_clip_workspace(S)
    call = lambda h=hp, mn=1.0, w=ws, wb=need, c=clip: L.zopt_adamw_clip_step(  # noqa: E731
        lay.handle, tab, p, p, p, p, 1, None, ctypes.byref(h), mn, w, wb, c, p, None)
    assert call(h=bad) == 1 and b"betas" in L.zopt_last_error()
    assert call(c=None) == 1 and b"NULL" in L.zopt_last_error()
    assert call(w=None) == 1 and b"NULL" in L.zopt_last_error()
    assert call(w=ctypes.c_void_p((1 << 12) + 8)) == 1 and b"aligned" in L.zopt_last_error()
    assert call(mn=-1.0) == 1 and b"max_norm" in L.zopt_last_error()
    assert call(mn=float("nan")) == 1 and b"max_norm" in L.zopt_last_error()
    assert call(wb=need - 1) == 1 and b"workspace" in L.zopt_last_error()
    assert L.zopt_adamw_clip_step(lay.handle, tab, p, p, p, p, 5, None, ctypes.byref(hp), 1.0, ws, need, clip, p,
                                  None) == 2  # another gradient dtype: EUNSUPPORTED
