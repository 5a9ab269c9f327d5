"""Python binding of libzopt — the rank-local optimizer step of a ZeRO-sharded trainer on
GB300 (sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA kernels. The
calls keep the C names: ``zopt_shard_layout`` (as :class:`ShardLayout`),
``zopt_grad_norm_clip``, ``zopt_adamw_step``, ``zopt_ns_orthogonalize``. PyTorch provides
device memory and streams. The library must be built (``build_lib.build()``); if it is
missing every call raises — there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import struct

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libzopt.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "zopt.h")

F32, BF16 = 0, 1
STATUS = {0: "ZOPT_OK", 1: "ZOPT_EINVAL", 2: "ZOPT_EUNSUPPORTED", 3: "ZOPT_ECUDA", 4: "ZOPT_ETIMEOUT"}

CLIP_STATS_BYTES = 24
ADAM_STATE_BYTES = 16

_lib = None


class ZoptError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class _Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("skip_on_inf", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class _MuonHparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("momentum", ctypes.c_double), ("weight_decay", ctypes.c_double),
                ("nesterov", ctypes.c_int32), ("adjust", ctypes.c_int32), ("ns_steps", ctypes.c_int32),
                ("abc", ctypes.c_float * 3), ("eps", ctypes.c_float), ("guard", ctypes.c_float)]


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libzopt.so is not built ({LIB_PATH}); run "
                           "`python -m zero_sharded_optimizer_flat_gb300.build_lib`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, u8p, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "zopt_last_error": (ctypes.c_char_p, []),
        "zopt_version": (ctypes.c_char_p, []),
        "zopt_shard_layout": (ctypes.c_int, [vp, u8p, i32, i64, i32, i32, ctypes.POINTER(vp)]),
        "zopt_layout_free": (None, [vp]),
        "zopt_layout_numel": (i64, [vp]),
        "zopt_layout_shard_len": (i64, [vp]),
        "zopt_layout_state_bytes": (i64, [vp, ctypes.c_int]),
        "zopt_layout_world": (i32, [vp]),
        "zopt_layout_rank": (i32, [vp]),
        "zopt_layout_num_buckets": (i32, [vp]),
        "zopt_layout_bucket": (ctypes.c_int, [vp, i32, vp, vp, vp, vp]),
        "zopt_layout_num_segments": (i64, [vp]),
        "zopt_layout_segments": (ctypes.c_int, [vp, vp, vp, vp, vp]),
        "zopt_layout_num_nodecay_runs": (i64, [vp]),
        "zopt_layout_nodecay_runs": (ctypes.c_int, [vp, vp]),
        "zopt_grad_norm_workspace": (sz, [i64]),
        "zopt_grad_norm_clip": (ctypes.c_int, [vp, ctypes.c_int, i64, ctypes.c_float, vp, sz, vp, vp]),
        "zopt_clip_finalize": (ctypes.c_int, [vp, ctypes.c_float, vp]),
        "zopt_grad_norm_clip_noalloc": (ctypes.c_int, [vp, ctypes.c_int, i64, ctypes.c_float, vp, vp]),
        "zopt_adamw_step": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, ctypes.POINTER(_Hparams),
                                           vp, vp, vp]),
        "zopt_adamw_clip_workspace": (sz, [i64]),
        "zopt_adamw_clip_step": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, ctypes.POINTER(_Hparams),
                                                ctypes.c_float, vp, sz, vp, vp, vp]),
        "zopt_adamw_rescale_step": (ctypes.c_int, [vp, vp, vp, vp, vp, ctypes.c_int, vp, ctypes.POINTER(_Hparams),
                                                   ctypes.c_float, ctypes.c_float, vp, vp, vp]),
        "zopt_grad_accumulate": (ctypes.c_int, [vp, vp, ctypes.c_int, i64, i32, ctypes.c_float, vp, sz, vp, vp]),
        "zopt_grad_accumulate2": (ctypes.c_int, [vp, vp, vp, ctypes.c_int, i64, i32, ctypes.c_float, vp, sz, vp,
                                                 vp]),
        "zopt_ns_workspace": (sz, [i64, i64, i32, ctypes.c_int]),
        "zopt_muon_workspace": (sz, [i64, i64, i32]),
        "zopt_take_device_error": (i32, []),
        "zopt_selftest_wait_timeout": (ctypes.c_int, [i64, vp]),
        "zopt_selftest_count_timeout": (ctypes.c_int, [i64, vp]),
        "zopt_selftest_div_by_const": (ctypes.c_int, [ctypes.c_float, vp, vp]),
        "zopt_muon_step": (ctypes.c_int, [vp, vp, vp, ctypes.c_int, vp, i64, i64, i32, ctypes.POINTER(_MuonHparams),
                                          vp, vp, sz, vp]),
        "zopt_ns_orthogonalize": (ctypes.c_int, [vp, vp, ctypes.c_int, i64, i64, i64, i64, i64, i64, i32,
                                                 ctypes.c_int, i32, ctypes.POINTER(ctypes.c_float), ctypes.c_float,
                                                 vp, sz, vp]),
        "zopt_ns_workspace_many": (sz, [ctypes.POINTER(_NsJob), i32]),
        "zopt_muon_workspace_many": (sz, [ctypes.POINTER(_MuonJob), i32]),
        "zopt_muon_step_many": (ctypes.c_int, [ctypes.POINTER(_MuonJob), i32, ctypes.POINTER(_MuonHparams), vp, sz,
                                               vp]),
        "zopt_ns_orthogonalize_many": (ctypes.c_int, [ctypes.POINTER(_NsJob), i32, i32,
                                                      ctypes.POINTER(ctypes.c_float), ctypes.c_float, vp, sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def declared_functions() -> list:
    """Every function the C header declares (used by the ABI export test)."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zopt_[a-z0-9_]+)\s*\(", text)))


def _check(status: int) -> None:
    if status != 0:
        raise ZoptError(status, lib().zopt_last_error().decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _count(t, n) -> int:
    """The element count a call covers: all of ``t``, or the first n (never more than it holds)."""
    if n is None:
        return t.numel()
    n = int(n)
    if n > t.numel():
        raise ValueError(f"n = {n} exceeds the tensor's {t.numel()} elements")
    return n


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    return -1


# --------------------------------------------------------------------------- layout

class ShardLayout:
    """``zopt_shard_layout``: rank ``rank``'s view of the flat bucketed layout."""

    def __init__(self, numel, decay=None, bucket: int = 1 << 25, world: int = 1, rank: int = 0):
        L = lib()
        n = np.ascontiguousarray(np.asarray(numel, dtype=np.int64))
        d = None if decay is None else np.ascontiguousarray(np.asarray(decay, dtype=np.uint8))
        if d is not None and d.shape != n.shape:
            raise ValueError("decay must have one flag per parameter")
        out = ctypes.c_void_p()
        _check(L.zopt_shard_layout(n.ctypes.data if n.size else None, None if d is None else d.ctypes.data,
                                   int(n.size), int(bucket), int(world), int(rank), ctypes.byref(out)))
        self._h = out
        self._keep = (n, d)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.zopt_layout_free(h)
            self._h = None

    @property
    def handle(self):
        return self._h

    @property
    def numel(self) -> int:
        return lib().zopt_layout_numel(self._h)

    @property
    def shard_len(self) -> int:
        return lib().zopt_layout_shard_len(self._h)

    def state_bytes(self, grad_dtype=F32) -> int:
        """``zopt_layout_state_bytes``: device bytes of this rank's master, moments and shard gradient."""
        return int(lib().zopt_layout_state_bytes(self._h, int(grad_dtype)))

    @property
    def world(self) -> int:
        return lib().zopt_layout_world(self._h)

    @property
    def rank(self) -> int:
        return lib().zopt_layout_rank(self._h)

    def buckets(self) -> list:
        L, out = lib(), []
        for b in range(L.zopt_layout_num_buckets(self._h)):
            v = [ctypes.c_int64() for _ in range(4)]
            _check(L.zopt_layout_bucket(self._h, b, *[ctypes.byref(x) for x in v]))
            out.append(tuple(x.value for x in v))
        return out

    def segments(self) -> np.ndarray:
        """(k, 4) int64: param index, offset in param, shard offset, length."""
        L = lib()
        k = L.zopt_layout_num_segments(self._h)
        p = np.zeros(k, np.int32)
        a = np.zeros((3, k), np.int64)
        _check(L.zopt_layout_segments(self._h, p.ctypes.data, a[0].ctypes.data, a[1].ctypes.data, a[2].ctypes.data))
        return np.stack([p.astype(np.int64), a[0], a[1], a[2]], axis=1)

    def nodecay_runs(self) -> np.ndarray:
        """(k, 2) int64 half-open shard ranges without weight decay."""
        L = lib()
        k = L.zopt_layout_num_nodecay_runs(self._h)
        r = np.zeros(2 * k, np.int64)
        _check(L.zopt_layout_nodecay_runs(self._h, r.ctypes.data if k else None))
        return r.reshape(k, 2)

    def device_table(self, device="cuda"):
        """The no-decay run table copied to the device (pass it to :func:`adamw_step`)."""
        import torch
        r = self.nodecay_runs().reshape(-1)
        return torch.from_numpy(r if r.size else np.zeros(2, np.int64)).to(device)


# --------------------------------------------------------------------------- device structs

def new_clip_stats(device="cuda"):
    import torch
    return torch.zeros(CLIP_STATS_BYTES, dtype=torch.uint8, device=device)


def new_adam_state(device="cuda"):
    import torch
    return torch.zeros(ADAM_STATE_BYTES, dtype=torch.uint8, device=device)


def read_clip_stats(t) -> dict:
    """Decode a zopt_clip_stats tensor (copies it to the host: logging/tests only)."""
    b = bytes(t.detach().cpu().numpy().tobytes())
    sumsq, norm, coef, clipped, found = struct.unpack("<dffBB6x", b)
    return {"sumsq": sumsq, "norm": np.float32(norm), "clip_coef": np.float32(coef), "clipped": bool(clipped),
            "found_inf": bool(found)}


def read_adam_state(t) -> dict:
    b = bytes(t.detach().cpu().numpy().tobytes())
    step, arrive, _ = struct.unpack("<qIi", b)
    return {"step": step, "arrive": arrive}


# --------------------------------------------------------------------------- calls

def grad_norm_workspace(n: int) -> int:
    return int(lib().zopt_grad_norm_workspace(int(n)))


def new_norm_workspace(n: int, device="cuda"):
    """A zero-filled workspace for :func:`grad_norm_clip` over n elements."""
    import torch
    return torch.zeros(max(grad_norm_workspace(n), 16), dtype=torch.uint8, device=device)


def grad_norm_clip(grad, max_norm: float, ws, stats, n: int | None = None, stream=None) -> None:
    """``zopt_grad_norm_clip`` over the first n elements of ``grad`` (default: all)."""
    n = _count(grad, n)
    _check(lib().zopt_grad_norm_clip(_ptr(grad), _dtype_code(grad), n, float(max_norm), _ptr(ws), ws.numel(),
                                     _ptr(stats), _stream(stream)))


def grad_norm_clip_noalloc(grad, max_norm: float, stats, n: int | None = None, stream=None) -> None:
    """``zopt_grad_norm_clip_noalloc``: the same reduction with the library's static scratch
    instead of a workspace, for callers that cannot allocate device memory."""
    n = _count(grad, n)
    _check(lib().zopt_grad_norm_clip_noalloc(_ptr(grad), _dtype_code(grad), n, float(max_norm), _ptr(stats),
                                             _stream(stream)))


def adamw_rescale_step(layout: ShardLayout, master, exp_avg, exp_avg_sq, grad, out_bf16, *, lr: float,
                       old_scale: float, new_scale: float = 1.0, beta1: float = 0.9, beta2: float = 0.95,
                       eps: float = 1e-8, weight_decay: float = 0.1, clip_stats=None, adam_state=None,
                       stream=None) -> None:
    """``zopt_adamw_rescale_step``: turn the last step on g*old_scale into the step on
    g*new_scale (or on the clip coefficient in ``clip_stats``)."""
    hp = _Hparams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), 1, 0)
    _check(lib().zopt_adamw_rescale_step(layout.handle, _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq), _ptr(grad),
                                         _dtype_code(grad), _ptr(out_bf16), ctypes.byref(hp), float(old_scale),
                                         float(new_scale), _ptr(clip_stats), _ptr(adam_state), _stream(stream)))


ACC_FIRST, ACC_LAST = 1, 2


def grad_accumulate(acc, micro_grad, *, first: bool, last: bool, max_norm: float = 1.0, ws=None, stats=None,
                    n: int | None = None, stream=None) -> None:
    """``zopt_grad_accumulate``: acc (fp32) = / += micro_grad; the last micro-step also
    writes the clip stats of the finished sum."""
    n = _count(acc, n)
    _count(micro_grad, n)
    flags = (ACC_FIRST if first else 0) | (ACC_LAST if last else 0)
    _check(lib().zopt_grad_accumulate(_ptr(acc), _ptr(micro_grad), _dtype_code(micro_grad), n, flags,
                                      float(max_norm), _ptr(ws), 0 if ws is None else ws.numel(), _ptr(stats),
                                      _stream(stream)))


def grad_accumulate2(acc, micro_grad_a, micro_grad_b, *, first: bool, last: bool, max_norm: float = 1.0, ws=None,
                     stats=None, n: int | None = None, stream=None) -> None:
    """``zopt_grad_accumulate2``: two micro-steps in one pass, bit for bit two grad_accumulate calls
    (``first`` applies to the first part, ``last`` to the second)."""
    if micro_grad_a.dtype != micro_grad_b.dtype:
        raise ValueError("both micro-step gradients must have one dtype")
    n = _count(acc, n)
    _count(micro_grad_a, n)
    _count(micro_grad_b, n)
    flags = (ACC_FIRST if first else 0) | (ACC_LAST if last else 0)
    _check(lib().zopt_grad_accumulate2(_ptr(acc), _ptr(micro_grad_a), _ptr(micro_grad_b), _dtype_code(micro_grad_a),
                                       n, flags, float(max_norm), _ptr(ws), 0 if ws is None else ws.numel(),
                                       _ptr(stats), _stream(stream)))


def clip_finalize(stats, max_norm: float, stream=None) -> None:
    _check(lib().zopt_clip_finalize(_ptr(stats), float(max_norm), _stream(stream)))


def adamw_step(layout: ShardLayout, table, master, exp_avg, exp_avg_sq, grad, out_bf16, *, lr: float,
               beta1: float = 0.9, beta2: float = 0.95, eps: float = 1e-8, weight_decay: float = 0.1,
               skip_on_inf: bool = True, clip_stats=None, adam_state=None, stream=None) -> None:
    """``zopt_adamw_step``: one AdamW step of the rank's shard, in place."""
    hp = _Hparams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(bool(skip_on_inf)), 0)
    _check(lib().zopt_adamw_step(layout.handle, _ptr(table), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                 _ptr(grad), _dtype_code(grad), _ptr(out_bf16), ctypes.byref(hp),
                                 _ptr(clip_stats), _ptr(adam_state), _stream(stream)))



def adamw_clip_workspace(shard_len: int) -> int:
    return int(lib().zopt_adamw_clip_workspace(int(shard_len)))


def new_adamw_clip_workspace(shard_len: int, device="cuda"):
    """A zero-filled workspace for :func:`adamw_clip_step` over a shard of this length (each call
    leaves its counters at zero again)."""
    import torch
    return torch.zeros(max(adamw_clip_workspace(shard_len), 16), dtype=torch.uint8, device=device)


def adamw_clip_step(layout: ShardLayout, table, master, exp_avg, exp_avg_sq, grad, out_bf16, *, lr: float,
                    max_norm: float, ws, clip_stats, adam_state, beta1: float = 0.9, beta2: float = 0.95,
                    eps: float = 1e-8, weight_decay: float = 0.1, skip_on_inf: bool = True, stream=None) -> None:
    """``zopt_adamw_clip_step``: the gradient's norm / clip / found_inf and the AdamW step of the
    rank's shard in one launch (the stats land in ``clip_stats`` as zopt_grad_norm_clip writes them)."""
    hp = _Hparams(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(bool(skip_on_inf)), 0)
    _check(lib().zopt_adamw_clip_step(layout.handle, _ptr(table), _ptr(master), _ptr(exp_avg), _ptr(exp_avg_sq),
                                      _ptr(grad), _dtype_code(grad), _ptr(out_bf16), ctypes.byref(hp),
                                      float(max_norm), _ptr(ws), ws.numel(), _ptr(clip_stats), _ptr(adam_state),
                                      _stream(stream)))


# --------------------------------------------------------------------------- Newton-Schulz

DEFAULT_ABC = (3.4445, -4.7750, 2.0315)


def ns_workspace(rows: int, cols: int, group: int = 1, compute=BF16) -> int:
    return int(lib().zopt_ns_workspace(int(rows), int(cols), int(group), int(compute)))


def new_ns_workspace(rows: int, cols: int, group: int = 1, compute=BF16, device="cuda"):
    """A workspace for processing ``group`` matrices of this shape per launch."""
    import torch
    return torch.empty(max(ns_workspace(rows, cols, group, compute), 16), dtype=torch.uint8, device=device)


class _NsJob(ctypes.Structure):
    """``zopt_ns_job``: one shape's matrices for ``zopt_ns_orthogonalize_many``."""
    _fields_ = [("G", ctypes.c_void_p), ("X", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld_g", ctypes.c_int64), ("ld_x", ctypes.c_int64), ("batch_stride_g", ctypes.c_int64),
                ("batch_stride_x", ctypes.c_int64), ("batch", ctypes.c_int32), ("io_dtype", ctypes.c_int32)]


def _ns_job(G, X) -> _NsJob:
    if G.dim() == 2:
        batch, rows, cols = 1, G.shape[0], G.shape[1]
        ldg, ldx, sg, sx = G.stride(0), X.stride(0), 0, 0
    else:
        batch, rows, cols = G.shape
        ldg, ldx, sg, sx = G.stride(1), X.stride(1), G.stride(0), X.stride(0)
    if G.stride(-1) != 1 or X.stride(-1) != 1 or G.dtype != X.dtype or X.shape != G.shape:
        raise ValueError("G and X must have the same shape and dtype, with a contiguous last dimension")
    return _NsJob(_ptr(G), _ptr(X), rows, cols, ldg, ldx, sg, sx, batch, _dtype_code(G))


def _shape_job(rows: int, cols: int, batch: int) -> _NsJob:
    return _NsJob(None, None, int(rows), int(cols), int(cols), int(cols), 0, 0, int(batch), BF16)


def ns_workspace_many(shapes) -> int:
    """``zopt_ns_workspace_many`` for jobs of the given (rows, cols, batch)."""
    arr = (_NsJob * len(shapes))(*[_shape_job(*sh) for sh in shapes])
    return int(lib().zopt_ns_workspace_many(arr, len(shapes)))


def new_ns_workspace_many(shapes, device="cuda"):
    import torch
    return torch.empty(max(ns_workspace_many(shapes), 16), dtype=torch.uint8, device=device)


def ns_orthogonalize_many(pairs, ws, steps: int = 5, abc=DEFAULT_ABC, eps: float = 1e-7, stream=None) -> None:
    """``zopt_ns_orthogonalize_many`` over [(G, X), ...]: each a 2-D matrix or a batch [b, rows, cols]."""
    arr = (_NsJob * len(pairs))(*[_ns_job(G, X) for G, X in pairs])
    coef = (ctypes.c_float * 3)(*[float(c) for c in abc])
    _check(lib().zopt_ns_orthogonalize_many(arr, len(pairs), int(steps), coef, float(eps), _ptr(ws), ws.numel(),
                                            _stream(stream)))


def ns_orthogonalize(G, X, ws, steps: int = 5, abc=DEFAULT_ABC, eps: float = 1e-7, compute=BF16, stream=None) -> None:
    """``zopt_ns_orthogonalize`` of a 2-D matrix or a batch [b, rows, cols] (last dim contiguous)."""
    if G.dim() == 2:
        batch, rows, cols = 1, G.shape[0], G.shape[1]
        ldg, ldx, sg, sx = G.stride(0), X.stride(0), 0, 0
    else:
        batch, rows, cols = G.shape
        ldg, ldx, sg, sx = G.stride(1), X.stride(1), G.stride(0), X.stride(0)
    if G.stride(-1) != 1 or X.stride(-1) != 1 or G.dtype != X.dtype or X.shape != G.shape:
        raise ValueError("G and X must have the same shape and dtype, with a contiguous last dimension")
    coef = (ctypes.c_float * 3)(*[float(c) for c in abc])
    _check(lib().zopt_ns_orthogonalize(_ptr(G), _ptr(X), _dtype_code(G), rows, cols, ldg, ldx, sg, sx, batch,
                                       int(compute), int(steps), coef, float(eps), _ptr(ws), ws.numel(),
                                       _stream(stream)))


# --------------------------------------------------------------------------- Muon

MUON_STATS_BYTES = 16


def muon_workspace(rows: int, cols: int, group: int = 1) -> int:
    return int(lib().zopt_muon_workspace(int(rows), int(cols), int(group)))


def new_muon_workspace(rows: int, cols: int, group: int = 1, device="cuda"):
    import torch
    return torch.empty(max(muon_workspace(rows, cols, group), 16), dtype=torch.uint8, device=device)


def new_muon_stats(batch: int = 1, device="cuda"):
    import torch
    return torch.zeros(MUON_STATS_BYTES * batch, dtype=torch.uint8, device=device)


def read_muon_stats(t) -> list:
    """Decode zopt_muon_stats entries (copies them to the host: logging/tests only)."""
    b = bytes(t.detach().cpu().numpy().tobytes())
    out = []
    for k in range(len(b) // MUON_STATS_BYTES):
        fro, ratio, mx, rej = struct.unpack("<fffI", b[16 * k:16 * k + 16])
        out.append({"update_fro": fro, "ns_ratio": ratio, "max_abs": mx, "rejected": bool(rej)})
    return out


def _muon_hparams(lr, momentum_coef, weight_decay, nesterov, match_rms_adamw, ns_steps, abc, eps, guard):
    return _MuonHparams(float(lr), float(momentum_coef), float(weight_decay), int(bool(nesterov)),
                        0 if match_rms_adamw else 1, int(ns_steps), (ctypes.c_float * 3)(*[float(c) for c in abc]),
                        float(eps), float(guard))


class _MuonJob(ctypes.Structure):
    """``zopt_muon_job``: one shape's matrices for ``zopt_muon_step_many``."""
    _fields_ = [("master", ctypes.c_void_p), ("momentum", ctypes.c_void_p), ("grad", ctypes.c_void_p),
                ("out_bf16", ctypes.c_void_p), ("d_stats", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("batch", ctypes.c_int32), ("grad_dtype", ctypes.c_int32)]


def muon_workspace_many(shapes) -> int:
    """``zopt_muon_workspace_many`` for jobs of the given (rows, cols, batch)."""
    arr = (_MuonJob * len(shapes))(*[_MuonJob(None, None, None, None, None, int(r), int(c), int(b), F32)
                                     for r, c, b in shapes])
    return int(lib().zopt_muon_workspace_many(arr, len(shapes)))


def new_muon_workspace_many(shapes, device="cuda"):
    import torch
    return torch.empty(max(muon_workspace_many(shapes), 16), dtype=torch.uint8, device=device)


def muon_step_many(jobs, ws, *, lr: float, momentum_coef: float = 0.95, weight_decay: float = 0.1,
                   nesterov: bool = True, match_rms_adamw: bool = True, ns_steps: int = 5, abc=DEFAULT_ABC,
                   eps: float = 1e-7, guard: float = 1000.0, stream=None) -> None:
    """``zopt_muon_step_many`` over [(master, momentum, grad, out_bf16, stats), ...], each a matrix
    [rows, cols] or a batch [b, rows, cols] (contiguous); out_bf16 may be None."""
    arr = []
    for master, momentum, grad, out_bf16, stats in jobs:
        shape = tuple(master.shape)
        batch, rows, cols = (1, *shape) if len(shape) == 2 else shape
        arr.append(_MuonJob(_ptr(master), _ptr(momentum), _ptr(grad), _ptr(out_bf16), _ptr(stats), rows, cols, batch,
                            _dtype_code(grad)))
    c_arr = (_MuonJob * len(arr))(*arr)
    hp = _muon_hparams(lr, momentum_coef, weight_decay, nesterov, match_rms_adamw, ns_steps, abc, eps, guard)
    _check(lib().zopt_muon_step_many(c_arr, len(arr), ctypes.byref(hp), _ptr(ws), ws.numel(), _stream(stream)))


def muon_step(master, momentum, grad, out_bf16, ws, stats, *, lr: float, momentum_coef: float = 0.95,
              weight_decay: float = 0.1, nesterov: bool = True, match_rms_adamw: bool = True, ns_steps: int = 5,
              abc=DEFAULT_ABC, eps: float = 1e-7, guard: float = 1000.0, stream=None) -> None:
    """``zopt_muon_step`` on a matrix [rows, cols] or a batch [b, rows, cols] (contiguous)."""
    shape = tuple(master.shape)
    batch, rows, cols = (1, *shape) if len(shape) == 2 else shape
    hp = _muon_hparams(lr, momentum_coef, weight_decay, nesterov, match_rms_adamw, ns_steps, abc, eps, guard)
    _check(lib().zopt_muon_step(_ptr(master), _ptr(momentum), _ptr(grad), _dtype_code(grad), _ptr(out_bf16), rows,
                                cols, batch, ctypes.byref(hp), _ptr(stats), _ptr(ws), ws.numel(), _stream(stream)))


def take_device_error() -> int:
    """The device error word (1 = a bounded wait ran out), cleared by the read."""
    return int(lib().zopt_take_device_error())


def selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Run the bounded-wait path on a barrier nothing completes (limit_ns <= 2 s)."""
    _check(lib().zopt_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def selftest_div_by_const(c: float, counter, stream=None) -> None:
    """Add to counter (a 1-element int64 CUDA tensor) the number of v >= 0 bit patterns for which
    the rescale kernel's sqrt(v) / c differs from the IEEE division."""
    _check(lib().zopt_selftest_div_by_const(ctypes.c_float(c), ctypes.c_void_p(counter.data_ptr()), _stream(stream)))


def selftest_count_timeout(limit_ns: int, stream=None) -> None:
    """Run the fused kernel's bounded counter wait on a counter nothing advances (limit_ns <= 2 s)."""
    _check(lib().zopt_selftest_count_timeout(int(limit_ns), _stream(stream)))
