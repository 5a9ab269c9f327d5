"""Per-tensor AdamW — oracle (test infrastructure only).

Sources:
* dmuon PR #16, "foreach AdamW" commit: the op order is decoupled weight decay, then the
  moments, then the bias-corrected addcdiv; bias corrections are per-step scalars.
* DeepSpeed PR #9021, grad_scale commit: each gradient element is multiplied by the scale
  as it is loaded, after the bf16 -> fp32 promotion; fp32 x fp32 rounds as a separate
  multiply would.  The clip coefficient enters the step this way.
* bluscript_zero_ckpt.cpp, ZeroConfig: beta = (0.9, 0.95), eps = 1e-8, weight decay with
  1-D parameters excluded; the fp32-master note (a bf16 master would round the decay away).
* deg/zero.py, ZeroMaster docstring: element-wise AdamW over the flat shard is the same
  arithmetic as over the separate tensors.

Readings where the pages are silent (all listed in the design notes):
* eps is added outside the square root: denom = sqrt(v)/sqrt(1-beta2^t) + eps.
* Hyper-parameters arrive as fp64 numbers; every derived scalar is formed in fp64 and
  rounded once to fp32: beta1, 1-beta1, beta2, 1-beta2, eps, 1-lr*wd,
  step_size = lr/(1-beta1^t), bc2s = sqrt(1-beta2^t).
* beta^t is an fp64 power by right-to-left binary exponentiation (square-and-multiply),
  a fixed sequence of IEEE multiplies; it is pinned against ``math.pow``.
* Moments: m = beta1*m + (1-beta1)*g; v = beta2*v + (1-beta2)*(g*g), each operation
  rounded to fp32 on its own (no fused multiply-add), in the order written.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

F32 = np.float32


@dataclass(frozen=True)
class Hyper:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


def beta_power(beta: float, t: int) -> float:
    """beta**t in fp64 by right-to-left square-and-multiply."""
    result, base, e = 1.0, float(beta), int(t)
    while e > 0:
        if e & 1:
            result = result * base
        base = base * base
        e >>= 1
    return result


@dataclass(frozen=True)
class Scalars32:
    beta1: np.float32
    one_minus_beta1: np.float32
    beta2: np.float32
    one_minus_beta2: np.float32
    eps: np.float32
    decay: np.float32        # 1 - lr*wd, for parameters that take weight decay
    step_size: np.float32    # lr / (1 - beta1^t)
    bc2_sqrt: np.float32     # sqrt(1 - beta2^t)


def scalars_f32(h: Hyper, t: int) -> Scalars32:
    """The step's scalars: formed in fp64, rounded once to fp32 (t = post-increment step)."""
    bc1 = 1.0 - beta_power(h.beta1, t)
    bc2 = 1.0 - beta_power(h.beta2, t)
    return Scalars32(F32(h.beta1), F32(1.0 - h.beta1), F32(h.beta2), F32(1.0 - h.beta2), F32(h.eps),
                     F32(1.0 - h.lr * h.weight_decay), F32(h.lr / bc1), F32(math.sqrt(bc2)))


def adamw_tensor_f32(p: np.ndarray, m: np.ndarray, v: np.ndarray, g_in: np.ndarray, coef: np.float32,
                     decays: bool, sc: Scalars32) -> None:
    """One AdamW step of one tensor, in place, every operation an fp32 rounding."""
    assert p.dtype == m.dtype == v.dtype == np.float32
    g = g_in.astype(np.float32) * F32(coef)            # grad scale on load
    if decays:
        p *= sc.decay                                   # decoupled weight decay
    m[...] = sc.beta1 * m + sc.one_minus_beta1 * g      # first moment
    v[...] = sc.beta2 * v + sc.one_minus_beta2 * (g * g)  # second moment
    denom = np.sqrt(v) / sc.bc2_sqrt + sc.eps           # bias-corrected denominator
    p -= sc.step_size * (m / denom)                     # bias-corrected addcdiv


def adamw_tensor_f64(p: np.ndarray, m: np.ndarray, v: np.ndarray, g_in: np.ndarray, coef: float,
                     decays: bool, h: Hyper, t: int) -> None:
    """The same step in fp64 with unrounded fp64 scalars (a precision reference)."""
    assert p.dtype == m.dtype == v.dtype == np.float64
    g = g_in.astype(np.float64) * float(coef)
    if decays:
        p *= 1.0 - h.lr * h.weight_decay
    m[...] = h.beta1 * m + (1.0 - h.beta1) * g
    v[...] = h.beta2 * v + (1.0 - h.beta2) * (g * g)
    bc1 = 1.0 - beta_power(h.beta1, t)
    bc2 = 1.0 - beta_power(h.beta2, t)
    denom = np.sqrt(v) / math.sqrt(bc2) + h.eps
    p -= (h.lr / bc1) * (m / denom)


def step_tensors(params: list, ms: list, vs: list, grads: list, decays: list, coef, h: Hyper, t: int,
                 mode: str = "f32") -> None:
    """One AdamW step over a list of separate tensors (the unsharded trainer's view)."""
    if mode == "f32":
        sc = scalars_f32(h, t)
        for p, m, v, g, d in zip(params, ms, vs, grads, decays):
            adamw_tensor_f32(p, m, v, g, F32(coef), bool(d), sc)
    elif mode == "f64":
        for p, m, v, g, d in zip(params, ms, vs, grads, decays):
            adamw_tensor_f64(p, m, v, g, coef, bool(d), h, t)
    else:
        raise ValueError(mode)


def step_flat_f32(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, decay_mask: np.ndarray,
                  coef, h: Hyper, t: int) -> None:
    """The same step over one flat vector with a per-element decay mask (the sharded view)."""
    sc = scalars_f32(h, t)
    g32 = g.astype(np.float32) * F32(coef)
    dec = decay_mask.astype(bool)
    p[dec] *= sc.decay
    m[...] = sc.beta1 * m + sc.one_minus_beta1 * g32
    v[...] = sc.beta2 * v + sc.one_minus_beta2 * (g32 * g32)
    denom = np.sqrt(v) / sc.bc2_sqrt + sc.eps
    p -= sc.step_size * (m / denom)


def rescale_step_f32(p: np.ndarray, m: np.ndarray, v: np.ndarray, g_in: np.ndarray, old_scale, new_scale,
                     h: Hyper, t: int) -> None:
    """Re-target the AdamW step t that was taken on g*old_scale to the step on g*new_scale, in
    place and in one pass (DeepSpeed PR #9021, adam_rescale_step commit):
        m += (1-beta1)*(new-old)*g;  v = max(0, v + (1-beta2)*(new^2-old^2)*g^2)  (NaN kept);
        p += step_size*(m_old/d_old - m_new/d_new)   (the decay does not depend on g: cancels)
    with d = sqrt(v)/sqrt(1-beta2^t) + eps. Readings: the page prints the weight change as
    step_size*(update_new - update_old) in a convention where the update is the signed
    increment; here it is written as what the commit states it achieves — the weights of the
    step on the new scale. km = fp32((1-beta1)*(new-old)) and kv = fp32((1-beta2)*(new^2-old^2))
    are formed in fp64; each array operation is an fp32 rounding in the order written."""
    sc = scalars_f32(h, t)
    old, new = float(old_scale), float(new_scale)
    km = F32((1.0 - h.beta1) * (new - old))
    kv = F32((1.0 - h.beta2) * (new * new - old * old))
    g = g_in.astype(np.float32)
    u_old = m / (np.sqrt(v) / sc.bc2_sqrt + sc.eps)
    m[...] = m + km * g
    vv = v + kv * (g * g)
    v[...] = np.where(vv < 0, F32(0.0), vv)
    u_new = m / (np.sqrt(v) / sc.bc2_sqrt + sc.eps)
    p += sc.step_size * (u_old - u_new)


def rescale_step_f64(p, m, v, g_in, old_scale, new_scale, h: Hyper, t: int) -> None:
    """The same re-targeting in fp64 with unrounded scalars (the precision reference)."""
    g = np.asarray(g_in, dtype=np.float64)
    bc2 = math.sqrt(1.0 - beta_power(h.beta2, t))
    step = h.lr / (1.0 - beta_power(h.beta1, t))
    u_old = m / (np.sqrt(v) / bc2 + h.eps)
    m[...] = m + (1.0 - h.beta1) * (new_scale - old_scale) * g
    v[...] = np.maximum(0.0, v + (1.0 - h.beta2) * (new_scale ** 2 - old_scale ** 2) * g * g)
    u_new = m / (np.sqrt(v) / bc2 + h.eps)
    p += step * (u_old - u_new)
