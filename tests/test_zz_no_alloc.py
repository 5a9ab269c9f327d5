"""zopt_grad_norm_clip_noalloc against zopt_grad_norm_clip and the oracle.

The no-alloc entry point serves callers that cannot allocate device memory (a C host or
plugin that only gets device pointers, a loop that forbids allocation after start-up, a
process whose device memory another runtime holds): its scratch is a static device array
inside the library instead of a caller workspace. This file is collected last on purpose.

Both entry points run the same kernel on the same grid on a GB300, so their stats must agree
bit for bit; against the oracle (deg/zero.py grad_sq_norm, bluscript_zero_ckpt.cpp clip block)
the sum of squares, norm and coefficient agree within 1e-6 relative and the flags exactly.
Two calls in a row on each size check that the array's leftover contents from one call (its
arrival counter and partials) never leak into the next; the second call also turns found_inf
on. Sizes: a tail-only gradient (fewer than 8 elements), one that spans a few blocks, and one
that fills the launch's whole wave of blocks.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import clip as OC

pytestmark = pytest.mark.gpu


def close(a, b, rel=1e-6):
    return float(a) == float(b) or abs(float(a) - float(b)) <= rel * abs(float(b))


@pytest.mark.parametrize("n", [5, 40_003, 8_388_617])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_entry_point_and_oracle(zopt, dtype, n):
    lib = zopt.lib()
    code = zopt.F32 if dtype == torch.float32 else zopt.BF16
    gen = torch.Generator(device="cuda").manual_seed(123 + n)
    grads = [(torch.randn(n, generator=gen, device="cuda") * 1e-3).to(dtype),
             (torch.randn(n, generator=gen, device="cuda") * 2.0).to(dtype)]
    grads[1][n - 2] = float("inf")  # the second call flips found_inf
    ws = zopt.new_norm_workspace(n)
    ref, new = zopt.new_clip_stats(), zopt.new_clip_stats()
    stream = torch.cuda.current_stream().cuda_stream
    for g in grads:  # two calls in a row
        zopt.grad_norm_clip(g, 1.0, ws, ref)
        st = lib.zopt_grad_norm_clip_noalloc(ctypes.c_void_p(g.data_ptr()), code, n, ctypes.c_float(1.0),
                                             ctypes.c_void_p(new.data_ptr()), ctypes.c_void_p(stream))
        assert st == 0, lib.zopt_last_error()
        torch.cuda.synchronize()
        # bit for bit the workspace entry point (same kernel, same grid)
        assert torch.equal(new, ref)
        a = zopt.read_clip_stats(new)
        o = OC.clip_stats(g.float().cpu().numpy(), 1.0)
        assert a["found_inf"] == o["found_inf"] and a["clipped"] == o["clipped"]
        if o["found_inf"]:
            assert a["clip_coef"] == 0.0
        else:
            assert close(a["sumsq"], o["sumsq"]) and close(a["norm"], o["norm"])
            assert close(a["clip_coef"], o["clip_coef"])


def test_noalloc_checks_its_count(zopt):
    g = torch.zeros(16, device="cuda")
    with pytest.raises(ValueError):
        zopt.grad_norm_clip_noalloc(g, 1.0, zopt.new_clip_stats(), n=17)
    with pytest.raises(zopt.ZoptError):
        zopt.grad_norm_clip_noalloc(g, 1.0, zopt.new_clip_stats(), n=0)
