"""zopt_grad_norm_clip_noalloc against zopt_grad_norm_clip.

The no-alloc entry point serves callers that cannot allocate device memory (a C host or
plugin that only gets device pointers, a loop that forbids allocation after start-up, a
process whose device memory another runtime holds): its scratch is a static device array
inside the library instead of a caller workspace. This file is collected last on purpose.
Two calls in a row check that the array's leftover contents from one call never leak into
the next.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def close(a, b, rel=1e-6):
    return a == b or abs(float(a) - float(b)) <= rel * abs(float(b))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_entry_point(zopt, dtype):
    lib = zopt.lib()
    code = zopt.F32 if dtype == torch.float32 else zopt.BF16
    gen = torch.Generator(device="cuda").manual_seed(123)
    n = 3_000_017
    grads = [(torch.randn(n, generator=gen, device="cuda") * 1e-3).to(dtype),
             (torch.randn(n, generator=gen, device="cuda") * 2.0).to(dtype)]
    grads[1][n - 5] = float("inf")  # the second call also flips found_inf
    ws = zopt.new_norm_workspace(n)
    ref, new = zopt.new_clip_stats(), zopt.new_clip_stats()
    stream = torch.cuda.current_stream().cuda_stream
    for g in grads:  # two calls in a row
        zopt.grad_norm_clip(g, 1.0, ws, ref)
        st = lib.zopt_grad_norm_clip_noalloc(ctypes.c_void_p(g.data_ptr()), code, n, ctypes.c_float(1.0),
                                             ctypes.c_void_p(new.data_ptr()), ctypes.c_void_p(stream))
        assert st == 0, lib.zopt_last_error()
        torch.cuda.synchronize()
        a, b = zopt.read_clip_stats(new), zopt.read_clip_stats(ref)
        assert a["found_inf"] == b["found_inf"] and a["clipped"] == b["clipped"]
        assert close(a["clip_coef"], b["clip_coef"]) and close(a["norm"], b["norm"])
        if not b["found_inf"]:
            assert close(a["sumsq"], b["sumsq"])
