"""GPU parity of zopt_ns_orthogonalize (bluscript_zero_ckpt.cpp, ShardedMuon note:
X <- aX + (bXX' + c(XX')^2)X on the whole matrix, 5 steps).

* White box, one step: the normalised X0, A = X0 X0', B' = cAA' + bA + aI (the bf16 path folds
  the step's aX term into the last product, X = B' X0) and the output are read back and each is
  checked against a float32 product of the kernel's own bf16 inputs (relative Frobenius error
  <= 4e-3: one bf16 rounding of the output plus fp32 accumulation order); A and B' must be
  exactly symmetric.
* End to end, 5 steps: relative Frobenius error against the fp64 oracle <= 2e-2 (bf16).
* Full-size stress matrices, in the benchmark's launch configuration: one matrix of each
  shape against the fp64 oracle <= 2e-2, every matrix against a float32 torch Newton-Schulz
  on the GPU (the checker) <= 2e-2, and the oracle on the top-left 256 x 1024 block taken as
  its own input.
"""
import numpy as np
import pytest
import torch

import workloads

from oracle.ns import DEFAULT_ABC, newton_schulz

pytestmark = pytest.mark.gpu

A_, B_, C_ = DEFAULT_ABC


def rup(x, a):
    return -(-x // a) * a


def plan(rows, cols, es=2, group=1):
    """Offsets of the library's workspace regions for matrix 0 of a group (white-box reading of
    its layout: a header of per-matrix reduction scratch and stats, then one region per matrix)."""
    m, n = min(rows, cols), max(rows, cols)
    ldx, lda = rup(n, 8), rup(m, 8)
    off_stats = rup(group * (256 + 8 * 512), 256)
    header = rup(off_stats + group * 32, 1024)
    xbytes, abytes = rup(m * ldx * es, 1024), rup(m * lda * es, 1024)
    return dict(m=m, n=n, ldx=ldx, lda=lda, x0=header, x1=header + xbytes, a=header + 2 * xbytes,
                b=header + 2 * xbytes + abytes, xbytes=xbytes, abytes=abytes, per=2 * xbytes + 2 * abytes)


def region(ws, off, rows, ld, cols):
    return ws[off:off + rows * ld * 2].view(torch.bfloat16).view(rows, ld)[:, :cols].float()


def rel(a, b):
    a, b = a.double(), b.double()
    return float(torch.linalg.norm(a - b) / torch.linalg.norm(b))


def gaussian(rows, cols, seed, dtype=torch.bfloat16):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(rows, cols, generator=g, device="cuda").to(dtype)


SHAPES_WB = [(256, 1024), (1024, 256), (300, 300), (200, 333), (130, 70), (1, 64), (64, 1), (17, 100), (768, 2304),
             (384, 640),
             # m >= 1024: the CTA-pair kernel (256 x 256 tiles), whole and ragged
             (1024, 1536), (1100, 1300), (2000, 1030), (1024, 1024)]


@pytest.mark.parametrize("rows,cols", SHAPES_WB)
def test_one_step_white_box(zopt, rows, cols):
    G = gaussian(rows, cols, rows * 7 + cols)
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(rows, cols)
    zopt.ns_orthogonalize(G, X, ws, steps=1)
    torch.cuda.synchronize()
    p = plan(rows, cols)
    m, n = p["m"], p["n"]
    Gd = G.double()
    ref0 = Gd / (torch.linalg.norm(Gd) + 1e-7)
    if rows > cols:
        ref0 = ref0.T
    if rows <= cols and cols % 8 == 0:
        # a bf16 input in X's orientation with 16-byte rows is read in place by the first step,
        # whose products apply the normalisation: X0 is never stored
        X0 = ref0.float()
    else:
        X0 = region(ws, p["x0"], m, p["ldx"], n)
        assert rel(X0, ref0) < 4e-3
    A = region(ws, p["a"], m, p["lda"], m)
    assert torch.equal(A, A.T)
    assert rel(A, X0 @ X0.T) < 4e-3
    # the bf16 path folds the step's a X term into the last product: B' = c A A' + b A + a I, X = B' X0
    B = region(ws, p["b"], m, p["lda"], m)
    assert torch.equal(B, B.T)
    eye = torch.eye(m, device=B.device)
    assert rel(B, C_ * (A @ A) + B_ * A + A_ * eye) < 4e-3
    out = X.float() if rows <= cols else X.float().T
    assert rel(out, B @ X0) < 4e-3


SHAPES_E2E = [(256, 768), (256, 256), (256, 1536), (768, 256),        # tiny decoder
              (768, 2304), (768, 768), (768, 3072), (3072, 768),       # GPT-2-small body
              (256, 1024), (1000, 1000), (129, 257), (1, 8), (8, 1), (5, 3),
              (1, 1)]                                                   # one element: sign(g) p^5(1)


@pytest.mark.parametrize("rows,cols", SHAPES_E2E)
def test_five_steps_match_fp64_oracle(zopt, rows, cols):
    G = gaussian(rows, cols, rows + 31 * cols)
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(rows, cols)
    zopt.ns_orthogonalize(G, X, ws, steps=5)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5)
    err = rel(X.cpu(), torch.from_numpy(ref))
    assert err <= 2e-2, err


def test_fp32_io_and_batch_strides(zopt):
    rows, cols, batch = 384, 1000, 3
    G = torch.randn(batch, rows, cols + 24, device="cuda")[:, :, :cols]  # padded rows: ld > cols
    X = torch.zeros(batch, rows, cols + 8, device="cuda")[:, :, :cols]
    ws = zopt.new_ns_workspace(rows, cols)
    zopt.ns_orthogonalize(G, X, ws, steps=5)
    torch.cuda.synchronize()
    for b in range(batch):
        ref = newton_schulz(G[b].double().cpu().numpy(), steps=5)
        assert rel(X[b].cpu(), torch.from_numpy(ref)) <= 2e-2
        one = torch.empty(rows, cols, device="cuda")
        zopt.ns_orthogonalize(G[b].contiguous(), one, ws, steps=5)
        torch.cuda.synchronize()
        assert torch.equal(one, X[b])  # a batch entry is bitwise the single call


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(300, 1000), (1000, 300)])
@pytest.mark.parametrize("pad,shift", [(8, 0), (3, 0), (0, 1), (8, 1)])
def test_output_pitch_and_alignment(zopt, pad, shift, rows, cols, dtype):
    """The last product writes the caller's X through the TMA (transposed for a tall matrix)
    when its rows are 16-byte aligned and by plain stores otherwise: padded rows (pitch cols +
    pad) and a base shifted by `shift` elements, bf16 and fp32, in groups of 2 and 1. Every
    result is bitwise the contiguous single call's, and the padding is left untouched."""
    batch = 3
    G = torch.randn(batch, rows, cols, device="cuda").to(dtype)
    ld = cols + pad
    flat = torch.full((batch * rows * ld + shift,), 7.0, device="cuda", dtype=dtype)
    full = flat[shift:].view(batch, rows, ld)
    X = full[:, :, :cols]
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols, group=2), steps=3)
    ws1 = zopt.new_ns_workspace(rows, cols)
    for b in range(batch):
        one = torch.empty(rows, cols, device="cuda", dtype=dtype)
        zopt.ns_orthogonalize(G[b].contiguous(), one, ws1, steps=3)
        torch.cuda.synchronize()
        assert torch.equal(one, X[b]), b
    if pad:
        assert bool((full[:, :, cols:] == 7.0).all())
    assert bool((flat[:shift] == 7.0).all())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(300, 1000), (1000, 300), (1000, 301), (301, 1000), (700, 13)])
@pytest.mark.parametrize("pad,shift", [(8, 0), (3, 0), (0, 1)])
def test_input_pitch_and_alignment(zopt, pad, shift, rows, cols, dtype):
    """The normalisation reads G through 16-byte accesses when its rows allow them and element by
    element otherwise (padded rows, a base off the 16-byte grid, a row length that leaves a
    partial piece): every result is within the oracle's tolerance, and where both reads visit
    the elements in the same order (16-byte rows, cols % 8 == 0) bitwise the contiguous call's."""
    batch = 2
    ld = cols + pad
    flat = torch.randn(batch * rows * ld + shift, device="cuda").to(dtype)
    G = flat[shift:].view(batch, rows, ld)[:, :, :cols]
    X = torch.empty(batch, rows, cols, device="cuda", dtype=dtype)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols, group=2), steps=3)
    torch.cuda.synchronize()
    esz = 2 if dtype == torch.bfloat16 else 4
    same_order = shift == 0 and (ld * esz) % 16 == 0 and cols % 8 == 0
    for b in range(batch):
        ref = newton_schulz(G[b].double().cpu().numpy(), steps=3)
        assert rel(X[b].cpu(), torch.from_numpy(ref)) <= 2e-2, b
        if same_order:
            one = torch.empty(rows, cols, device="cuda", dtype=dtype)
            zopt.ns_orthogonalize(G[b].contiguous(), one, zopt.new_ns_workspace(rows, cols), steps=3)
            torch.cuda.synchronize()
            assert torch.equal(one, X[b]), b


@pytest.mark.parametrize("compute", ["bf16", "f32"])
def test_grouped_batch_equals_single_calls(zopt, compute):
    """A workspace for 2 matrices runs a batch of 5 as groups of 2, 2, 1: every product is one
    launch over the group. Each result is bitwise the single-matrix call's."""
    code = zopt.BF16 if compute == "bf16" else zopt.F32
    rows, cols, batch = 700, 300, 5  # tall: processed transposed (single-CTA products)
    G = torch.randn(batch, rows, cols, device="cuda").to(torch.bfloat16)
    X = torch.empty_like(G)
    ws2 = zopt.new_ns_workspace(rows, cols, group=2, compute=code)
    assert ws2.numel() < zopt.ns_workspace(rows, cols, 3, code)
    zopt.ns_orthogonalize(G, X, ws2, steps=5, compute=code)
    ws1 = zopt.new_ns_workspace(rows, cols, compute=code)
    for b in range(batch):
        one = torch.empty(rows, cols, device="cuda", dtype=torch.bfloat16)
        zopt.ns_orthogonalize(G[b], one, ws1, steps=5, compute=code)
        torch.cuda.synchronize()
        assert torch.equal(one, X[b]), b
        ref = newton_schulz(G[b].double().cpu().numpy(), steps=5)
        assert rel(X[b].cpu(), torch.from_numpy(ref)) <= 2e-2


def test_grouped_batch_pair_kernel(zopt):
    """The same for m >= 1024 (CTA-pair products): 3 matrices of 1100 x 1300 in groups of 2."""
    rows, cols, batch = 1100, 1300, 3
    G = torch.randn(batch, rows, cols, device="cuda").to(torch.bfloat16)
    X = torch.empty_like(G)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols, group=2), steps=5)
    ws1 = zopt.new_ns_workspace(rows, cols)
    for b in range(batch):
        one = torch.empty(rows, cols, device="cuda", dtype=torch.bfloat16)
        zopt.ns_orthogonalize(G[b], one, ws1, steps=5)
        torch.cuda.synchronize()
        assert torch.equal(one, X[b]), b
    ref = newton_schulz(G[1].double().cpu().numpy(), steps=5)
    assert rel(X[1].cpu(), torch.from_numpy(ref)) <= 2e-2


@pytest.mark.parametrize("rows,cols,abc", [(256, 768, DEFAULT_ABC), (1024, 1536, DEFAULT_ABC),
                                            (512, 1024, (1.5, -0.5, 0.0))])
def test_first_step_reads_g_in_place_grouped_and_strided(zopt, rows, cols, abc):
    """A bf16 input no taller than wide, with 16-byte rows, is read in place by the first step
    (through its own tensor maps, with the caller's pitch and batch stride) on every product
    path: the fused launch (256 x 768), the CTA-pair launches (1024 x 1536), the single-CTA
    launches (a zero c rules out the identity MMAs). Rows padded to ld = cols + 16, three rows'
    gap between matrices, a workspace for groups of 2 over a batch of 3: every matrix bitwise the
    contiguous single call's, and within the tolerance of the fp64 oracle."""
    batch, ld, gap = 3, cols + 16, 3
    flat = torch.randn(batch * (rows + gap) * ld, device="cuda").to(torch.bfloat16)
    G = flat.view(batch, rows + gap, ld)[:, :rows, :cols]
    X = torch.empty(batch, rows, cols, device="cuda", dtype=torch.bfloat16)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols, group=2), steps=5, abc=abc)
    ws1 = zopt.new_ns_workspace(rows, cols)
    for b in range(batch):
        one = torch.empty(rows, cols, device="cuda", dtype=torch.bfloat16)
        zopt.ns_orthogonalize(G[b].contiguous(), one, ws1, steps=5, abc=abc)
        torch.cuda.synchronize()
        assert torch.equal(one, X[b]), b
        ref = newton_schulz(G[b].double().cpu().numpy(), steps=5, abc=abc)
        assert rel(X[b].cpu(), torch.from_numpy(ref)) <= 2e-2, b


def test_deterministic(zopt):
    G = gaussian(768, 3072, 1)
    ws = zopt.new_ns_workspace(768, 3072)
    outs = []
    for _ in range(2):
        X = torch.empty_like(G)
        zopt.ns_orthogonalize(G, X, ws, steps=5)
        outs.append(X)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def torch_ns_fp32(G, steps=5, abc=DEFAULT_ABC, eps=1e-7):
    a, b, c = abc
    X = G.float()
    X = X / (torch.linalg.norm(X) + eps)
    tr = X.shape[0] > X.shape[1]
    if tr:
        X = X.T
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if tr else X


@pytest.mark.parametrize("rows,cols", [(2048, 2048), (2048, 512), (2048, 11264)])
def test_llama_owned_matrices_match_fp64_oracle(zopt, rows, cols):
    """The 1.1B set's matrices owned by rank 0 of 8 (Wq, Wv, gate_up shapes), 5 steps."""
    G = gaussian(rows, cols, rows + cols)
    X = torch.empty_like(G)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols), steps=5)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5)
    assert rel(X.cpu(), torch.from_numpy(ref)) <= 2e-2


def test_stress_set_as_benchmarked_against_fp64_oracle(zopt):
    """The Newton-Schulz stress set in the launch configuration the benchmark times: 16 each of
    4096x4096, 4096x14336 and 14336x4096 bf16 matrices (entries N(0, 1), each divided by its
    Frobenius norm) in one zopt_ns_orthogonalize_many call, 5 steps, on the CTA-pair kernels.
    The first matrix of each shape is checked against the fp64 oracle fed the same bf16 input
    (relative Frobenius error <= 2e-2; bluscript_zero_ckpt.cpp, ShardedMuon note: the polynomial
    over the whole matrix); every matrix against a float32 Newton-Schulz on the GPU (the checker,
    TF32 off); and the top-left 256 x 1024 block of each shape's first matrix, taken as its own
    input, against the oracle."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        gen = torch.Generator(device="cuda").manual_seed(5)
        pairs = []
        for r, c in ((4096, 4096), (4096, 14336), (14336, 4096)):
            G = torch.randn(16, r, c, generator=gen, device="cuda")
            G /= torch.linalg.vector_norm(G, dim=(1, 2), keepdim=True)
            G = G.to(torch.bfloat16)
            pairs.append((G, torch.empty_like(G)))
        ws = zopt.new_ns_workspace_many([(G.shape[1], G.shape[2], G.shape[0]) for G, _ in pairs])
        zopt.ns_orthogonalize_many(pairs, ws, steps=5)
        torch.cuda.synchronize()
        del ws
        for G, X in pairs:
            ref = newton_schulz(G[0].double().cpu().numpy(), steps=5)
            err = rel(X[0].cpu(), torch.from_numpy(ref))
            assert err <= 2e-2, (tuple(G.shape), err)
            for i in range(G.shape[0]):
                assert rel(X[i].float(), torch_ns_fp32(G[i])) <= 2e-2, (tuple(G.shape), i)
            blk = G[0, :256, :1024].contiguous()
            Xb = torch.empty_like(blk)
            zopt.ns_orthogonalize(blk, Xb, zopt.new_ns_workspace(256, 1024), steps=5)
            torch.cuda.synchronize()
            refb = newton_schulz(blk.double().cpu().numpy(), steps=5)
            assert rel(Xb.cpu(), torch.from_numpy(refb)) <= 2e-2
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def test_rejects_bad_arguments(zopt):
    G = torch.zeros(8, 8, device="cuda", dtype=torch.bfloat16)
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(8, 8)
    with pytest.raises(zopt.ZoptError):
        zopt.ns_orthogonalize(G, X, ws, steps=0)
    with pytest.raises(zopt.ZoptError):
        zopt.ns_orthogonalize(G, X, ws[:16], steps=5)
    with pytest.raises(zopt.ZoptError):
        zopt.ns_orthogonalize(G, X, ws, abc=(float("nan"), 1.0, 1.0))


SHAPES_F32 = [(256, 768), (768, 256), (256, 1024), (300, 300), (129, 257), (1, 8), (8, 1), (768, 2304), (1000, 130)]


@pytest.mark.parametrize("rows,cols", SHAPES_F32)
def test_fp32_mode_matches_fp64_oracle_to_1e4(zopt, rows, cols):
    """compute_dtype fp32 with fp32 input/output: relative Frobenius error <= 1e-4."""
    g = torch.Generator(device="cuda").manual_seed(rows * 3 + cols)
    G = torch.randn(rows, cols, generator=g, device="cuda")
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(rows, cols, compute=zopt.F32)
    zopt.ns_orthogonalize(G, X, ws, steps=5, compute=zopt.F32)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5)
    err = rel(X.cpu(), torch.from_numpy(ref))
    assert err <= 1e-4, err


def test_fp32_mode_white_box_symmetric_products(zopt):
    rows, cols = 200, 333
    G = torch.randn(rows, cols, device="cuda")
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(rows, cols, compute=zopt.F32)
    zopt.ns_orthogonalize(G, X, ws, steps=1, compute=zopt.F32)
    torch.cuda.synchronize()
    p = plan(rows, cols, es=4)
    m, n = p["m"], p["n"]
    xbytes, abytes = p["xbytes"], p["abytes"]
    f32 = lambda off, r, ld, c: ws[off:off + r * ld * 4].view(torch.float32).view(r, ld)[:, :c]  # noqa: E731
    X0 = f32(p["x0"], m, p["ldx"], n).double()
    A = f32(p["x0"] + 2 * xbytes, m, p["lda"], m).double()
    B = f32(p["x0"] + 2 * xbytes + abytes, m, p["lda"], m).double()
    assert torch.equal(A, A.T) and torch.equal(B, B.T)
    assert rel(A, X0 @ X0.T) < 1e-5
    assert rel(B, C_ * (A @ A) + B_ * A) < 1e-5
    assert rel(X.double(), A_ * X0 + B @ X0) < 1e-5


def test_fp32_compute_with_bf16_io(zopt):
    G = gaussian(384, 1000, 77)
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(384, 1000, compute=zopt.F32)
    zopt.ns_orthogonalize(G, X, ws, steps=5, compute=zopt.F32)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5)
    assert rel(X.cpu(), torch.from_numpy(ref)) <= 4e-3  # one bf16 rounding of the output


def test_many_jobs_equal_single_calls(zopt):
    """zopt_ns_orthogonalize_many over jobs of different shapes, dtypes and orientations: five
    fused jobs, CTA-pair matrices with two 768-wide jobs riding their launches, and an output
    the TMA cannot address (product by product). Each job's result is bitwise
    zopt_ns_orthogonalize's with a workspace holding its whole batch, except the riders': each
    of those is bitwise what it gives beside another CTA-pair job, and within 2e-2 of the fp64
    oracle; one other job is checked against the oracle too."""
    gen = torch.Generator(device="cuda").manual_seed(11)
    specs = [(12, 768, 2304, torch.bfloat16, 0), (5, 768, 768, torch.bfloat16, 0), (3, 1000, 300, torch.float32, 0),
             (2, 130, 70, torch.bfloat16, 0), (1, 256, 512, torch.bfloat16, 0), (2, 64, 64, torch.float32, 0),
             (1, 17, 100, torch.bfloat16, 0), (2, 1100, 1300, torch.bfloat16, 0), (1, 300, 1000, torch.bfloat16, 3)]
    pairs, shapes = [], []
    for b, r, c, dt, pad in specs:
        G = torch.randn(b, r, c, generator=gen, device="cuda").to(dt)
        X = torch.zeros(b, r, c + pad, device="cuda", dtype=dt)[:, :, :c]
        pairs.append((G, X))
        shapes.append((r, c, b))
    ws = zopt.new_ns_workspace_many(shapes)
    zopt.ns_orthogonalize_many(pairs, ws, steps=5)
    torch.cuda.synchronize()
    other = torch.randn(1, 1024, 1024, generator=gen, device="cuda").bfloat16()
    for (G, X), (r, c, b) in zip(pairs, shapes):
        one = torch.empty(b, r, c, device="cuda", dtype=G.dtype)
        if 512 <= min(r, c) < 1024:  # a rider of the 1100 x 1300 job's CTA-pair launches
            zopt.ns_orthogonalize_many([(other, torch.empty_like(other)), (G, one)],
                                       zopt.new_ns_workspace_many([(1024, 1024, 1), (r, c, b)]), steps=5)
            torch.cuda.synchronize()
            assert torch.equal(one, X), (r, c, b)
            ref = newton_schulz(G[b - 1].double().cpu().numpy(), steps=5)
            assert rel(X[b - 1].cpu(), torch.from_numpy(ref)) <= 2e-2
            continue
        zopt.ns_orthogonalize(G, one, zopt.new_ns_workspace(r, c, b), steps=5)
        torch.cuda.synchronize()
        assert torch.equal(one, X), (r, c, b)
    ref = newton_schulz(pairs[2][0][1].double().cpu().numpy(), steps=5)
    assert rel(pairs[2][1][1].cpu(), torch.from_numpy(ref)) <= 2e-2


@pytest.mark.parametrize("steps", [1, 2, 7])
def test_many_jobs_step_counts(zopt, steps):
    """The fused work list at other step counts: with one step the first B'X is also the last
    (into the caller's X); each job still equals its single call bit for bit."""
    gen = torch.Generator(device="cuda").manual_seed(steps)
    specs = [(3, 256, 768, torch.bfloat16), (2, 768, 256, torch.float32), (1, 100, 130, torch.bfloat16)]
    pairs = [(torch.randn(b, r, c, generator=gen, device="cuda").to(dt),
              torch.empty(b, r, c, device="cuda", dtype=dt)) for b, r, c, dt in specs]
    zopt.ns_orthogonalize_many(pairs, zopt.new_ns_workspace_many([(r, c, b) for b, r, c, _ in specs]), steps=steps)
    torch.cuda.synchronize()
    for (G, X), (b, r, c, _) in zip(pairs, specs):
        one = torch.empty_like(X)
        zopt.ns_orthogonalize(G, one, zopt.new_ns_workspace(r, c, b), steps=steps)
        torch.cuda.synchronize()
        assert torch.equal(one, X), (r, c, steps)
        ref = newton_schulz(G[0].double().cpu().numpy(), steps=steps)
        assert rel(X[0].cpu(), torch.from_numpy(ref)) <= 2e-2


def test_many_jobs_beyond_one_preparation_list(zopt):
    """Nineteen jobs: more than one preparation launch's worth of items (the norm list holds 19,
    the scaling list 17, the transpose list 2), three fused launches of six jobs, and one job
    (fp32, 33 columns) whose output the TMA cannot address, product by product. Each job equals
    its single call bit for bit."""
    gen = torch.Generator(device="cuda").manual_seed(41)
    specs = [(1 + j % 3, 64 + 16 * j, 96 + 24 * j, torch.bfloat16 if j % 2 == 0 else torch.float32) for j in range(17)]
    specs += [(2, 300, 120, torch.bfloat16), (1, 257, 33, torch.float32)]
    pairs = [(torch.randn(b, r, c, generator=gen, device="cuda").to(dt),
              torch.empty(b, r, c, device="cuda", dtype=dt)) for b, r, c, dt in specs]
    zopt.ns_orthogonalize_many(pairs, zopt.new_ns_workspace_many([(r, c, b) for b, r, c, _ in specs]), steps=2)
    torch.cuda.synchronize()
    for (G, X), (b, r, c, _) in zip(pairs, specs):
        one = torch.empty_like(X)
        zopt.ns_orthogonalize(G, one, zopt.new_ns_workspace(r, c, b), steps=2)
        torch.cuda.synchronize()
        assert torch.equal(one, X), (r, c, b)
    ref = newton_schulz(pairs[17][0][1].double().cpu().numpy(), steps=2)
    assert rel(pairs[17][1][1].cpu(), torch.from_numpy(ref)) <= 2e-2


def test_gpt2_small_body_in_one_call(zopt):
    """The GPT-2-small body's 48 Muon matrices (12 each of 768x2304, 768x768, 768x3072,
    3072x768; 1e-3-scaled Gaussian gradients) in one zopt_ns_orthogonalize_many call, the launch
    configuration the small-matrix benchmark times: every shape bitwise its own single call, and
    the first and last matrix of every shape within 2e-2 of the fp64 oracle."""
    w = workloads.get("c2")
    shapes = sorted({p.shape for p in w.muon})
    pairs = []
    for k, (r, c) in enumerate(shapes):
        count = sum(1 for p in w.muon if p.shape == (r, c))
        G = torch.stack([workloads.ns_input(r, c, w.seed, 100 * k + i, dtype=torch.float32)
                         for i in range(count)]) * 1e-3
        G = G.to(torch.bfloat16).cuda()
        pairs.append((G, torch.empty_like(G)))
    assert sum(G.shape[0] for G, _ in pairs) == 48
    zopt.ns_orthogonalize_many(pairs, zopt.new_ns_workspace_many([(G.shape[1], G.shape[2], G.shape[0])
                                                                  for G, _ in pairs]), steps=5)
    torch.cuda.synchronize()
    for G, X in pairs:
        one = torch.empty_like(X)
        zopt.ns_orthogonalize(G, one, zopt.new_ns_workspace(G.shape[1], G.shape[2], G.shape[0]), steps=5)
        torch.cuda.synchronize()
        assert torch.equal(one, X), tuple(G.shape)
        for i in (0, G.shape[0] - 1):
            ref = newton_schulz(G[i].double().cpu().numpy(), steps=5)
            assert rel(X[i].cpu(), torch.from_numpy(ref)) <= 2e-2, (tuple(G.shape), i)


def test_many_pair_jobs_batched(zopt):
    """zopt_ns_orthogonalize_many runs each product of a step for all its CTA-pair jobs (m >= 1024)
    in one launch, four jobs to a launch and those with the same epilogue together: six pair jobs
    of different shapes, dtypes and orientations (two launches per product), one whose output the
    TMA cannot address (its last product by plain stores, in a launch of its own) and a fused job
    beside them. Each result is bitwise its single call's; one is checked against the oracle."""
    gen = torch.Generator(device="cuda").manual_seed(29)
    specs = [(1, 1024, 1024, torch.bfloat16, 0), (2, 1024, 1536, torch.bfloat16, 0), (1, 1100, 1300, torch.float32, 0),
             (1, 2000, 1030, torch.bfloat16, 0), (1, 1030, 1100, torch.bfloat16, 3), (1, 1280, 1024, torch.float32, 0),
             (2, 300, 700, torch.bfloat16, 0)]
    pairs, shapes = [], []
    for b, r, c, dt, pad in specs:
        G = torch.randn(b, r, c, generator=gen, device="cuda").to(dt)
        X = torch.zeros(b, r, c + pad, device="cuda", dtype=dt)[:, :, :c]
        pairs.append((G, X))
        shapes.append((r, c, b))
    zopt.ns_orthogonalize_many(pairs, zopt.new_ns_workspace_many(shapes), steps=3)
    torch.cuda.synchronize()
    for (G, X), (r, c, b) in zip(pairs, shapes):
        one = torch.empty(b, r, c, device="cuda", dtype=G.dtype)
        zopt.ns_orthogonalize(G, one, zopt.new_ns_workspace(r, c, b), steps=3)
        torch.cuda.synchronize()
        assert torch.equal(one, X), (r, c, b)
    ref = newton_schulz(pairs[3][0][0].double().cpu().numpy(), steps=3)
    assert rel(pairs[3][1][0].cpu(), torch.from_numpy(ref)) <= 2e-2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols", [(300, 700), (700, 300), (1024, 1100)])
def test_zero_matrix_gives_zero(zopt, rows, cols, dtype):
    """G = 0: ||G|| = 0, X0 = 0 / (0 + eps) = 0 and every product stays 0, so the output is
    exactly zero, as the oracle's plain definition gives; in a many-jobs call as well."""
    G = torch.zeros(rows, cols, device="cuda", dtype=dtype)
    X = torch.full_like(G, 7.0)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols), steps=5)
    torch.cuda.synchronize()
    assert bool((X == 0).all())
    assert np.all(newton_schulz(np.zeros((rows, cols)), steps=5) == 0)
    if dtype == torch.bfloat16:
        Y = torch.full((1, rows, cols), 7.0, device="cuda", dtype=dtype)
        H = torch.randn(2, 256, 512, device="cuda").to(dtype)
        Hx = torch.empty_like(H)
        zopt.ns_orthogonalize_many([(G[None], Y), (H, Hx)],
                                   zopt.new_ns_workspace_many([(rows, cols, 1), (256, 512, 2)]), steps=5)
        torch.cuda.synchronize()
        assert bool((Y == 0).all()) and bool(torch.isfinite(Hx.float()).all())


def p5(s, abc=DEFAULT_ABC, steps=5):
    a, b, c = abc
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


@pytest.mark.parametrize("rows,cols", [(256, 768), (768, 256), (1024, 1536)])
def test_rank_one_closed_form(zopt, rows, cols):
    """An exactly rank-1 G = u v' (entries that bf16 holds exactly) has the one singular value
    ||G||_F: X0 = G / (||G|| + eps) has singular value s = ||G|| / (||G|| + eps), a step maps it by
    p(s) = a s + b s^3 + c s^5 and keeps the singular vectors, so one step gives
    p(s) u v' / (|u| |v|); the GPU result is within the bf16 tolerance of that closed form (the
    fp64 oracle agrees to 1e-10). One step only: the bf16 rounding of X0 leaves noise of ~2^-9 in
    the null directions, which every step multiplies by about a = 3.44 (5 steps: ~490x), so
    a rank-deficient input is a case where bf16 Newton-Schulz parts from the exact result."""
    g = torch.Generator().manual_seed(rows + cols)
    u = torch.randint(-4, 5, (rows,), generator=g).double() / 4
    v = torch.randint(-4, 5, (cols,), generator=g).double() / 4
    u[0], v[0] = 1.0, 1.0  # nonzero vectors
    Gd = torch.outer(u, v)
    G = Gd.to(torch.bfloat16).cuda()
    assert torch.equal(G.double().cpu(), Gd)  # exactly representable
    X = torch.empty_like(G)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols), steps=1)
    torch.cuda.synchronize()
    fro = float(torch.linalg.norm(Gd))
    closed = p5(fro / (fro + 1e-7), steps=1) * torch.outer(u / torch.linalg.norm(u), v / torch.linalg.norm(v))
    assert rel(torch.from_numpy(newton_schulz(Gd.numpy(), steps=1)), closed) <= 1e-10
    closed5 = p5(fro / (fro + 1e-7)) * torch.outer(u / torch.linalg.norm(u), v / torch.linalg.norm(v))
    assert rel(torch.from_numpy(newton_schulz(Gd.numpy(), steps=5)), closed5) <= 1e-10
    assert rel(X.cpu(), closed) <= 2e-2


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_input_propagates_and_context_survives(zopt, bad):
    """A non-finite element makes ||G|| non-finite: the output carries non-finite values (as the
    oracle's does); the call returns normally and the next call on finite input is correct."""
    rows, cols = 256, 768
    G = gaussian(rows, cols, 3)
    G[5, 7] = bad
    X = torch.empty_like(G)
    ws = zopt.new_ns_workspace(rows, cols)
    zopt.ns_orthogonalize(G, X, ws, steps=5)
    torch.cuda.synchronize()
    assert not bool(torch.isfinite(X.float()).all())
    with np.errstate(invalid="ignore"):  # inf / inf in the oracle's normalisation is the point
        assert not np.all(np.isfinite(newton_schulz(G.double().cpu().numpy(), steps=5)))
    G2 = gaussian(rows, cols, 4)
    zopt.ns_orthogonalize(G2, X, ws, steps=5)
    torch.cuda.synchronize()
    assert rel(X.cpu(), torch.from_numpy(newton_schulz(G2.double().cpu().numpy(), steps=5))) <= 2e-2


@pytest.mark.parametrize("abc", [(1.5, -0.5, 0.0), (2.0, -1.5, 0.5), (3.0, -3.2, 1.2)])
@pytest.mark.parametrize("rows,cols", [(256, 768), (768, 256), (1024, 1100)])
def test_other_coefficients_match_fp64_oracle(zopt, abc, rows, cols):
    """The triple is an argument: with c = 0 (the cubic Newton-Schulz 1.5 X - 0.5 X X' X) the b A
    term cannot ride on identity MMAs scaled by 1/c, so B' takes it through the R epilogue
    instead of the fused kernel; other triples take the usual paths. Each result is within the
    bf16 tolerance of the fp64 oracle run with the same triple, and in a many-jobs call bitwise
    the single call's."""
    G = gaussian(rows, cols, rows + cols + int(abc[0] * 10))
    X = torch.empty_like(G)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(rows, cols), steps=5, abc=abc)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5, abc=abc)
    assert rel(X.cpu(), torch.from_numpy(ref)) <= 2e-2
    Y = torch.empty(1, rows, cols, device="cuda", dtype=torch.bfloat16)
    H = gaussian(300, 700, 5)[None]
    Hx = torch.empty_like(H)
    zopt.ns_orthogonalize_many([(G[None], Y), (H, Hx)],
                               zopt.new_ns_workspace_many([(rows, cols, 1), (300, 700, 1)]), steps=5, abc=abc)
    torch.cuda.synchronize()
    assert torch.equal(Y[0], X)


@pytest.mark.parametrize("abc", [(1.5, -0.5, 0.0), (2.0, -1.5, 0.5)])
def test_other_coefficients_fp32_mode(zopt, abc):
    G = torch.randn(256, 640, device="cuda")
    X = torch.empty_like(G)
    zopt.ns_orthogonalize(G, X, zopt.new_ns_workspace(256, 640, compute=zopt.F32), steps=5, abc=abc,
                          compute=zopt.F32)
    torch.cuda.synchronize()
    ref = newton_schulz(G.double().cpu().numpy(), steps=5, abc=abc)
    assert rel(X.cpu(), torch.from_numpy(ref)) <= 1e-4
