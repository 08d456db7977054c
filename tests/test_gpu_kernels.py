"""GPU parity of every kernel against the oracle on small and ragged shapes.

Tolerances:
  * AdamW and the momentum buffer M: bit-exact (both sides evaluate the same
    separately rounded fp32 operations; division and sqrt are correctly
    rounded on both).
  * Newton-Schulz output and the Muon update dW: relative Frobenius error
    <= 1e-2 per matrix.  Both sides store A, B and X in bf16 at the same
    points; they differ in accumulation (fp32 tensor-core vs fp64), which
    flips a small fraction of bf16 roundings.  Measured between an fp32-
    and an fp64-accumulating evaluation of the same iteration the gap is
    0.3-0.5% on Gaussian inputs from 256x512 to 1408x2048.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m
import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
NS_TOL = 1e-2


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (d if d > 0 else 1.0)


def bf16_to_np(t):
    return t.float().cpu().numpy()


# --------------------------------------------------------------------------
# AdamW
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, 4097, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1])
def test_adamw_bit_exact(lib, n, offset):
    a = workloads.make_adamw(n + offset, seed=n, device=DEV)
    p, g, mm, v = (x[offset:] for x in (a.p, a.g, a.m, a.v))  # offset 1 -> scalar path
    host = [x.cpu().numpy() for x in (p, g, mm, v)]
    hp = m.AdamwHparams()
    m.adamw_step(p, g, mm, v, hp, step=100)
    rp, rm, rv = oracle.adamw_step(*host, oracle.AdamwConfig(), t=100)
    assert np.array_equal(p.cpu().numpy(), rp)
    assert np.array_equal(mm.cpu().numpy(), rm)
    assert np.array_equal(v.cpu().numpy(), rv)


def test_adamw_first_step_and_decay(lib):
    a = workloads.make_adamw(4096, seed=9, device=DEV)
    a.m.zero_()
    a.v.zero_()
    host = [x.cpu().numpy() for x in (a.p, a.g, a.m, a.v)]
    hp = m.AdamwHparams(lr=1e-3, weight_decay=0.05)
    m.adamw_step(a.p, a.g, a.m, a.v, hp, step=1)
    rp, _, _ = oracle.adamw_step(*host, oracle.AdamwConfig(lr=1e-3, weight_decay=0.05), t=1)
    assert np.array_equal(a.p.cpu().numpy(), rp)


# --------------------------------------------------------------------------
# Newton-Schulz (tcgen05 GEMMs)
# --------------------------------------------------------------------------

def run_ns(shape, count, steps=5, coeffs=oracle.QUINTIC, seed=0, kind="gaussian"):
    mp, np_ = shape
    X = torch.stack([workloads.ns_input(mp, np_, seed + i, kind) for i in range(count)]).to(DEV)
    out = m.muon_newton_schulz(X, steps=steps, coeffs=coeffs)
    torch.cuda.synchronize()
    return X.float().cpu().numpy(), bf16_to_np(out)


@pytest.mark.parametrize("coeffs,what", [((1.0, 0.0, 0.0), "identity"), ((0.0, 1.0, 0.0), "AX"),
                                         ((0.0, 0.0, 1.0), "AAX")])
@pytest.mark.parametrize("shape", [(64, 64), (128, 256), (200, 328), (256, 512), (520, 1100), (512, 900),
                                   (1152, 1536), (1370, 1500), (1600, 1664)])
def test_ns_single_stage_isolation(lib, shape, coeffs, what):
    """One step with one coefficient set isolates one product:
    (1,0,0) -> X;  (0,1,0) -> (X X^T) X;  (0,0,1) -> (X X^T)^2 X."""
    X, got = run_ns(shape, 2, steps=1, coeffs=coeffs, seed=3)
    for i in range(2):
        ref = oracle.newton_schulz(X[i], steps=1, coeffs=coeffs)
        if what == "identity":
            assert np.array_equal(got[i], ref)
        else:
            assert rel_fro(got[i], ref) < NS_TOL, what


# m' above 512 and within 1/8 of a multiple of 256 runs on CTA pairs
# (256x256 pair tiles, two 64-deep k-blocks per ring stage), other m' on
# single CTAs; both kinds, ragged edges and odd k-block counts (a
# half-filled last stage) included, are covered here.  Symmetric factors are
# read transposed left of the diagonal block: (520, 1100) has single-CTA
# tiles whose two 128-row halves of B take different layouts in one k-block,
# (1000, 1100) and (960, 1100) pair tiles with a ragged last row block,
# (720, 900) a last pair row with 48 padded rows (between 1/16 and 1/8 of m',
# like the 1408-row experts); (768, 960) pair tiles on 64-aligned shapes
# (chunked MN-major copies) with a ragged last column tile, and (512, 832)
# the same shape class on single CTAs.
# (1152, 1536), (1408, 2048) and (1408, 2112) run on pairs with a
# half-empty last pair row (m' an odd multiple of 128), the last two with the
# mixed step's expert rows and n' on and off the 256 grid.  (1150, 1300) and
# (1370, 1500) have ragged last pair rows of 126 and 90 rows on plain maps,
# and (1600, 1664) one of 64 rows on chunked maps, where the second CTA's
# half lies wholly past the matrix.
@pytest.mark.parametrize("shape", [(1, 1), (7, 13), (8, 8), (64, 64), (128, 256), (129, 257),
                                   (200, 328), (256, 512), (300, 1000), (384, 384), (464, 600), (720, 900), (520, 1100),
                                   (512, 512), (512, 832), (512, 900), (768, 800), (768, 960), (960, 1100),
                                   (1000, 1100), (1152, 1536), (1408, 2048), (1408, 2112), (1150, 1300),
                                   (1370, 1500), (1600, 1664)])
def test_ns_parity(lib, shape):
    count = 3 if shape[0] * shape[1] < 200_000 else 1
    X, got = run_ns(shape, count, seed=11)
    for i in range(count):
        ref = oracle.newton_schulz(X[i])
        assert rel_fro(got[i], ref) < NS_TOL, (shape, i)


@pytest.mark.parametrize("shape", [(256, 512), (130, 300)])
def test_ns_batches_in_several_passes_match_single_calls(lib, shape):
    """Five matrices through a workspace that holds two run in three passes
    (2, 2, 1); each result must equal the matrix run on its own, bit for
    bit.  (256, 512) has unpadded workspace rows, so each pass moves its
    matrices in and out with one strided copy; (130, 300) has padded rows
    (300 is not a multiple of 8) and copies matrix by matrix."""
    mp, np_ = shape
    X = torch.stack([workloads.ns_input(mp, np_, 40 + i) for i in range(5)]).to(DEV)
    ws = m.allocate_workspace(2 * m.muon_workspace_bytes_per_matrix(mp, np_))
    got = m.muon_newton_schulz(X, workspace=ws)
    for i in range(5):
        alone = m.muon_newton_schulz(X[i:i + 1].contiguous())
        assert torch.equal(got[i], alone[0]), i


def test_ns_zero_steps_copies(lib):
    X, got = run_ns((40, 72), 2, steps=0)
    assert np.array_equal(X, got)


def test_ns_cubic_page_coefficients(lib):
    """The page's cubic (1.5, -0.5, 0) runs through the same kernels."""
    X, got = run_ns((128, 384), 1, steps=8, coeffs=oracle.CUBIC, seed=5)
    ref = oracle.newton_schulz(X[0], steps=8, coeffs=oracle.CUBIC)
    assert rel_fro(got[0], ref) < NS_TOL


def test_ns_deterministic(lib):
    X = torch.stack([workloads.ns_input(256, 640, 1 + i) for i in range(4)]).to(DEV)
    a = m.muon_newton_schulz(X)
    b = m.muon_newton_schulz(X)
    assert torch.equal(a, b)


# --------------------------------------------------------------------------
# Full Muon step
# --------------------------------------------------------------------------

def make_mats(shapes, dtypes, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    W, G, M = [], [], []
    for (r, c), dt in zip(shapes, dtypes):
        W.append(torch.randn(r, c, device=DEV, generator=gen) * 0.02)
        G.append((torch.randn(r, c, device=DEV, generator=gen) * 1e-2).to(dt))
        M.append(torch.randn(r, c, device=DEV, generator=gen) * 1e-2)
    return W, G, M


def check_step(W0, G0, M0, W1, M1, hp):
    cfg = oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                            nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a,
                            ns_b=hp.ns_b, ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale)
    oW, oM, _, _ = oracle.muon_step_matrix(W0, G0, M0, cfg)
    assert np.array_equal(M1, oM)
    assert rel_fro(W1.astype(np.float64) - W0, oW.astype(np.float64) - W0) < NS_TOL
    return oW


SHAPES = [(256, 512), (512, 256), (7, 13), (13, 7), (1, 1), (130, 70), (64, 1024), (300, 300),
          (512, 900), (900, 512), (1152, 1536), (1536, 1152)]


@pytest.mark.parametrize("gdt", [torch.float32, torch.bfloat16])
def test_step_mixed_shapes(lib, gdt):
    W, G, M = make_mats(SHAPES, [gdt] * len(SHAPES), seed=1)
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams()
    ws = m.muon_step_batched(W, G, M, hp)
    assert m.muon_query_status(ws) == 0
    for i, (w0, g0, m0) in enumerate(host):
        check_step(w0, g0, m0, W[i].cpu().numpy(), M[i].cpu().numpy(), hp)


def test_step_mixed_dtypes_and_unaligned(lib):
    shapes = [(96, 160), (160, 96), (33, 65), (65, 33)]
    W, G, M = make_mats(shapes, [torch.float32, torch.bfloat16, torch.float32, torch.float32], seed=2)
    # unaligned views force the scalar paths, for a wide and a tall matrix
    for k in (2, 3):
        base = torch.randn(33 * 65 + 1, device=DEV) * 0.02
        W[k] = base[1:].view(*shapes[k])
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)
    for i, (w0, g0, m0) in enumerate(host):
        check_step(w0, g0, m0, W[i].cpu().numpy(), M[i].cpu().numpy(), hp)


def test_step_chunking_is_bit_identical(lib):
    shapes = [(256, 512)] * 3 + [(512, 256)] * 2 + [(64, 64)] * 4
    W, G, M = make_mats(shapes, [torch.float32] * len(shapes), seed=3)
    W2, G2, M2 = [w.clone() for w in W], G, [x.clone() for x in M]
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)  # one chunk
    small = max(m.muon_workspace_bytes_per_matrix(*s) for s in shapes)
    plan = m.muon_plan(shapes, small)
    assert plan["chunk_id"].max() >= 4
    ws = m.allocate_workspace(small)
    m.muon_step_batched(W2, G2, M2, hp, workspace=ws)
    for a, b in zip(W, W2):
        assert torch.equal(a, b)
    for a, b in zip(M, M2):
        assert torch.equal(a, b)


def test_step_zero_gradient_is_pure_decay(lib):
    shapes = [(128, 256), (256, 128)]
    W, G, M = make_mats(shapes, [torch.float32] * 2, seed=4)
    for g, mm in zip(G, M):
        g.zero_()
        mm.zero_()
    W0 = [w.cpu().numpy() for w in W]
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)
    for w0, w in zip(W0, W):
        ref = oracle.final_update(w0, np.zeros((min(w0.shape), max(w0.shape)), np.float32),
                                  hp.lr, hp.weight_decay, hp.rms_scale)
        got = w.cpu().numpy()
        assert np.array_equal(got, ref)
        assert np.isfinite(got).all()


@pytest.mark.parametrize("magnitude", [1e-16, 1e14])
def test_step_extreme_gradient_scale(lib, magnitude):
    """Norms far outside [2^-40, 2^40]: X0 is normalised in place before the
    first NS step instead of inside it (products of unnormalised bf16
    elements would leave the normal fp32 range).  (1152, 1536) runs on CTA
    pairs with a half-empty last pair row."""
    shapes = [(128, 256), (384, 128), (1152, 1536)]
    W, G, M = make_mats(shapes, [torch.float32] * len(shapes), seed=8)
    for g, mm in zip(G, M):
        g.mul_(magnitude / 1e-2)
        mm.mul_(magnitude / 1e-2)
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)
    for i, (w0, g0, m0) in enumerate(host):
        check_step(w0, g0, m0, W[i].cpu().numpy(), M[i].cpu().numpy(), hp)


@pytest.mark.parametrize("p2", [2.0 ** 50, 2.0 ** -50])
def test_out_of_range_norm_path_is_exact(lib, p2):
    """Scaling G and M by a power of two scales u, bf16(u) and the norm
    exactly, so with norm_eps = 0 the NS input s * bf16(u) is unchanged.
    The scaled norms lie outside [2^-40, 2^40], where X0 takes a power of two
    from the scale; the update must still be bit-identical (also on the CTA
    pairs of (1536, 1152), tall, with a half-empty last pair row)."""
    shapes = [(128, 256), (384, 128), (1536, 1152)]
    W, G, M = make_mats(shapes, [torch.float32] * len(shapes), seed=10)
    W2 = [w.clone() for w in W]
    G2 = [g * p2 for g in G]
    M2 = [x * p2 for x in M]
    hp = m.MuonHparams(norm_eps=0.0)
    m.muon_step_batched(W, G, M, hp)
    m.muon_step_batched(W2, G2, M2, hp)
    for a, b in zip(W, W2):
        assert torch.equal(a, b)
    for a, b in zip(M, M2):
        assert torch.equal(a * p2, b)


def test_step_without_ns_steps(lib):
    """ns_steps = 0: the update is the normalised look-ahead itself."""
    shapes = [(96, 160), (160, 96)]
    W, G, M = make_mats(shapes, [torch.float32] * 2, seed=9)
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams(ns_steps=0)
    m.muon_step_batched(W, G, M, hp)
    for i, (w0, g0, m0) in enumerate(host):
        check_step(w0, g0, m0, W[i].cpu().numpy(), M[i].cpu().numpy(), hp)


@pytest.mark.parametrize("nesterov", [False, True])
def test_step_hparam_variants(lib, nesterov):
    shapes = [(192, 320)]
    W, G, M = make_mats(shapes, [torch.bfloat16], seed=5)
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams(lr=0.05, weight_decay=0.0, momentum=0.9, nesterov=nesterov, ns_steps=3)
    m.muon_step_batched(W, G, M, hp)
    check_step(*host[0], W[0].cpu().numpy(), M[0].cpu().numpy(), hp)


def test_step_two_steps_resume_exact(lib):
    """The library is stateless: two steps in a row equal step, copy the
    state out and back in, step again."""
    shapes = [(128, 384), (384, 128)]
    W, G, M = make_mats(shapes, [torch.float32] * 2, seed=6)
    Wb, Mb = [w.clone() for w in W], [x.clone() for x in M]
    hp = m.MuonHparams()
    m.muon_step_batched(W, G, M, hp)
    m.muon_step_batched(W, G, M, hp)
    m.muon_step_batched(Wb, G, Mb, hp)
    Wc = [torch.from_numpy(w.cpu().numpy()).to(DEV) for w in Wb]
    Mc = [torch.from_numpy(x.cpu().numpy()).to(DEV) for x in Mb]
    m.muon_step_batched(Wc, G, Mc, hp)
    for a, b in zip(W + M, Wc + Mc):
        assert torch.equal(a, b)


@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float32])
def test_step_ragged_tall_multi_tile_units(lib, gdt):
    """A tall matrix with more 64x64 tiles than one momentum partial per tile
    allows (2100 x 2050: 33 x 33 tiles), so the momentum pass walks units of
    two row tiles (for bf16 gradients prefetching the next tile across
    partial ones), and the final update walks units of up to four row tiles
    with a partial last row group and a partial last column.  The momentum
    is bit-exact; the update matches the oracle's full step."""
    shapes = [(2100, 2050)]
    W, G, M = make_mats(shapes, [gdt], seed=12)
    host = [(w.cpu().numpy(), g.float().cpu().numpy(), mm.cpu().numpy()) for w, g, mm in zip(W, G, M)]
    hp = m.MuonHparams()
    ws = m.muon_step_batched(W, G, M, hp)
    assert m.muon_query_status(ws) == 0
    check_step(*host[0], W[0].cpu().numpy(), M[0].cpu().numpy(), hp)


def test_caller_kernel_after_the_step_sees_its_results(lib):
    """The step's kernels are chained by programmatic dependent launch; a
    kernel the caller enqueues next on the same stream (here torch's clone
    and add, with no synchronisation in between) must still see the final W
    and M.  Repeated over back-to-back steps, each checked against the
    step computed once more on copies."""
    shapes = [(256, 512), (512, 256), (1152, 1536)]
    W, G, M = make_mats(shapes, [torch.float32] * len(shapes), seed=21)
    Wr, Mr = [w.clone() for w in W], [x.clone() for x in M]
    hp = m.MuonHparams()
    ws = m.allocate_workspace(m.muon_workspace_size(shapes, 1 << 34))
    for _ in range(3):
        m.muon_step_batched(W, G, M, hp, workspace=ws)
        seen_W = [w.clone() + 0.0 for w in W]     # caller kernels, same stream, no sync
        seen_M = [x.clone() + 0.0 for x in M]
        m.muon_step_batched(Wr, G, Mr, hp, workspace=ws)
        torch.cuda.synchronize()
        for a, b in zip(seen_W + seen_M, Wr + Mr):
            assert torch.equal(a, b)


def test_step_over_more_matrices_than_one_launch_grid(lib):
    """70,000 small matrices in one call and one workspace chunk: more than
    the 65,535 rows one launch grid takes, so the momentum, final-update
    and statistics passes each split into two launches, the records go up
    in 313 uploads of up to 224, and one NS group holds them all.  Wide
    8x16 and tall 16x8 matrices alternate, with fp32 and bf16 gradients.
    Sampled matrices around the 65,535 boundary, the last one and a spread
    between are checked against the oracle (momentum bit-exact, update
    within the parity tolerance, statistics as in test_gpu_stats)."""
    n = 70_000
    shapes = [(8, 16) if i % 2 == 0 else (16, 8) for i in range(n)]
    gen = torch.Generator(device=DEV).manual_seed(71)
    Wf = torch.randn(n * 128, device=DEV, generator=gen) * 0.02
    Gf = torch.randn(n * 128, device=DEV, generator=gen) * 1e-2
    Gh = Gf.to(torch.bfloat16)
    Mf = torch.randn(n * 128, device=DEV, generator=gen) * 1e-2
    W = [Wf[128 * i:128 * (i + 1)].view(*shapes[i]) for i in range(n)]
    G = [(Gh if i % 4 >= 2 else Gf)[128 * i:128 * (i + 1)].view(*shapes[i]) for i in range(n)]
    M = [Mf[128 * i:128 * (i + 1)].view(*shapes[i]) for i in range(n)]
    sample = sorted({0, 1, 2, 3, 65533, 65534, 65535, 65536, 65537, n - 2, n - 1} | set(range(97, n, 4999)))
    W0 = {i: W[i].cpu().numpy() for i in sample}
    G0 = {i: G[i].float().cpu().numpy() for i in sample}
    M0 = {i: M[i].cpu().numpy() for i in sample}
    hp = m.MuonHparams()
    ws_bytes = m.muon_workspace_size(shapes, 1 << 34)
    assert m.muon_plan(shapes, ws_bytes)["chunk_id"].max() == 0   # one chunk: every launch sees all 70,000
    ws = m.allocate_workspace(ws_bytes)
    stats = torch.empty(n, 2, dtype=torch.float64, device=DEV)
    m.muon_step_batched(W, G, M, hp, workspace=ws, stats=stats)
    torch.cuda.synchronize()
    assert m.muon_query_status(ws) == 0
    st = stats.cpu().numpy()
    cfg = oracle.MuonConfig()
    for i in sample:
        oW, oM, _, O = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
        assert np.array_equal(M[i].cpu().numpy(), oM), i
        dW = W[i].cpu().numpy().astype(np.float64) - W0[i]
        assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < NS_TOL, i
        _, u = oracle.momentum(G0[i], M0[i], cfg.momentum, cfg.nesterov)
        u_norm, rms = oracle.step_stats(u, O, cfg.rms_scale, cfg.scale_mode)
        assert abs(st[i, 0] - u_norm) <= 1e-5 * u_norm, i
        assert abs(st[i, 1] - rms) <= 2e-3 * rms, i


def test_step_sees_a_gradient_the_caller_wrote_just_before(lib):
    """The step's first kernel may launch before the caller's previous
    kernel on the same stream has finished (programmatic dependent launch),
    but it waits for it before reading: a gradient scaled by the caller's own
    kernel right before the call, with no synchronisation, is the one the
    step uses.  Checked against the step on a gradient scaled beforehand."""
    shapes = [(256, 512), (1152, 1536)]
    W, G, M = make_mats(shapes, [torch.float32] * len(shapes), seed=22)
    W2, M2 = [w.clone() for w in W], [x.clone() for x in M]
    G2 = [g * 3.0 for g in G]
    torch.cuda.synchronize()
    hp = m.MuonHparams()
    ws = m.allocate_workspace(m.muon_workspace_size(shapes, 1 << 34))
    m.muon_step_batched(W2, G2, M2, hp, workspace=ws)
    torch.cuda.synchronize()
    for g in G:
        g.mul_(3.0)                               # the caller's kernel, same stream, no sync
    m.muon_step_batched(W, G, M, hp, workspace=ws)
    torch.cuda.synchronize()
    for a, b in zip(W + M, W2 + M2):
        assert torch.equal(a, b)
