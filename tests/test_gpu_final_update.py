"""The final update W = W - lr (wd W + scale O) writes every element of every
W and nothing else.

The update kernels take W in the caller's layout: flat tiles for wide
matrices, 64x64 tiles transposed through shared memory for tall ones, with
bounds checks at every ragged edge.  These tests place every W inside one
shared buffer, at offsets that break 16-byte alignment (the scalar paths),
with guard gaps filled with a sentinel, and check after one step from
W = 0 that:

  * every element of every W is nonzero (no element was missed);
  * every guard element is unchanged (nothing was written past a row or
    past a matrix);
  * W and M agree with the oracle (tolerances as in test_gpu_kernels.py).

The shapes cover wide and tall matrices on both NS kernels (CTA pairs for
256-row-aligned or lightly padded groups above 512 rows, single CTAs
otherwise) with row
and column counts that are not multiples of 32, 64, 128 or 256, after five
NS steps and after none.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2
GUARD = 37          # floats between matrices (odd: W starts are only 4-byte aligned)
SENTINEL = 12345.0


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def cfg_of(hp):
    return oracle.MuonConfig(lr=hp.lr, weight_decay=hp.weight_decay, momentum=hp.momentum,
                             nesterov=hp.nesterov, ns_steps=hp.ns_steps, ns_a=hp.ns_a, ns_b=hp.ns_b,
                             ns_c=hp.ns_c, norm_eps=hp.norm_eps, rms_scale=hp.rms_scale,
                             scale_mode=hp.scale_mode, skip_nonfinite=hp.skip_nonfinite,
                             max_grad_norm=hp.max_grad_norm, ns_coeffs=hp.ns_coeffs)


def packed_weights(shapes):
    """Zero W views inside one buffer, GUARD sentinel floats before, between
    and after.  From W = 0 the update is -lr * scale * O, which is nonzero
    wherever O is (a bf16 O of exactly 0 would take an fp32 value below
    1e-40), so an element left at 0 is one the update missed."""
    total = GUARD + sum(r * c + GUARD for r, c in shapes)
    buf = torch.full((total,), SENTINEL, device=DEV)
    views, off = [], GUARD
    for r, c in shapes:
        v = buf[off:off + r * c].view(r, c)
        v.zero_()
        views.append(v)
        off += r * c + GUARD
    return buf, views


def guard_mask(shapes):
    total = GUARD + sum(r * c + GUARD for r, c in shapes)
    mask = torch.ones(total, dtype=torch.bool, device=DEV)
    off = GUARD
    for r, c in shapes:
        mask[off:off + r * c] = False
        off += r * c + GUARD
    return mask


CASES = {
    # CTA pairs: m' above 512, a multiple of 256 or with at most 1/8 padding
    "pairs": [(768, 1000), (1000, 768), (1024, 1090), (1090, 1024)],
    # single CTAs: m' with more than 1/8 pair padding; ragged everywhere
    "singles": [(130, 70), (70, 130), (300, 333), (333, 300), (33, 1000), (1000, 33)],
    "mixed": [(256, 512), (200, 328), (640, 1000), (1000, 640), (7, 13)],
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("ns_steps", [5, 0])
def test_final_update_covers_every_element_and_nothing_else(lib, case, ns_steps):
    shapes = CASES[case]
    gen = torch.Generator(device=DEV).manual_seed(41 + len(shapes))
    buf, W = packed_weights(shapes)
    G = [(torch.randn(r, c, device=DEV, generator=gen) * 1e-2).to(
        torch.bfloat16 if i % 2 else torch.float32) for i, (r, c) in enumerate(shapes)]
    M = [torch.randn(r, c, device=DEV, generator=gen) * 1e-2 for r, c in shapes]
    W0 = [w.cpu().numpy().copy() for w in W]
    G0 = [g.float().cpu().numpy() for g in G]
    M0 = [x.cpu().numpy() for x in M]
    hp = m.MuonHparams(lr=0.02, weight_decay=0.1, ns_steps=ns_steps)
    m.muon_step_batched(W, G, M, hp)
    torch.cuda.synchronize()
    mask = guard_mask(shapes)
    assert bool((buf[mask] == SENTINEL).all()), "a guard element was written"
    cfg = cfg_of(hp)
    for i, (r, c) in enumerate(shapes):
        got = W[i].cpu().numpy()
        assert (got != 0).all(), f"matrix {i} ({r}x{c}): an element was not updated"
        oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M0[i], cfg)
        assert np.array_equal(M[i].cpu().numpy(), oM)
        assert rel_fro(got.astype(np.float64) - W0[i], oW.astype(np.float64) - W0[i]) < TOL
