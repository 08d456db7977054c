"""Multi-tensor AdamW (adamw_step_batched) against the oracle.

Everything Muon does not take -- embedding, LM head, norm gains and biases
("LLM training series, part 2: optimizers", section 4.3) -- goes to AdamW:
a few large tensors and many small ones.  One launch per 448 tensors must
update every tensor exactly as the oracle does (bit for bit, as the
single-tensor kernel does), whatever the sizes, alignments and empty
tensors in the list.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"


def make_tensors(sizes, seed, offsets):
    """(p, g, m, v) per size; offset 1 starts the views 4 bytes into their
    buffers (the scalar path); v is nonnegative."""
    gen = torch.Generator(device=DEV).manual_seed(seed)
    out = []
    for n, off in zip(sizes, offsets):
        bufs = [torch.randn(n + off, device=DEV, generator=gen) * s for s in (0.02, 1e-3, 1e-3, 1e-3)]
        p, g, mm, v = (b[off:] for b in bufs)
        v.abs_().mul_(1e-3)
        out.append((p, g, mm, v))
    return out


def check_against_oracle(tensors, host, hp, step):
    cfg = oracle.AdamwConfig(lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps, weight_decay=hp.weight_decay)
    for i, ((p, g, mm, v), h) in enumerate(zip(tensors, host)):
        if p.numel() == 0:
            continue
        rp, rm, rv = oracle.adamw_step(*h, cfg, t=step)
        assert np.array_equal(p.cpu().numpy(), rp), i
        assert np.array_equal(mm.cpu().numpy(), rm), i
        assert np.array_equal(v.cpu().numpy(), rv), i


def test_many_tensors_bit_exact(lib):
    rng = np.random.default_rng(81)
    sizes = [int(x) for x in rng.integers(0, 5000, size=300)] + [0, 1, 3, (1 << 20) + 5, 3 * 16384]
    offsets = [int(x) for x in rng.integers(0, 2, size=len(sizes))]
    tensors = make_tensors(sizes, seed=81, offsets=offsets)
    host = [[x.cpu().numpy() for x in quad] for quad in tensors]
    hp = m.AdamwHparams()
    m.adamw_step_batched(tensors, hp, step=100)
    check_against_oracle(tensors, host, hp, 100)


def test_batched_equals_single_tensor_calls_and_launch_count(lib):
    sizes = [7 + (i % 97) * 13 for i in range(1000)]          # 1000 tensors: three launches
    tensors = make_tensors(sizes, seed=82, offsets=[i % 2 for i in range(1000)])
    twins = [tuple(x.clone() for x in quad) for quad in tensors]
    hp = m.AdamwHparams(lr=1e-3, weight_decay=0.05)
    n0 = m.muon_launch_count()
    m.adamw_step_batched(tensors, hp, step=3)
    assert m.muon_launch_count() - n0 == 3
    for quad in twins:
        m.adamw_step(*quad, hp, step=3)
    torch.cuda.synchronize()
    for a, b in zip(tensors, twins):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_overlapping_tensors_are_rejected(lib):
    buf = torch.zeros(4 * 1000, device=DEV)
    p, g, mm, v = (buf[k * 1000:(k + 1) * 1000] for k in range(4))
    other = make_tensors([500], seed=83, offsets=[0])[0]
    with pytest.raises(m.MuonError):   # the second tensor's p lies inside the first one's m
        m.adamw_step_batched([(p, g, mm, v), (buf[2100:2600], other[1], other[2], other[3])])
