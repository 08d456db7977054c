"""MuonAdamW, the torch.optim.Optimizer over the library, against the oracle.

The pages' interface is ``optimizer.zero_grad(); optimizer.step()``;
"LLM training series, part 2: optimizers" (section 4.3) puts the hidden
matrices under Muon and the rest under AdamW, and section 5.3 warns that
resuming without the optimizer state is not resuming.  Checked here: two
steps of both parts against the oracle (momentum and AdamW state bit-exact,
the Muon update within 1e-2), and a save / load round trip that continues
bit for bit like an uninterrupted run.
"""
import numpy as np
import pytest
import torch

import oracle
import optimizer_muon_step_gb300 as m

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = 1e-2
MUON_SHAPES = [(256, 512), (512, 256), (130, 70)]
ADAMW_SHAPES = [(1000, 64), (64,), (7,)]   # embedding-like, a norm gain, a bias


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)


def make_params(seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    mu = [torch.nn.Parameter(torch.randn(*s, device=DEV, generator=gen) * 0.02) for s in MUON_SHAPES]
    ad = [torch.nn.Parameter(torch.randn(*s, device=DEV, generator=gen) * 0.02) for s in ADAMW_SHAPES]
    return mu, ad


def set_grads(params, seed):
    gen = torch.Generator(device=DEV).manual_seed(seed)
    for p in params:
        p.grad = torch.randn(p.shape, device=DEV, generator=gen) * 1e-2


def test_two_steps_match_the_oracle(lib):
    mu, ad = make_params(91)
    muon_hp, adamw_hp = m.MuonHparams(), m.AdamwHparams(lr=1e-3)
    opt = m.MuonAdamW(mu, ad, muon_hp, adamw_hp)
    mcfg = oracle.MuonConfig()
    acfg = oracle.AdamwConfig(lr=1e-3)
    Mh = [np.zeros(s, np.float32) for s in MUON_SHAPES]
    mh = [np.zeros(s, np.float32).reshape(-1) for s in ADAMW_SHAPES]
    vh = [np.zeros(s, np.float32).reshape(-1) for s in ADAMW_SHAPES]
    for t in (1, 2):
        set_grads(mu + ad, seed=100 + t)
        W0 = [p.detach().cpu().numpy() for p in mu]
        G0 = [p.grad.cpu().numpy() for p in mu]
        P0 = [p.detach().cpu().numpy().reshape(-1) for p in ad]
        g0 = [p.grad.cpu().numpy().reshape(-1) for p in ad]
        opt.step()
        opt.zero_grad()
        for i, p in enumerate(mu):
            oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0[i], Mh[i], mcfg)
            assert np.array_equal(opt.state[p]["momentum_buffer"].cpu().numpy(), oM)
            dW = p.detach().cpu().numpy().astype(np.float64) - W0[i]
            assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL
            Mh[i] = oM
        for i, p in enumerate(ad):
            rp, rm, rv = oracle.adamw_step(P0[i], g0[i], mh[i], vh[i], acfg, t=t)
            assert np.array_equal(p.detach().cpu().numpy().reshape(-1), rp)
            assert opt.state[p]["step"] == t
            mh[i], vh[i] = rm, rv


def test_state_dict_round_trip_resumes_bit_for_bit(lib, tmp_path):
    mu, ad = make_params(92)
    mu2 = [torch.nn.Parameter(p.detach().clone()) for p in mu]
    ad2 = [torch.nn.Parameter(p.detach().clone()) for p in ad]
    straight = m.MuonAdamW(mu, ad)
    first = m.MuonAdamW(mu2, ad2)
    set_grads(mu + ad, seed=201)
    set_grads(mu2 + ad2, seed=201)
    straight.step()
    first.step()
    path = tmp_path / "opt.pt"
    torch.save(first.state_dict(), path)
    resumed = m.MuonAdamW(mu2, ad2)        # a fresh optimizer, as after a restart
    resumed.load_state_dict(torch.load(path))
    set_grads(mu + ad, seed=202)
    set_grads(mu2 + ad2, seed=202)
    straight.step()
    resumed.step()
    for a, b in zip(mu + ad, mu2 + ad2):
        assert torch.equal(a.detach(), b.detach())


def test_rejected_adamw_step_leaves_the_state_alone(lib):
    """A step the library refuses (here a NaN learning rate set through the
    param group) raises before anything is enqueued and changes no state:
    step counts, m, v and the parameters stay as they were, so a retry with
    a valid lr applies the right bias correction (checked against the
    oracle's second step).  torch itself refuses a .grad whose dtype, shape
    or device differs from its fp32 parameter's, so the optimizer's own
    gradient checks are a second line behind that."""
    _, ad = make_params(94)
    opt = m.MuonAdamW([], ad, adamw_hp=m.AdamwHparams(lr=1e-3))
    set_grads(ad, seed=401)
    opt.step()
    before = {p: (opt.state[p]["step"], opt.state[p]["exp_avg"].clone(), opt.state[p]["exp_avg_sq"].clone())
              for p in ad}
    set_grads(ad, seed=402)
    P0 = [p.detach().clone() for p in ad]
    opt.param_groups[0]["lr"] = float("nan")
    with pytest.raises(m.MuonError):
        opt.step()
    for p, p0 in zip(ad, P0):
        assert opt.state[p]["step"] == before[p][0] == 1
        assert torch.equal(opt.state[p]["exp_avg"], before[p][1])
        assert torch.equal(opt.state[p]["exp_avg_sq"], before[p][2])
        assert torch.equal(p.detach(), p0)
    opt.param_groups[0]["lr"] = 1e-3
    host = [(p.detach().cpu().numpy().reshape(-1), p.grad.cpu().numpy().reshape(-1),
             before[p][1].cpu().numpy().reshape(-1), before[p][2].cpu().numpy().reshape(-1)) for p in ad]
    opt.step()
    for p, (p0, g0, m0, v0) in zip(ad, host):
        rp, _, _ = oracle.adamw_step(p0, g0, m0, v0, oracle.AdamwConfig(lr=1e-3), t=2)
        assert np.array_equal(p.detach().cpu().numpy().reshape(-1), rp)
        assert opt.state[p]["step"] == 2


def test_muon_gradient_layouts_and_a_skipped_parameter(lib):
    """A gradient given as a transposed view (strided; made contiguous
    before the call), and a parameter without a gradient on one step: it is
    skipped with its momentum kept, and on the next step continues from that
    momentum.  All against the oracle.  (fp16 and bf16 gradients reach the
    library through muon_step_batched, covered in test_gpu_fp16.py; torch
    does not let them onto an fp32 parameter's .grad.)"""
    mu, _ = make_params(95)
    opt = m.MuonAdamW(mu, [])
    cfg = oracle.MuonConfig()
    Mh = [np.zeros(s, np.float32) for s in MUON_SHAPES]
    gen = torch.Generator(device=DEV).manual_seed(501)
    for t in range(3):
        grads = []
        for i, (r, c) in enumerate(MUON_SHAPES):
            g = torch.randn(c, r, device=DEV, generator=gen).t() * 1e-2    # a transposed view
            grads.append(g)
        skip = 2 if t == 1 else None                                       # no gradient on step 1
        for i, p in enumerate(mu):
            p.grad = None if i == skip else grads[i]
        assert not grads[0].is_contiguous()
        W0 = [p.detach().cpu().numpy() for p in mu]
        M_before = [opt.state[p]["momentum_buffer"].clone() if p in opt.state else None for p in mu]
        opt.step()
        for i, p in enumerate(mu):
            if i == skip:
                assert np.array_equal(p.detach().cpu().numpy(), W0[i])
                assert torch.equal(opt.state[p]["momentum_buffer"], M_before[i])
                continue
            G0 = grads[i].float().cpu().numpy()
            oW, oM, _, _ = oracle.muon_step_matrix(W0[i], G0, Mh[i], cfg)
            assert np.array_equal(opt.state[p]["momentum_buffer"].cpu().numpy(), oM), (t, i)
            dW = p.detach().cpu().numpy().astype(np.float64) - W0[i]
            assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL, (t, i)
            Mh[i] = oM


def test_lr_scheduler_drives_both_parts(lib):
    """lr lives in the param groups, so a torch scheduler sets it: after one
    LambdaLR step (factor 0.5) the second step uses half of each part's lr."""
    mu, ad = make_params(93)
    opt = m.MuonAdamW(mu, ad, m.MuonHparams(lr=0.02), m.AdamwHparams(lr=1e-3))
    sched = torch.optim.lr_scheduler.LambdaLR(opt, lambda k: 0.5 ** k)
    set_grads(mu + ad, seed=301)
    opt.step()
    sched.step()
    assert [g["lr"] for g in opt.param_groups] == [0.01, 5e-4]
    M1 = [opt.state[p]["momentum_buffer"].cpu().numpy() for p in mu]
    st = [(opt.state[p]["exp_avg"].cpu().numpy().reshape(-1), opt.state[p]["exp_avg_sq"].cpu().numpy().reshape(-1))
          for p in ad]
    set_grads(mu + ad, seed=302)
    W0 = [p.detach().cpu().numpy() for p in mu]
    G0 = [p.grad.cpu().numpy() for p in mu]
    P0 = [p.detach().cpu().numpy().reshape(-1) for p in ad]
    g0 = [p.grad.cpu().numpy().reshape(-1) for p in ad]
    opt.step()
    for i, p in enumerate(mu):
        oW, _, _, _ = oracle.muon_step_matrix(W0[i], G0[i], M1[i], oracle.MuonConfig(lr=0.01))
        dW = p.detach().cpu().numpy().astype(np.float64) - W0[i]
        assert rel_fro(dW, oW.astype(np.float64) - W0[i]) < TOL
    for i, p in enumerate(ad):
        rp, _, _ = oracle.adamw_step(P0[i], g0[i], st[i][0], st[i][1], oracle.AdamwConfig(lr=5e-4), t=2)
        assert np.array_equal(p.detach().cpu().numpy().reshape(-1), rp)
