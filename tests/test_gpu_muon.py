"""The Muon optimizer (pimou.com article, sections "优化器的优势" and "相关技术的追溯":
Newton-Schulz orthogonalization, after Bernstein & Newhouse 2024) through the C ABI
against the oracle.

The iteration runs in bf16 on the tensor cores (fp32 accumulation): it stores X, the
Gram matrix S and T = 1.5 I - 0.5 S in bf16.  Against the oracle's iteration with the
same three roundings (bf16=True) what remains is the fp32 accumulation order, which can
move a stored value to its neighbouring bf16 number (2^-8 relative); the step maps a
singular value s to 1.5 s - 0.5 s^3, whose slope is at most 1.5, so such a difference can
grow by up to 1.5 per remaining step in the directions of small singular values: the
bound after k steps is 2^-8 * 1.5^k (measured 0.6e-3, 1.1e-2, 4.6e-2 and 8.2e-2 at 0, 5,
8 and 12 steps on gradient-like matrices).  Where the iteration has converged it
contracts instead: on a well-conditioned matrix 15 steps must reach the orthogonal
polar factor U V^T of the SVD at bf16 accuracy, whatever the rounding order."""
import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import dev_tokens, ensure_built, gpu_model, norm_err

pytestmark = pytest.mark.gpu

NS_EXACT_TOL_5 = 4e-2      # against the exact iterate, 5 steps
POLAR_TOL = 4e-2           # converged iterate against the SVD polar factor (see below)


def ns_tol(k):
    """Against the bf16-rounding oracle after k steps (see the module notes)."""
    return 2.0 ** -8 * 1.5 ** k
LOSS_ABS = 2e-2


@pytest.fixture(scope="module")
def G():
    ensure_built()
    import torch
    from step_gpt_train_03_b300 import gpt2lib
    torch.cuda.init()
    return gpt2lib


@pytest.mark.parametrize("r,c,iters", [(2304, 768, 5), (768, 768, 5), (3072, 768, 8), (768, 3072, 5),
                                       (64, 192, 12), (200, 64, 0), (768, 768, 12)])
def test_newton_schulz_against_oracle(G, r, c, iters):
    import torch
    rng = np.random.default_rng(r + c + iters)
    # a gradient-like matrix: a few strong directions over a noise floor
    g = rng.standard_normal((r, c)) * 0.1 + rng.standard_normal((r, 4)) @ rng.standard_normal((4, c))
    g = g.astype(np.float32)
    out = torch.empty((r, c), dtype=torch.bfloat16, device="cuda")
    G.newton_schulz(out, torch.as_tensor(g).cuda(), iters)
    G.layer_check()
    got = out.float().cpu().numpy()
    e = norm_err(got, O.newton_schulz(g.astype(np.float64), iters, bf16=True))
    assert e <= ns_tol(iters), e
    if iters <= 5:
        e = norm_err(got, O.newton_schulz(g.astype(np.float64), iters))
        assert e <= NS_EXACT_TOL_5, e


@pytest.mark.parametrize("r,c", [(2304, 768), (768, 3072), (768, 768)])
def test_newton_schulz_reaches_the_polar_factor(G, r, c):
    """Singular values spread over [0.3, 1] times a scale: 15 steps converge (exactly,
    every s within 1e-6 of 1), and the bf16 iterate must equal U V^T of the SVD.  At the
    fixed point a bf16 iteration still rounds T = 1.5 I - 0.5 X^T X ~ I, whose entries near
    1 have a spacing of 2^-8, into X every step: the bf16-rounding oracle sits at
    1.7-1.8e-2 of U V^T on these matrices, hence the bound 4e-2."""
    import torch
    rng = np.random.default_rng(r * c)
    k = min(r, c)
    U, _ = np.linalg.qr(rng.standard_normal((r, k)))
    V, _ = np.linalg.qr(rng.standard_normal((c, k)))
    g = ((U * np.linspace(0.3, 1.0, k) * 5.0) @ V.T).astype(np.float32)
    out = torch.empty((r, c), dtype=torch.bfloat16, device="cuda")
    G.newton_schulz(out, torch.as_tensor(g).cuda(), 15)
    G.layer_check()
    Uf, _, Vt = np.linalg.svd(g.astype(np.float64), full_matrices=False)
    got = out.float().cpu().numpy()
    e = norm_err(got, Uf @ Vt)
    assert e <= POLAR_TOL, e
    # converged, the iteration contracts: the rounding-order difference to the
    # bf16-rounding oracle stays at the level of a single step (measured 0.6-1.0e-2)
    e = norm_err(got, O.newton_schulz(g.astype(np.float64), 15, bf16=True))
    assert e <= 2e-2, e


def _muon_run(shape, B, T, batches, hp, precision="bf16"):
    m = gpu_model(shape, B, T, precision, 0)
    o = O.from_shape(shape, np.float64)
    o.load(synth.init_params(shape, 0))
    lg, lo = [], []
    for i, (tok, tgt) in enumerate(batches):
        lg.append(m.forward(dev_tokens(tok), dev_tokens(tgt)))
        m.zero_grad()
        m.backward()
        m.update_muon(hp["lr_muon"], hp["mu"], hp["iters"], hp["lr"], 0.9, 0.95, 1e-8, hp["wd"], i + 1)
        lo.append(o.forward(tok, tgt))
        o.zero_grad()
        o.backward()
        o.update_muon(hp["lr_muon"], hp["mu"], hp["iters"], hp["lr"], 0.9, 0.95, 1e-8, hp["wd"], i + 1)
    return m, o, lg, lo


def test_muon_tiny_model_steps(G):
    """Tiny model (one head of 64), 8 steps of Muon + AdamW: losses track the oracle's, and
    after the first step every block matrix moved as the oracle's did."""
    shape = synth.TINY_HS64
    batches = synth.workload_batches(synth.WORKLOADS["tiny_fp32"], 8)
    hp = dict(lr_muon=0.02, mu=0.95, iters=5, lr=1e-3, wd=0.01)
    p0 = synth.init_params(shape, 0)
    m, o, lg, lo = _muon_run(shape, 2, 32, batches[:1], hp)
    P = {k: v.detach().cpu().numpy().astype(np.float64) for k, v in m.params().items()}
    for k in O.MUON_TENSORS:
        e = norm_err(P[k] - p0[k], o.p[k] - p0[k])
        assert e <= NS_EXACT_TOL_5, (k, e)
    _, _, lg, lo = _muon_run(shape, 2, 32, batches, hp)
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS, (lg, lo)


@pytest.mark.slow
def test_muon_gpt2_124m_short_sequences(G):
    shape = synth.GPT2_124M
    batches = synth.zipf_batches(50257, 2, 128, 5, 21)
    hp = dict(lr_muon=0.02, mu=0.95, iters=5, lr=6e-4, wd=0.0)
    _, _, lg, lo = _muon_run(shape, 2, 128, batches, hp)
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS, (lg, lo)


@pytest.mark.parametrize("shape", [synth.TINY_HS64, synth.ModelShape(64, 512, 512, 2, 4, 256)],
                         ids=["layer-by-layer", "batched"])
def test_muon_graph_steps_match_eager_steps_bitwise(G, shape):
    """gpt2_step_muon replays one captured CUDA graph (forward, backward, Muon + AdamW)
    per shape and Muon constants; every step -- the AdamW learning rate changing each
    time, a Muon momentum change in the middle forcing a new capture -- equals the
    kernel-by-kernel step bit for bit.  The C = 256 shape takes the batched Newton-Schulz
    products (all matrix sides multiples of 256), the tiny one the layer-by-layer path."""
    import torch
    batches = synth.zipf_batches(shape.vocab_size, 2, 32, 8, 13)
    g = gpu_model(shape, 2, 32, "bf16", 4)
    e = gpu_model(shape, 2, 32, "bf16", 4)
    e.set_graphs(False)
    for i, (tok, tgt) in enumerate(batches):
        tk, tg = dev_tokens(tok), dev_tokens(tgt)
        lr, mom = 1e-3 * (1 + 0.1 * i), (0.95 if i < 4 else 0.9)
        lg = g.step_muon_device(tk, tg, 0.02, mom, 5, lr, 0.9, 0.95, 1e-8, 0.1, i + 1, want_loss=True)
        le = e.step_muon_device(tk, tg, 0.02, mom, 5, lr, 0.9, 0.95, 1e-8, 0.1, i + 1, want_loss=True)
        assert lg == le, (i, lg, le)
        assert torch.equal(g.flat_params(), e.flat_params()), i
