"""Pins of the oracle's Muon optimizer (pimou.com article, sections "优化器的优势" and
"相关技术的追溯": Muon orthogonalizes the update with Newton-Schulz iterations after
Bernstein & Newhouse (2024)).  CPU only.

The iteration is pinned to what the mathematics fixes: its limit is the orthogonal
polar factor U V^T of the SVD (a library routine), each step maps every singular value
s to 1.5 s - 0.5 s^3 with the singular vectors unchanged, and the tall and wide forms
are transposes of each other."""
import numpy as np

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth


def _with_singular_values(m, n, s, seed):
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.standard_normal((m, len(s))))
    V, _ = np.linalg.qr(rng.standard_normal((n, len(s))))
    return (U * s) @ V.T, U, V


def test_newton_schulz_converges_to_the_polar_factor():
    for m, n in ((96, 48), (48, 96), (64, 64)):
        k = min(m, n)
        s = np.linspace(0.5, 1.0, k) * 3.0
        G, U, V = _with_singular_values(m, n, s, m + n)
        X = O.newton_schulz(G, 40)
        assert np.abs(X - U @ V.T).max() < 1e-10
        gram = X.T @ X if m >= n else X @ X.T
        assert np.abs(gram - np.eye(k)).max() < 1e-10


def test_each_step_maps_singular_values_by_the_cubic():
    s = np.array([2.0, 1.0, 0.5, 0.1, 0.01])
    G, U, V = _with_singular_values(40, 30, s, 7)
    for iters in (0, 1, 3, 7):
        x = s / np.sqrt((s * s).sum())                    # Frobenius normalization
        for _ in range(iters):
            x = 1.5 * x - 0.5 * x ** 3
        X = O.newton_schulz(G, iters)
        assert np.abs(X - (U * x) @ V.T).max() < 1e-12, iters


def test_tall_and_wide_forms_agree():
    rng = np.random.default_rng(1)
    G = rng.standard_normal((30, 70))
    assert np.abs(O.newton_schulz(G.T, 6) - O.newton_schulz(G, 6).T).max() < 1e-13
    assert np.array_equal(O.newton_schulz(np.zeros((4, 3)), 5), np.zeros((4, 3)))


def test_muon_step_closed_forms():
    """With zero iterations the direction is the momentum over its Frobenius norm: two
    steps give mom = momentum g1 + g2 and the decoupled decay of the weights."""
    rng = np.random.default_rng(2)
    L, r, c = 2, 12, 8
    p0 = {k: rng.standard_normal((L, r, c)) for k in O.MUON_TENSORS}
    g1 = {k: rng.standard_normal((L, r, c)) for k in O.MUON_TENSORS}
    g2 = {k: rng.standard_normal((L, r, c)) for k in O.MUON_TENSORS}
    p = {k: v.copy() for k, v in p0.items()}
    mom = {k: np.zeros_like(v) for k, v in p0.items()}
    lr, mu, wd = 0.02, 0.9, 0.1
    O.muon_update(p, g1, mom, lr, mu, wd, 0)
    O.muon_update(p, g2, mom, lr, mu, wd, 0)
    for k in O.MUON_TENSORS:
        for l in range(L):
            a = g1[k][l]
            q1 = p0[k][l] - lr * (a / np.linalg.norm(a) + wd * p0[k][l])
            b = mu * a + g2[k][l]
            q2 = q1 - lr * (b / np.linalg.norm(b) + wd * q1)
            assert np.abs(p[k][l] - q2).max() < 1e-13
            assert np.abs(mom[k][l] - b).max() < 1e-13


def test_model_muon_update_leaves_adamw_on_the_other_tensors():
    shape = synth.TINY_HS64
    params = synth.init_params(shape, 0)
    tok, tgt = synth.uniform_tokens(shape.vocab_size, 2, 32, 0)
    a, b = O.from_shape(shape), O.from_shape(shape)
    for o in (a, b):
        o.load(params)
        o.forward(tok, tgt)
        o.zero_grad()
        o.backward()
    a.update_muon(0.02, 0.95, 5, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    b.update(1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    for k in O.PARAM_ORDER:
        if k in O.MUON_TENSORS:
            # a Muon step moves every layer's matrix by lr times an update of spectral
            # norm <= 1 plus the decay
            for l in range(shape.num_layers):
                d = (params[k][l] - a.p[k][l]) / 0.02 - 0.1 * params[k][l]
                assert np.linalg.norm(d, 2) <= 1.0 + 1e-9, k
        else:
            assert np.array_equal(a.p[k], b.p[k]), k


def test_bf16_rounding_against_torch():
    import torch
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000)),
                        [1.0, -1.0, 0.0, 1.00390625, 1.001953125, 3.0 + 2 ** -7]]).astype(np.float32)
    ref = torch.tensor(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(O.round_bf16(x), ref)


def test_bf16_iteration_is_the_exact_one_rounded():
    """With bf16=True the iterate differs from the exact one by rounding only: one step
    from a matrix already on the bf16 grid equals the exact step's products rounded."""
    rng = np.random.default_rng(6)
    G = O.round_bf16(rng.standard_normal((24, 16)))
    X0 = O.round_bf16(G / np.sqrt((G * G).sum()))
    S = O.round_bf16(X0.T @ X0)
    T = O.round_bf16(1.5 * np.eye(16) - 0.5 * S)
    assert np.array_equal(O.newton_schulz(G, 1, bf16=True), O.round_bf16(X0 @ T))
    # and few bf16 steps stay close to the exact iterate
    assert np.abs(O.newton_schulz(G, 3, bf16=True) - O.newton_schulz(G, 3)).max() < 2e-2
