"""Whole-step parity: forward + zero_grad + backward + AdamW through the C ABI against
the CPU oracle on the same seeded weights and tokens.

Bars (the training-step spec): fp32 path -- loss within 1e-5 relative, every gradient
tensor within 1e-3 of the oracle's, max-abs error normalised by the tensor's max
magnitude; bf16 path with fp32 master weights -- loss within 2e-2 absolute.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth
from tests.gpu_helpers import (dev_tokens, ensure_built, gpu_grads_numpy, gpu_model, hp_of, norm_err,
                               run_gpu, run_oracle)

pytestmark = pytest.mark.gpu

LOSS_REL_FP32 = 1e-5
GRAD_NORM_FP32 = 1e-3
LOSS_ABS_BF16 = 2e-2
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    import torch
    torch.cuda.init()


def _grad_errors(g_gpu, g_ref):
    return {k: norm_err(g_gpu[k], g_ref[k]) for k in O.PARAM_ORDER}


def test_tiny_fp32_one_step_matches_oracle():
    """Tiny GPT-2 (L=2, C=64, NH=4, V=512, B=2, T=32), fp32, one step."""
    w = synth.WORKLOADS["tiny_fp32"]
    batches = synth.workload_batches(w)
    hp = hp_of(w)
    m, lg, gg = run_gpu(w.shape, "fp32", w.seed, batches, hp)
    o, lo, go = run_oracle(w.shape, w.seed, batches, hp)
    assert abs(lg[0] - lo[0]) <= LOSS_REL_FP32 * abs(lo[0]), (lg, lo)
    errs = _grad_errors(gg[0], go[0])
    assert max(errs.values()) <= GRAD_NORM_FP32, errs
    assert max(errs.values()) <= 1e-5, errs           # fp32 is far inside the bar
    # after the AdamW step: coordinates with a clear gradient move identically; those whose
    # gradient is at rounding level may step either way (|difference| <= 2 lr)
    pg = {k: v.detach().cpu().numpy().astype(np.float64) for k, v in m.params().items()}
    for k in O.PARAM_ORDER:
        g = go[0][k]
        clear = np.abs(g) > 1e-4 * np.abs(g).max()
        d = np.abs(pg[k] - o.p[k])
        assert d[clear].max(initial=0.0) < 1e-6, k
        assert d.max() <= 2.01 * hp["lr"], k


def test_tiny_padded_vocab_fp32():
    """V=500 padded to 512: pad rows of dwte stay exactly zero; loss/grads match."""
    shape = synth.ModelShape(32, 500, 512, 2, 4, 64)
    batches = [synth.uniform_tokens(500, 2, 32, 5)]
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    m, lg, gg = run_gpu(shape, "fp32", 7, batches, hp)
    o, lo, go = run_oracle(shape, 7, batches, hp)
    assert abs(lg[0] - lo[0]) <= LOSS_REL_FP32 * abs(lo[0])
    assert max(_grad_errors(gg[0], go[0]).values()) <= GRAD_NORM_FP32
    assert np.all(gg[0]["wte"][500:] == 0.0)
    assert np.all(m.params()["wte"][500:].cpu().numpy() == 0.0)


def test_ragged_sequence_and_batch_fp32():
    """T and B smaller than the build maxima, T not a multiple of any tile (T=37, B=3)."""
    shape = synth.ModelShape(64, 512, 512, 2, 4, 64)
    tok, tgt = synth.uniform_tokens(512, 3, 37, 11)
    from step_gpt_train_03_b300.gpt2lib import GPT2
    m = GPT2(shape, 4, 64, "fp32")
    m.load_params(synth.init_params(shape, 3))
    loss = m.forward(dev_tokens(tok), dev_tokens(tgt))
    m.zero_grad()
    m.backward()
    gg = gpu_grads_numpy(m)
    from tests.oracle_helpers import make_oracle
    o = make_oracle(shape, 3)
    lo = o.forward(tok, tgt)
    o.zero_grad()
    o.backward()
    assert abs(loss - lo) <= LOSS_REL_FP32 * lo
    assert max(_grad_errors(gg, o.g).values()) <= GRAD_NORM_FP32


@pytest.mark.slow
def test_gpt2_124m_fp32_each_of_ten_steps_from_the_oracle_state():
    """124M shape, fp32, B=4, T=64, one fixed Zipf batch, Adam 1e-4, 10 steps.  Before
    every step the GPU gets the oracle's current weights and AdamW moments, so each of
    the 10 steps is held to the fp32 bar on its own: loss within 1e-5 relative and every
    gradient within 1e-3 (normalised max-abs)."""
    w = synth.WORKLOADS["gpt2_124m_fp32_b4_t64"]
    batches = synth.workload_batches(w)
    hp = hp_of(w)
    from tests.oracle_helpers import make_oracle
    o = make_oracle(w.shape, w.seed)
    m = gpu_model(w.shape, w.B, w.T, "fp32", w.seed)
    for i, (tok, tgt) in enumerate(batches):
        m.load_state(o.p, o._views(o.m), o._views(o.v))
        lg = m.forward(dev_tokens(tok), dev_tokens(tgt))
        m.zero_grad()
        m.backward()
        gg = gpu_grads_numpy(m)
        lo = o.forward(tok, tgt)
        o.zero_grad()
        o.backward()
        assert abs(lg - lo) <= LOSS_REL_FP32 * abs(lo), (i, lg, lo)
        errs = _grad_errors(gg, o.g)
        assert max(errs.values()) <= GRAD_NORM_FP32, (i, errs)
        o.update(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], i + 1)


@pytest.mark.slow
def test_gpt2_124m_fp32_free_running_ten_steps():
    """The same 10 steps run freely on each side.  Up to step 5 the curves agree to 1e-5
    relative.  At step 6 this workload's loss jumps (10.57 after 7.08) and Adam amplifies
    rounding differences: two independent fp32 programs (PyTorch's layers with
    torch.optim.AdamW and the fp32 oracle) already differ by 4.7e-5 relative at step 9.
    From step 6 on the bound is therefore 1e-3 relative, the spread that jump allows."""
    w = synth.WORKLOADS["gpt2_124m_fp32_b4_t64"]
    batches = synth.workload_batches(w)
    hp = hp_of(w)
    _, lg, gg = run_gpu(w.shape, "fp32", w.seed, batches, hp)
    _, lo, go = run_oracle(w.shape, w.seed, batches, hp)
    errs = _grad_errors(gg[0], go[0])
    assert max(errs.values()) <= GRAD_NORM_FP32, errs
    rel = [abs(a - b) / abs(b) for a, b in zip(lg, lo)]
    assert max(rel[:6]) <= LOSS_REL_FP32, (rel, lg, lo)
    assert max(rel) <= 1e-3, (rel, lg, lo)


def test_bf16_tiny_ten_steps():
    """bf16 activations/weights with fp32 master weights and AdamW state, tiny model with
    one head of size 64 (the tensor-core attention's head size)."""
    shape = synth.TINY_HS64
    batches = synth.workload_batches(synth.WORKLOADS["tiny_fp32"], 10)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    _, lg, _ = run_gpu(shape, "bf16", 0, batches, hp)
    _, lo, _ = run_oracle(shape, 0, batches, hp)
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS_BF16, (lg, lo)


@pytest.mark.slow
def test_bf16_gpt2_124m_short_sequences_ten_steps():
    """124M shape in bf16 (B=2, T=128, fresh Zipf batches, lr 6e-4, wd 0.1) vs the oracle."""
    shape = synth.GPT2_124M
    batches = synth.zipf_batches(50257, 2, 128, 10, 21)
    hp = dict(lr=6e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    _, lg, gg = run_gpu(shape, "bf16", 2, batches, hp)
    _, lo, go = run_oracle(shape, 2, batches, hp, np.float32)
    assert max(abs(a - b) for a, b in zip(lg, lo)) <= LOSS_ABS_BF16, (lg, lo)
    # bf16 gradients against the fp32 oracle: each stored activation and activation
    # gradient is rounded to bf16 (relative 2^-9 = 2e-3), and the backward chains about
    # ten such roundings per layer through 12 layers; on this workload every tensor's
    # normalised error measured <= 9.7e-3 (ln1w; most 5e-3..7e-3) on a B300.  The bound
    # 2e-2 keeps a factor 2 over that; a dropped term or a wrong constant is O(0.1..1).
    errs = _grad_errors(gg[0], go[0])
    assert max(errs.values()) < 2e-2, errs


def _golden(name):
    p = os.path.join(GOLDEN, f"{name}_oracle_losses.json")
    if not os.path.exists(p):
        pytest.skip(f"no stored oracle curve for {name}")
    with open(p) as f:
        return json.load(f)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gpt2_124m_bf16_b16_t1024", "gpt2_350m_bf16_b8_t1024"])
def test_bf16_full_size_ten_steps_against_stored_oracle_curve(name):
    """Full-size bf16 workloads: 10 steps on fresh Zipf batches; every step's loss and the
    loss after the 10th update within 2e-2 of the fp32 oracle's stored curve."""
    g = _golden(name)
    w = synth.WORKLOADS[name]
    n = g["steps"]
    batches = synth.workload_batches(w, n + 1)
    hp = hp_of(w)
    m = gpu_model(w.shape, w.B, w.T, "bf16", w.seed)
    losses = []
    for i in range(n):
        losses.append(m.step(dev_tokens(batches[i][0]), dev_tokens(batches[i][1]), hp["lr"], hp["beta1"],
                             hp["beta2"], hp["eps"], hp["weight_decay"], i + 1))
    final = m.forward(dev_tokens(batches[n][0]), dev_tokens(batches[n][1]))
    diffs = [abs(a - b) for a, b in zip(losses + [final], g["losses"] + [g["loss_after_updates"]])]
    assert max(diffs) <= LOSS_ABS_BF16, (losses, final, g)


@pytest.mark.slow
def test_bf16_full_size_per_position_losses_sampled_rows():
    """124M, B=16, T=1024 bf16 forward: the per-position losses of sampled batch rows
    agree with the oracle run on those rows alone (each row is an independent sequence)."""
    w = synth.WORKLOADS["gpt2_124m_bf16_b16_t1024"]
    tok, tgt = synth.workload_batches(w, 1)[0]
    m = gpu_model(w.shape, w.B, w.T, "bf16", w.seed)
    m.forward(dev_tokens(tok), dev_tokens(tgt))
    per_pos = m.losses(w.B * w.T).cpu().numpy().reshape(w.B, w.T)
    from tests.oracle_helpers import make_oracle
    o = make_oracle(w.shape, w.seed, np.float32)
    o.keep_preatt = False
    for b in (0, 7, 15):
        o.forward(tok[b:b + 1], tgt[b:b + 1])
        ref = o.acts["losses"][0]
        assert np.abs(per_pos[b] - ref).max() <= LOSS_ABS_BF16 * 2.5, b
        assert abs(per_pos[b].mean() - ref.mean()) <= LOSS_ABS_BF16, b


def test_steps_are_bitwise_deterministic():
    """Two runs from the same state give bit-identical gradients (no float atomics)."""
    import torch
    for precision in ("fp32", "bf16"):
        shape = synth.ModelShape(64, 512, 512, 2, 4 if precision == "fp32" else 1, 64)
        tok, tgt = synth.zipf_batches(512, 4, 64, 1, 4)[0]
        out = []
        for _ in range(2):
            m = gpu_model(shape, 4, 64, precision, 1)
            m.forward(dev_tokens(tok), dev_tokens(tgt))
            m.zero_grad()
            m.backward()
            out.append(m.flat_grads().clone())
        assert torch.equal(out[0], out[1]), precision


@pytest.mark.parametrize("precision", ["bf16", "fp8"])
def test_fused_step_stores_every_gradient(precision):
    """gpt2_step does not clear the gradients: in its backward each gradient's first
    writer stores instead of adding, and what no writer covers (the position rows past
    T, alignment gaps) is cleared.  From a gradient buffer full of NaN, the fused step's
    gradients -- eager, graph-capturing and graph-replayed calls -- equal those of
    zero_grad + backward element for element, at a T shorter than the model's."""
    import torch
    shape = synth.TINY_HS64
    tok, tgt = synth.uniform_tokens(shape.vocab_size, 2, 24, 5)
    ref = gpu_model(shape, 2, 32, precision, 3)
    ref.forward(dev_tokens(tok), dev_tokens(tgt))
    ref.zero_grad()
    ref.backward()
    g_ref = ref.flat_grads().clone()
    m = gpu_model(shape, 2, 32, precision, 3)
    for call in range(3):
        m.flat_grads().fill_(float("nan"))
        m.step_device(dev_tokens(tok), dev_tokens(tgt), 0.0, 0.9, 0.999, 1e-8, 0.0, call + 1)
        torch.cuda.synchronize()
        g = m.flat_grads()
        assert torch.equal(g, g_ref), (call, int(torch.isnan(g).sum()), float((g - g_ref).abs().nan_to_num(1e9).max()))


def test_errors_are_reported_not_faulted():
    from step_gpt_train_03_b300.gpt2lib import GPT2Error
    shape = synth.TINY
    m = gpu_model(shape, 2, 32, "fp32", 0)
    tok, tgt = synth.uniform_tokens(512, 2, 32, 0)
    with pytest.raises(GPT2Error) as e:
        m.backward()                                   # no forward yet
    assert e.value.status == 2
    bad = tok.copy()
    bad[1, 5] = 512                                    # id == V
    with pytest.raises(GPT2Error) as e:
        m.forward(dev_tokens(bad), dev_tokens(tgt))
    assert e.value.status == 4
    with pytest.raises(GPT2Error) as e:
        m.forward(dev_tokens(np.zeros((3, 32), np.int32)), dev_tokens(np.zeros((3, 32), np.int32)))
    assert e.value.status == 1                         # B > max_B
    # the context is still usable
    loss = m.forward(dev_tokens(tok), dev_tokens(tgt))
    assert math.isfinite(loss)
    # a non-finite weight gives a non-finite loss, reported as such
    m.params()["lnfw"][3] = float("nan")
    m.sync_params()
    with pytest.raises(GPT2Error) as e:
        m.forward(dev_tokens(tok), dev_tokens(tgt))
    assert e.value.status == 5


def test_step_from_host_buffers_matches_device_path():
    import torch
    w = synth.WORKLOADS["tiny_fp32"]
    tok, tgt = synth.workload_batches(w)[0]
    hp = hp_of(w)
    a = gpu_model(w.shape, 2, 32, "fp32", 0)
    la = a.step(dev_tokens(tok), dev_tokens(tgt), hp["lr"], hp["beta1"], hp["beta2"], hp["eps"],
                hp["weight_decay"], 1)
    b = gpu_model(w.shape, 2, 32, "fp32", 0)
    th = torch.as_tensor(tok).pin_memory()
    gh = torch.as_tensor(tgt).pin_memory()
    lb = b.step_host(th, gh, hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], 1)
    assert la == lb
    assert torch.equal(a.flat_params(), b.flat_params())


@pytest.mark.parametrize("precision", ["bf16", "fp32"])
def test_graph_steps_match_eager_steps_bitwise(precision):
    """gpt2_step replays one captured CUDA graph per (B, T) from its third step of that
    shape; every step (learning rate changing each time, a batch-size change in the
    middle forcing a new capture) equals the kernel-by-kernel step bit for bit."""
    import torch
    shape = synth.ModelShape(64, 512, 512, 2, 4 if precision == "fp32" else 1, 64)
    batches = synth.zipf_batches(512, 4, 64, 9, 11)
    g = gpu_model(shape, 4, 64, precision, 3)
    e = gpu_model(shape, 4, 64, precision, 3)
    e.set_graphs(False)
    for i, (tok, tgt) in enumerate(batches):
        Bi = 4 if i < 5 else 2                          # shape change at step 5
        tk, tg = dev_tokens(tok[:Bi]), dev_tokens(tgt[:Bi])
        lr = 1e-3 * (1 + 0.1 * i)
        lg = g.step_device(tk, tg, lr, 0.9, 0.95, 1e-8, 0.1, i + 1, want_loss=True)
        le = e.step_device(tk, tg, lr, 0.9, 0.95, 1e-8, 0.1, i + 1, want_loss=True)
        assert lg == le, (i, lg, le)
        assert torch.equal(g.flat_params(), e.flat_params()), i


def test_split_weight_gradients_are_bitwise_deterministic():
    """At the 124M shape with B*T = 1024 rows, the weight-gradient products of the fc and
    attention layers split their 1024-row contraction; the splits add into the gradient
    in a fixed order, so two runs from the same state agree bit for bit."""
    import torch
    shape = synth.GPT2_124M
    tok, tgt = synth.zipf_batches(shape.vocab_size, 2, 512, 1, 5)[0]
    out = []
    for _ in range(2):
        m = gpu_model(shape, 2, 512, "bf16", 1)
        m.forward(dev_tokens(tok), dev_tokens(tgt))
        m.zero_grad()
        m.backward()
        out.append(m.flat_grads().clone())
    assert torch.equal(out[0], out[1])
