"""Helpers for the GPU parity tests: run the CUDA library and the oracle on the same
seeded inputs and compare."""
from __future__ import annotations

import numpy as np

from step_gpt_train_03_b300 import synth


def ensure_built():
    from step_gpt_train_03_b300 import build
    build.build()


def dev_tokens(a):
    import torch
    return torch.as_tensor(np.ascontiguousarray(a, np.int32)).cuda()


def norm_err(got, ref):
    """max |got - ref| / max |ref| (the parity measure for tensors)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (d if d > 0 else 1.0))


def gpu_model(shape, B, T, precision, seed):
    from step_gpt_train_03_b300.gpt2lib import GPT2
    m = GPT2(shape, B, T, precision)
    m.load_params(synth.init_params(shape, seed))
    return m


def gpu_grads_numpy(m):
    return {k: v.detach().cpu().numpy().astype(np.float64) for k, v in m.grads().items()}


def gpu_params_numpy(m):
    return {k: v.detach().cpu().numpy().astype(np.float64) for k, v in m.params().items()}


def run_gpu(shape, precision, seed, batches, hp, grads_at=(0,)):
    """Train on the GPU over `batches`; returns (losses, {step: grads}, final loss)."""
    B, T = batches[0][0].shape
    m = gpu_model(shape, B, T, precision, seed)
    losses, grads = [], {}
    for i, (tok, tgt) in enumerate(batches):
        losses.append(m.forward(dev_tokens(tok), dev_tokens(tgt)))
        m.zero_grad()
        m.backward()
        if i in grads_at:
            grads[i] = gpu_grads_numpy(m)
        m.update(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], i + 1)
    return m, losses, grads


def run_oracle(shape, seed, batches, hp, dtype=np.float64, grads_at=(0,)):
    from tests.oracle_helpers import make_oracle
    o = make_oracle(shape, seed, dtype)
    losses, grads = [], {}
    for i, (tok, tgt) in enumerate(batches):
        losses.append(o.forward(tok, tgt))
        o.zero_grad()
        o.backward()
        if i in grads_at:
            grads[i] = {k: v.copy() for k, v in o.g.items()}
        o.update(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], i + 1)
    return o, losses, grads


def hp_of(w: synth.Workload):
    return dict(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay)
