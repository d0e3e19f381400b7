"""Shared helpers for the tests: build oracles and PyTorch restatements from synth inputs."""
from __future__ import annotations

import os

import numpy as np

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_header():
    out = {}
    with open(os.path.join(GOLDEN, "llmc_header.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = int(v)
    return out


def make_oracle(shape, seed, dtype=np.float64):
    o = O.from_shape(shape, dtype)
    o.load(synth.init_params(shape, seed))
    return o


def torch_model_loss(P, tokens, targets, shape):
    """GPT-2 loss written with PyTorch library layers (autograd gives the grads).

    Independent of the oracle's hand-written formulas: F.layer_norm, F.linear,
    F.scaled_dot_product_attention(is_causal=True), F.gelu(approximate='tanh'),
    F.cross_entropy over the real vocabulary columns.
    """
    import torch
    import torch.nn.functional as F
    C, NH, L, V = shape.channels, shape.num_heads, shape.num_layers, shape.vocab_size
    hs = C // NH
    tok = torch.as_tensor(tokens, dtype=torch.long)
    tgt = torch.as_tensor(targets, dtype=torch.long)
    B, T = tok.shape
    x = P["wte"][tok] + P["wpe"][:T]
    for l in range(L):
        h = F.layer_norm(x, (C,), P["ln1w"][l], P["ln1b"][l], eps=1e-5)
        qkv = F.linear(h, P["qkvw"][l], P["qkvb"][l])
        q, k, v = qkv.split(C, dim=-1)
        q, k, v = (z.reshape(B, T, NH, hs).transpose(1, 2) for z in (q, k, v))
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(y, P["attprojw"][l], P["attprojb"][l])
        h = F.layer_norm(x, (C,), P["ln2w"][l], P["ln2b"][l], eps=1e-5)
        h = F.gelu(F.linear(h, P["fcw"][l], P["fcb"][l]), approximate="tanh")
        x = x + F.linear(h, P["fcprojw"][l], P["fcprojb"][l])
    x = F.layer_norm(x, (C,), P["lnfw"], P["lnfb"], eps=1e-5)
    logits = F.linear(x, P["wte"])[..., :V]
    return F.cross_entropy(logits.reshape(-1, V), tgt.reshape(-1)), logits


def rel_max_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    denom = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / denom)
